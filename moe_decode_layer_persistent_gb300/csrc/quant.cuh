// quant.cuh -- shared-memory operand layouts and the NVFP4 activation
// quantiser run on the GPU.
//
// Operand layouts (tcgen05, K-major, 128-byte swizzle): a K-block is 128 bytes
// of every row (64 bf16 or 256 fp4 elements); rows are 128 B apart and 8-row
// groups 1024 B apart; the 16-byte chunk c of row r sits at chunk c ^ (r % 8).
//
// Scale-factor layout (block-scaled MMA, one E4M3 per 16 elements): a chunk
// covers 128 rows x 64 elements (4 scale bytes per row) in 512 bytes; the
// scale of row m, sub-block j (0..3) is byte (m % 32) * 16 + (m / 32) * 4 + j.
//
// Quantiser (the expert inputs: one row = one token's pooled vector, or one
// (token, expert) pair's SwiGLU output), page "Muse Spark Open: 1,109 Tokens a
// Second Is a Kernel Change, Not a Model Change", section "Where the kernel
// boundary sits ...": the expert GEMMs consume fp4 activations.  Each step is
// a correctly rounded float32 operation:
//   s_row = amax(|row|) / 2688  (1 when the row is all zero)
//   per 16 elements: s_b = E4M3_rn_satfinite(amax16 / (6 * s_row)),
//                    q_i = E2M1_rn_satfinite(x_i / (s_b * s_row)), 0 if s_b = 0.
#pragma once
#include "ptx.cuh"

namespace mk {

// Byte offset of (row r, byte b of the row's K-block) inside one K-block tile
// of an operand with 128-byte swizzle.
MK_DEV uint32_t sw128_offset(uint32_t r, uint32_t b) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((((b >> 4) ^ r) & 7u) << 4) + (b & 15u);
}

MK_DEV uint32_t sf_atom_offset(uint32_t m, uint32_t j) {
  return (m & 31u) * 16u + (m >> 5) * 4u + j;
}

MK_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
MK_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

MK_DEV void load_bf16x16(const __nv_bfloat16* p, float (&x)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 a = q[0], b = q[1];
  uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// The same from global memory written earlier in this launch by other CTAs
// (loaded from L2, never from the SM's non-coherent L1).
MK_DEV void load_bf16x16_cg(const __nv_bfloat16* p, float (&x)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 a = __ldcg(q), b = __ldcg(q + 1);
  uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// E2M1 codes (two packed words, element 0 in the low nibble) of the
// correctly rounded quotients x_i / c, without sixteen divisions: with
// rc = 1/c rounded, x_i * rc lies within 2 ulp of the rounded quotient, so the
// interval r(1 - 2^-20) .. r(1 + 2^-20) holds it.  Rounding to E2M1 is
// monotone, so when both ends of every interval give the same codes those are
// the quotients' codes; otherwise (a quotient near a rounding boundary, or
// 1/c out of range) the sixteen exact divisions decide.
MK_DEV void e2m1_codes16(const float (&x)[16], float c, uint32_t& w0, uint32_t& w1) {
  const float rc = __frcp_rn(c);
  float lo[16], hi[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float r = __fmul_rn(x[i], rc);
    lo[i] = __fmul_rn(r, 0.99999904632568359375f);   // 1 - 2^-20
    hi[i] = __fmul_rn(r, 1.00000095367431640625f);   // 1 + 2^-20
  }
  const uint32_t l0 = cvt_e2m1x4(lo[0], lo[1], lo[2], lo[3]) | (cvt_e2m1x4(lo[4], lo[5], lo[6], lo[7]) << 16);
  const uint32_t l1 = cvt_e2m1x4(lo[8], lo[9], lo[10], lo[11]) | (cvt_e2m1x4(lo[12], lo[13], lo[14], lo[15]) << 16);
  const uint32_t h0 = cvt_e2m1x4(hi[0], hi[1], hi[2], hi[3]) | (cvt_e2m1x4(hi[4], hi[5], hi[6], hi[7]) << 16);
  const uint32_t h1 = cvt_e2m1x4(hi[8], hi[9], hi[10], hi[11]) | (cvt_e2m1x4(hi[12], hi[13], hi[14], hi[15]) << 16);
  if (l0 == h0 && l1 == h1 && rc < 3.0e38f) {
    w0 = l0;
    w1 = l1;
    return;
  }
  float r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __fdiv_rn(x[i], c);
  w0 = cvt_e2m1x4(r[0], r[1], r[2], r[3]) | (cvt_e2m1x4(r[4], r[5], r[6], r[7]) << 16);
  w1 = cvt_e2m1x4(r[8], r[9], r[10], r[11]) | (cvt_e2m1x4(r[12], r[13], r[14], r[15]) << 16);
}

// One warp quantises one row of K bf16 values (K % 16 == 0, row 16-byte
// aligned).  For every 16-element block b the sink receives the 8 code bytes
// (two 32-bit words, element 16b in the low nibble of the first byte) and the
// scale byte.  Returns s_row (same value in every lane).
template <class Sink>
MK_DEV float quantize_row_nvfp4(const __nv_bfloat16* row, int K, Sink& sink) {
  const int lane = lane_id();
  const int nblk = K >> 4;
  float amax = 0.f;
  for (int b = lane; b < nblk; b += 32) {
    float x[16];
    load_bf16x16(row + b * 16, x);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = warp_max(amax);
  const float s_row = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  const float d6 = __fmul_rn(6.0f, s_row);
  for (int b = lane; b < nblk; b += 32) {
    float x[16];
    load_bf16x16(row + b * 16, x);
    float a16 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a16 = fmaxf(a16, fabsf(x[i]));
    const uint32_t sb = cvt_e4m3(__fdiv_rn(a16, d6));
    const float sbf = e4m3_to_float(sb);
    uint32_t w0 = 0, w1 = 0;
    if (sbf > 0.f) {
      e2m1_codes16(x, __fmul_rn(sbf, s_row), w0, w1);
    }
    sink.put(b, w0, w1, sb);
  }
  return s_row;
}

// One 16-element block of a row whose scale s_row is known: E4M3 block scale
// sb and the E2M1 codes (w0, w1), by the rule above.
MK_DEV void quantize_block16(const float (&x)[16], float s_row, uint32_t& w0, uint32_t& w1,
                             uint32_t& sb) {
  float a16 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a16 = fmaxf(a16, fabsf(x[i]));
  sb = cvt_e4m3(__fdiv_rn(a16, __fmul_rn(6.0f, s_row)));
  const float sbf = e4m3_to_float(sb);
  w0 = w1 = 0;
  if (sbf > 0.f) e2m1_codes16(x, __fmul_rn(sbf, s_row), w0, w1);
}

// Sink writing row-major codes [K/2] and scales [K/16] (used by self-tests).
struct RowMajorSink {
  uint8_t* codes;
  uint8_t* scales;
  MK_DEV void put(int b, uint32_t w0, uint32_t w1, uint32_t sb) {
    reinterpret_cast<uint2*>(codes)[b] = make_uint2(w0, w1);
    scales[b] = static_cast<uint8_t>(sb);
  }
};

// Sink writing row `r` of a block-scaled MMA operand: codes into K-blocks of
// 2048 bytes (16 rows x 128 B, 128-byte swizzle) and scales into 512-byte
// chunks (one per 64 elements).
struct OperandSink {
  uint8_t* codes;   // K-block 0 of the operand
  uint8_t* sf;      // chunk 0 of the scale factors
  uint32_t r;       // operand row (< 16)
  MK_DEV void put(int b, uint32_t w0, uint32_t w1, uint32_t sb) {
    const uint32_t byte = static_cast<uint32_t>(b) * 8u;          // byte in row
    const uint32_t kb = byte >> 7;
    *reinterpret_cast<uint2*>(codes + kb * 2048u + sw128_offset(r, byte & 127u)) =
        make_uint2(w0, w1);
    sf[(b >> 2) * 512u + sf_atom_offset(r, b & 3)] = static_cast<uint8_t>(sb);
  }
};

}  // namespace mk
