// selftest.cu -- small kernels that exercise the layer's building blocks in
// isolation (NVFP4 quantiser; TMA + tcgen05 MMA tile, bf16 and block-scaled
// NVFP4) so the test suite can check each against the CPU oracle.
#include "../../include/mk_selftest.h"
#include "host_util.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mk {
mk_status launch_sf_repack(const void* in, void* out, int G, int N, int K, cudaStream_t s);
size_t sf_repacked_bytes(int G, int N, int K);

__global__ void k_selftest_quant(const __nv_bfloat16* x, int rows, int K, uint8_t* codes,
                                 uint8_t* scales, float* s_row) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (warp >= rows) return;
  RowMajorSink sink{codes + static_cast<size_t>(warp) * (K / 2),
                    scales + static_cast<size_t>(warp) * (K / 16)};
  const float s = quantize_row_nvfp4(x + static_cast<size_t>(warp) * K, K, sink);
  if (lane_id() == 0) s_row[warp] = s;
}

// Single CTA, 256 threads: warp 0 issues TMA, warp 1 allocates TMEM and issues
// the MMAs, warps 2-3 stage B, warps 4-7 read the accumulator.
template <bool FP4>
__global__ void __launch_bounds__(256, 1)
    k_selftest_mma(const __grid_constant__ CUtensorMap tmA, const uint8_t* sfa_rep,
                   const uint8_t* b, const uint8_t* b_scales, int K, float* out,
                   uint32_t* status) {
  constexpr uint64_t kTimeout = 200ull * 1000 * 1000;  // 200 ms
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int KB = FP4 ? K / 256 + (K % 256 ? 1 : 0) : K / 64;  // K-blocks of 128 B per row
  uint8_t* sA = smem;                       // KB x 16 KB
  uint8_t* sSFA = sA + KB * 16384;          // KB x 2 KB
  uint8_t* sB = sSFA + KB * 2048;           // KB x 2 KB
  uint8_t* sSFB = sB + KB * 2048;           // KB x 2 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sSFB + KB * 2048);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  // zero B / SFB (rows past the data and padding K-blocks must read as 0)
  for (int i = threadIdx.x; i < KB * 4096 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sB)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  if (warp == 0 && lane_id() == 0) {
    const uint32_t bytes = KB * 16384 + (FP4 ? KB * 2048 : 0);
    mbar_arrive_expect_tx(&bars[0], bytes);
    const uint64_t pol = policy_evict_first();
    for (int kb = 0; kb < KB; ++kb) {
      tma_load_2d(sA + kb * 16384, &tmA, &bars[0], kb * (FP4 ? 128 : 64), 0, pol);
      if (FP4) bulk_load(sSFA + kb * 2048, sfa_rep + kb * 2048, 2048, &bars[0], pol);
    }
  }
  if (warp == 2 || warp == 3) {
    const int t = threadIdx.x - 64;
    const int row_bytes = FP4 ? K / 2 : K * 2;
    const int chunks = row_bytes / 16;
    for (int i = t; i < 16 * chunks; i += 64) {
      const int n = i / chunks, c = i % chunks;
      const int byte = c * 16;
      const uint4 v = *reinterpret_cast<const uint4*>(b + static_cast<size_t>(n) * row_bytes + byte);
      *reinterpret_cast<uint4*>(sB + (byte >> 7) * 2048 + sw128_offset(n, byte & 127)) = v;
    }
    if (FP4) {
      const int K16 = K / 16;
      for (int i = t; i < 16 * K16; i += 64) {
        const int n = i / K16, k16 = i % K16;
        sSFB[(k16 >> 2) * 512 + sf_atom_offset(n, k16 & 3)] = b_scales[n * K16 + k16];
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 1 && lane_id() == 0) {
    const bool ok = mbar_wait_bounded(&bars[0], 0, kTimeout);
    tc_fence_after();
    const uint32_t acc = tbase;
    if (!ok) atomicExch(status, 1u);
    for (int kb = 0; ok && kb < KB; ++kb) {
      const uint64_t da = sdesc_kmajor_sw128(smem_u32(sA + kb * 16384));
      const uint64_t db = sdesc_kmajor_sw128(smem_u32(sB + kb * 2048));
      if (FP4) {
        const uint32_t sfa_col = tbase + 32 + kb * 16, sfb_col = tbase + 128 + kb * 16;
        for (int c = 0; c < 4; ++c) {
          tmem_cp_sf(sfa_col + 4 * c, sdesc_sf_chunk(smem_u32(sSFA + kb * 2048 + c * 512)));
          tmem_cp_sf(sfb_col + 4 * c, sdesc_sf_chunk(smem_u32(sSFB + kb * 2048 + c * 512)));
        }
        for (int kk = 0; kk < 4; ++kk)
          mma_nvf4(acc, da + 2 * kk, db + 2 * kk, idesc_nvf4(128, 16), sfa_col + 4 * kk,
                   sfb_col + 4 * kk, (kb | kk) != 0);
      } else {
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(acc, da + 2 * kk, db + 2 * kk, idesc_bf16(128, 16), (kb | kk) != 0);
      }
    }
    mma_commit(&bars[1]);
  }
  if (warp >= 4) {
    const bool ok = mbar_wait_bounded(&bars[1], 0, kTimeout);
    tc_fence_after();
    if (!ok) atomicExch(status, 2u);
    const int q = warp - 4;
    float v[16];
    tmem_ld16(tbase + (static_cast<uint32_t>(32 * q) << 16), v);
    const int m = 32 * q + lane_id();
    for (int n = 0; n < 16; ++n) out[n * 128 + m] = v[n];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 256);
}

// Intra-GPU synchronisation costs (the synchronisation bill of page "Muse
// Spark Open: 1,109 Tokens a Second ...", section "Three bills a kernel this
// big has to pay", measured within one GPU).  modes 0/1: CTAs 0 and 1 of a
// cooperative launch (one per SM) ping-pong `iters` rounds; CTA 0 times the
// rounds with %globaltimer and reports half a round trip:
//   0: a flag word: st.release.gpu of the round number, polled with
//      ld.acquire.gpu;
//   1: the data as the signal: each round's value (a bf16 number that
//      differs from the previous round's) is written with a relaxed store and
//      polled with relaxed loads until the word holds it -- no fence, no
//      acquire.
// mode 2: one ld.acquire.gpu poll of a resident word, back to back (CTA 0).
// mode 3: one fence.acq_rel.gpu with no memory traffic in flight (CTA 0).
// Every poll gives up after kPollLimit tries and sets *status.
constexpr uint32_t kPollLimit = 1u << 20;

MK_DEV uint16_t ld_relaxed_u16(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.relaxed.gpu.global.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
  return v;
}
MK_DEV void st_relaxed_u16(uint16_t* p, uint16_t v) {
  asm volatile("st.relaxed.gpu.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}
MK_DEV void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__global__ void __launch_bounds__(32, 1)
    k_selftest_sync(int mode, int iters, uint32_t* flags, uint16_t* slots, uint32_t* status,
                    unsigned long long* ns) {
  if (threadIdx.x != 0) return;
  const int me = blockIdx.x;
  uint64_t t0 = globaltimer();
  if (mode == 0) {
    for (int r = 1; r <= iters; ++r) {
      // CTA 0 sends round r on flags[0] and waits for the echo on flags[1]
      if (me == 0) st_release(flags, static_cast<uint32_t>(r));
      const uint32_t* in = flags + (me == 0 ? 1 : 0);
      uint32_t n = 0;
      while (ld_acquire(in) != static_cast<uint32_t>(r)) {
        if (++n == kPollLimit) { atomicExch(status, 1u); return; }
      }
      if (me == 1) st_release(flags + 1, static_cast<uint32_t>(r));
    }
  } else if (mode == 1) {
    uint16_t* out = slots + me;
    const uint16_t* in = slots + (me ^ 1);
    for (int r = 1; r <= iters; ++r) {
      const uint16_t val = static_cast<uint16_t>(0x3F80u + (r & 63));  // a bf16 number
      if (me == 0) st_relaxed_u16(out, val);
      uint32_t n = 0;
      while (ld_relaxed_u16(in) != val) {
        if (++n == kPollLimit) { atomicExch(status, 1u); return; }
      }
      if (me == 1) st_relaxed_u16(out, val);
    }
  } else if (mode == 2) {
    if (me != 0) return;
    uint32_t acc = 0;
    for (int r = 0; r < iters; ++r) acc += ld_acquire(flags + 2);
    if (acc == 0xFFFFFFFFu) flags[3] = acc;  // keeps the loads
  } else {
    if (me != 0) return;
    for (int r = 0; r < iters; ++r) fence_acq_rel_gpu();
  }
  if (me == 0) *ns = globaltimer() - t0;
}

}  // namespace mk

using namespace mk;

extern "C" mk_status mk_selftest_sync(int32_t mode, int32_t iters, double* ns_per_op) {
  if (!ns_per_op || mode < 0 || mode > 3 || iters < 1 || iters > (1 << 20)) return MK_ERR_INVALID_ARG;
  uint8_t* buf = nullptr;
  MK_CUDA_TRY(cudaMalloc(&buf, 256));
  uint32_t* flags = reinterpret_cast<uint32_t*>(buf);
  uint16_t* slots = reinterpret_cast<uint16_t*>(buf + 64);
  uint32_t* status = reinterpret_cast<uint32_t*>(buf + 128);
  unsigned long long* ns = reinterpret_cast<unsigned long long*>(buf + 192);
  cudaError_t e = cudaMemset(buf, 0, 256);
  // 150 KB of shared memory per CTA: the two CTAs land on different SMs
  const int smem = 150 * 1024;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_selftest_sync, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  void* args[] = {&mode, &iters, &flags, &slots, &status, &ns};
  if (e == cudaSuccess)
    e = cudaLaunchCooperativeKernel(reinterpret_cast<void*>(k_selftest_sync), dim3(2), dim3(32), args, smem, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  unsigned long long h_ns = 0;
  uint32_t h_status = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&h_ns, ns, sizeof(h_ns), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&h_status, status, sizeof(h_status), cudaMemcpyDeviceToHost);
  cudaFree(buf);
  if (e != cudaSuccess) return MK_ERR_CUDA;
  if (h_status) return MK_ERR_TIMEOUT;
  // modes 0/1: a round is two hops
  *ns_per_op = static_cast<double>(h_ns) / iters / (mode <= 1 ? 2.0 : 1.0);
  return MK_OK;
}

extern "C" mk_status mk_selftest_quantize(const void* x, int32_t rows, int32_t K, void* codes,
                                          void* scales, float* s_row, void* stream) {
  if (!x || !codes || !scales || !s_row || rows <= 0 || K <= 0 || K % 16) return MK_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int threads = 128;
  const int blocks = (rows * 32 + threads - 1) / threads;
  k_selftest_quant<<<blocks, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows, K,
                                              static_cast<uint8_t*>(codes),
                                              static_cast<uint8_t*>(scales), s_row);
  MK_CUDA_TRY(cudaGetLastError());
  MK_CUDA_TRY(cudaStreamSynchronize(s));
  return MK_OK;
}

extern "C" mk_status mk_selftest_mma(int32_t fp4, const void* a, const void* a_scales,
                                     const void* b, const void* b_scales, int32_t K, float* out,
                                     void* stream) {
  if (!a || !b || !out || K <= 0 || K % 64) return MK_ERR_INVALID_ARG;
  if (fp4 && (!a_scales || !b_scales || K > 1024)) return MK_ERR_INVALID_ARG;
  if (!fp4 && K > 512) return MK_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap map;
  mk_status st = fp4 ? encode_tmap_2d(&map, a, 1, K / 2, 128, 128, 128)
                     : encode_tmap_2d(&map, a, 2, K, 128, 64, 128);
  if (st != MK_OK) return st;
  uint8_t* sfa = nullptr;
  uint32_t* status = nullptr;
  MK_CUDA_TRY(cudaMalloc(&status, sizeof(uint32_t)));
  MK_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(uint32_t), s));
  const int KB = fp4 ? (K + 255) / 256 : K / 64;
  if (fp4) {
    MK_CUDA_TRY(cudaMalloc(&sfa, sf_repacked_bytes(1, 128, K)));
    st = launch_sf_repack(a_scales, sfa, 1, 128, K, s);
    if (st != MK_OK) { cudaFree(sfa); cudaFree(status); return st; }
  }
  const size_t smem = 1024 + KB * (16384 + 3 * 2048) + 64;
  cudaError_t e;
  if (fp4) {
    cudaFuncSetAttribute(k_selftest_mma<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_selftest_mma<true><<<1, 256, smem, s>>>(map, sfa, static_cast<const uint8_t*>(b),
                                              static_cast<const uint8_t*>(b_scales), K, out, status);
  } else {
    cudaFuncSetAttribute(k_selftest_mma<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_selftest_mma<false><<<1, 256, smem, s>>>(map, nullptr, static_cast<const uint8_t*>(b),
                                               nullptr, K, out, status);
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  uint32_t h_status = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&h_status, status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (sfa) cudaFree(sfa);
  cudaFree(status);
  if (e != cudaSuccess) return MK_ERR_CUDA;
  return h_status ? MK_ERR_TIMEOUT : MK_OK;
}
