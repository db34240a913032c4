"""Number formats used by the layer, restated from their definitions.

* bfloat16 rounding (round-to-nearest-even, taken directly from float64 so no
  double rounding through float32 occurs).
* A generic minifloat decoder (sign / exponent / mantissa / bias), from which
  E2M1 (the NVFP4 element) and E4M3 (the NVFP4 block scale) are instantiated.
* Round-to-nearest-even, saturating encoders for E2M1 and E4M3.
* NVFP4 as the layer uses it (page "Muse Spark Open: 1,109 Tokens a Second Is a
  Kernel Change ...", section "Where the kernel boundary sits ...": experts
  stored in 4-bit NVFP4, fp4 data after the first expert GEMM): E2M1 codes with
  one E4M3 scale per 16 consecutive elements along K and one float32 scale per
  tensor (weights) or per row (activations).

Packing: a row of K elements is stored as K/2 bytes; element 2i is the low
nibble of byte i, element 2i+1 the high nibble.  Scales are one byte per 16
elements.  Nibble bit 3 is the sign.
"""

import numpy as np

# ----------------------------------------------------------------------------
# bfloat16 / float32 rounding
# ----------------------------------------------------------------------------

_BF16_MAX = float.fromhex("0x1.fe00000000000p+127")


def bf16_round(x):
    """Nearest bfloat16 value of float64 ``x`` (ties to even), as float64.

    bfloat16 has 8 significant bits and float32's exponent range (subnormal
    quantum 2^-133).  Rounding is done once, from the float64 value.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x)
    xf = x[fin]
    _, e = np.frexp(xf)                      # xf = m * 2**e, 0.5 <= |m| < 1
    q_exp = np.maximum(e - 8, -133)          # quantum of the bf16 binade
    r = np.rint(np.ldexp(xf, -q_exp))        # exact scaling, then RNE
    v = np.ldexp(r, q_exp)
    big = np.abs(v) > _BF16_MAX
    v[big] = np.copysign(np.inf, v[big])
    out[fin] = v
    return out


def f32(x):
    """Round float64 to the nearest float32 (ties to even), returned as float32."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# ----------------------------------------------------------------------------
# Minifloat decoding from the bit-field definition
# ----------------------------------------------------------------------------

def minifloat_decode(codes, exp_bits, man_bits, bias, specials):
    """Decode integer codes of a sign/exponent/mantissa format to float64.

    specials: "ieee"  -> all-ones exponent is inf (mantissa 0) or NaN;
              "fn"    -> only all-ones exponent and all-ones mantissa is NaN;
              "none"  -> every code is finite.
    Exponent field 0 encodes subnormals  m / 2^man_bits * 2^(1 - bias);
    otherwise (1 + m / 2^man_bits) * 2^(e - bias).
    """
    c = np.asarray(codes, dtype=np.int64)
    sign = (c >> (exp_bits + man_bits)) & 1
    e = (c >> man_bits) & ((1 << exp_bits) - 1)
    m = c & ((1 << man_bits) - 1)
    frac = m.astype(np.float64) / float(1 << man_bits)
    mag = np.where(e == 0,
                   np.ldexp(frac, 1 - bias),
                   np.ldexp(1.0 + frac, e - bias))
    emax = (1 << exp_bits) - 1
    mmax = (1 << man_bits) - 1
    if specials == "ieee":
        mag = np.where((e == emax) & (m == 0), np.inf, mag)
        mag = np.where((e == emax) & (m != 0), np.nan, mag)
    elif specials == "fn":
        mag = np.where((e == emax) & (m == mmax), np.nan, mag)
    elif specials != "none":
        raise ValueError(specials)
    return np.where(sign == 1, -mag, mag)


def e2m1_decode(codes):
    """E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/NaN."""
    return minifloat_decode(codes, 2, 1, 1, "none")


def e4m3_decode(codes):
    """E4M3 ('fn' variant): bias 7, no inf, 0x7F/0xFF are NaN, max 448."""
    return minifloat_decode(codes, 4, 3, 7, "fn")


_E2M1_POS = e2m1_decode(np.arange(8))        # 0, .5, 1, 1.5, 2, 3, 4, 6
_E4M3_POS = e4m3_decode(np.arange(127))      # finite non-negative, ascending


def _rne_encode(mag, table, max_code):
    """Nearest entry of the ascending ``table`` (index = code) to ``mag`` >= 0,
    ties to the even code, values above the last entry saturate to it."""
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(table, mag, side="left")
    hi = np.clip(hi, 0, max_code)
    lo = np.clip(hi - 1, 0, max_code)
    d_lo = mag - table[lo]
    d_hi = table[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= table[max_code], max_code, code)
    return code.astype(np.uint8)


def e2m1_encode(x):
    """float32 -> E2M1 code, round to nearest even, saturating at +-6.

    The sign bit follows the sign of x (so small negatives give code 8, -0)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    code = _rne_encode(np.abs(x), _E2M1_POS, 7)
    return (code | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def e4m3_encode(x):
    """float32 -> E4M3 code, round to nearest even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    code = _rne_encode(np.abs(x), _E4M3_POS, 126)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


# ----------------------------------------------------------------------------
# NVFP4 packing, decoding and the activation quantiser
# ----------------------------------------------------------------------------

def unpack_nibbles(packed):
    """[..., K/2] bytes -> [..., K] codes (element 2i = low nibble of byte i)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def pack_nibbles(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def nvfp4_dequantize(packed, scales, tensor_scale):
    """Value = e2m1(code) * e4m3(block scale) * tensor_scale, in float64.

    packed: [..., K/2] uint8; scales: [..., K/16] uint8 (E4M3 bytes);
    tensor_scale: float32 scalar or array broadcastable to the rows.
    """
    codes = unpack_nibbles(packed)
    K = codes.shape[-1]
    v = e2m1_decode(codes)
    sb = e4m3_decode(scales)
    v = v.reshape(v.shape[:-1] + (K // 16, 16)) * sb[..., None]
    ts = np.asarray(tensor_scale, dtype=np.float32).astype(np.float64)
    if ts.ndim:
        ts = ts.reshape(ts.shape + (1, 1))
    return (v * ts).reshape(codes.shape)


def nvfp4_quantize_rows(x):
    """Quantise each row of ``x`` (values that are exactly bfloat16) to NVFP4.

    The rule, taken in float32 arithmetic (each operation correctly rounded):
      s_row = amax(|row|) / 2688            (2688 = 6 * 448; s_row = 1 if amax = 0)
      for each block of 16 along the row:
        d   = 6 * s_row
        s_b = E4M3_rne_satfinite(amax16 / d)
        c   = s_b * s_row
        q_i = E2M1_rne_satfinite(x_i / c)   (q = 0 when s_b = 0)
    Returns (packed codes [rows, K/2] uint8, scales [rows, K/16] uint8,
             s_row [rows] float32).
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    rows, K = x32.shape
    assert K % 16 == 0
    amax = np.max(np.abs(x32), axis=1)
    s_row = np.where(amax > 0, amax / np.float32(2688.0), np.float32(1.0)).astype(np.float32)
    blk = x32.reshape(rows, K // 16, 16)
    amax16 = np.max(np.abs(blk), axis=2)
    d = (np.float32(6.0) * s_row).astype(np.float32)
    t = (amax16 / d[:, None]).astype(np.float32)
    sb = e4m3_encode(t)
    sbv = e4m3_decode(sb).astype(np.float32)
    c = (sbv * s_row[:, None]).astype(np.float32)
    safe_c = np.where(c > 0, c, np.float32(1.0)).astype(np.float32)
    ratio = (blk / safe_c[:, :, None]).astype(np.float32)
    codes = e2m1_encode(ratio)
    codes = np.where((sbv > 0)[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    return pack_nibbles(codes.reshape(rows, K)), sb, s_row
