"""Pins for the oracle's number formats (CPU only)."""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import numerics as n

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((float(a), float(b)))
    return rows


@pytest.mark.parametrize("dtype,ebits,mbits,bias,spec,ncodes", [
    (torch.float16, 5, 10, 15, "ieee", 1 << 16),
    (torch.bfloat16, 8, 7, 127, "ieee", 1 << 16),
    (torch.float8_e5m2, 5, 2, 15, "ieee", 256),
    (torch.float8_e4m3fn, 4, 3, 7, "fn", 256),
])
def test_minifloat_decoder_matches_torch(dtype, ebits, mbits, bias, spec, ncodes):
    codes = np.arange(ncodes)
    mine = n.minifloat_decode(codes, ebits, mbits, bias, spec)
    itype = torch.int16 if ncodes > 256 else torch.uint8
    raw = torch.from_numpy(codes.astype(np.int64)).to(torch.int32)
    if itype == torch.int16:
        raw = raw.to(torch.int32).sub((raw >= 32768).to(torch.int32) * 65536).to(torch.int16)
    else:
        raw = raw.to(torch.uint8)
    ref = raw.view(dtype).to(torch.float64).numpy()
    both_nan = np.isnan(mine) & np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~both_nan], ref[~both_nan])
    # signed zeros too
    assert np.array_equal(np.signbit(mine[~both_nan]), np.signbit(ref[~both_nan]))


def test_e2m1_table_golden():
    rows = _read_pairs("e2m1_table.txt")
    codes = np.array([int(a) for a, _ in rows])
    vals = np.array([b for _, b in rows])
    assert np.array_equal(n.e2m1_decode(codes), vals)
    assert np.array_equal(n.e2m1_decode(codes | 8), -vals)


def test_e2m1_rne_golden_ties():
    for x, code in _read_pairs("e2m1_rne_ties.txt"):
        assert int(n.e2m1_encode(np.float32(x))) == int(code), x


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.uniform(-8, 8, 4000), np.arange(-70, 71) / 10.0,
                         np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])]).astype(np.float32)
    grid = [Fraction(v).limit_denominator(4) for v in (0, .5, 1, 1.5, 2, 3, 4, 6)]
    got = n.e2m1_encode(xs)
    for x, c in zip(xs, got):
        fx = Fraction(float(x))
        mag = abs(fx)
        best = None
        for code, g in enumerate(grid):
            dist = abs(mag - g)
            if best is None or dist < best[0] or (dist == best[0] and code % 2 == 0):
                best = (dist, code)
        exp = best[1] if mag < 6 else 7
        if x < 0 or (x == 0 and np.signbit(x)):
            exp |= 8
        assert int(c) == exp, (x, int(c), exp)


def test_e4m3_encode_matches_torch():
    rng = np.random.default_rng(2)
    vals = n.e4m3_decode(np.arange(127))
    mids = (vals[:-1] + vals[1:]) / 2
    xs = np.concatenate([rng.uniform(0, 448, 20000), rng.uniform(0, 0.02, 5000),
                         vals, mids, -rng.uniform(0, 448, 1000)]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(n.e4m3_encode(xs), ref)
    # saturation (torch's cast turns these into NaN; the encoder saturates)
    assert np.array_equal(n.e4m3_encode(np.float32([449, 464, 1e6, -1e6])),
                          np.uint8([0x7E, 0x7E, 0x7E, 0xFE]))


def test_bf16_round_matches_torch_on_float32():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
                        rng.standard_normal(1000) * 1e-39]).astype(np.float32)
    # exact midpoints between bf16 neighbours
    b = torch.from_numpy(rng.standard_normal(2000).astype(np.float32)).bfloat16().float().numpy()
    mid = (b.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, mid])
    ref = torch.from_numpy(x).bfloat16().double().numpy()
    assert np.array_equal(n.bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_is_single_rounding_from_float64():
    # 1 + 2^-8 + 2^-40 is just above a bf16 midpoint; a float32 detour would
    # land on the midpoint and round to even (1.0).
    cases = [(1 + 2 ** -8 + 2 ** -40, 1 + 2 ** -7), (1 + 2 ** -8, 1.0),
             (1 + 3 * 2 ** -8, 1 + 2 ** -6), (-(1 + 2 ** -8 + 2 ** -40), -(1 + 2 ** -7))]
    for x, want in cases:
        assert n.bf16_round(np.float64(x)) == want
    # against exact rational rounding on random float64 values
    rng = np.random.default_rng(4)
    xs = rng.standard_normal(3000) * 10.0 ** rng.integers(-5, 5, 3000)
    got = n.bf16_round(xs)
    for x, g in zip(xs, got):
        fx = Fraction(float(x))
        e = int(np.floor(np.log2(abs(float(x)))))
        q = Fraction(2) ** (e - 7)
        k = fx / q
        lo = k.numerator // k.denominator
        rem = k - lo
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
            lo += 1
        assert Fraction(float(g)) == lo * q


def test_nvfp4_dequantize_exhaustive():
    e2m1 = np.array([b for _, b in _read_pairs("e2m1_table.txt")])
    e2m1 = np.concatenate([e2m1, -e2m1])
    e4m3 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for ts in (1.0, 2.0 ** -10, 3.7e-5, 0.0123456789):
        ts32 = np.float32(ts)
        codes = np.repeat(np.arange(16, dtype=np.uint8), 127 * 16).reshape(16 * 127, 16)
        scales = np.tile(np.arange(127, dtype=np.uint8), 16).reshape(16 * 127, 1)
        got = n.nvfp4_dequantize(n.pack_nibbles(codes), scales, ts32)
        want = (e2m1[np.repeat(np.arange(16), 127)][:, None] * e4m3[np.tile(np.arange(127), 16)][:, None]
                * float(ts32)) * np.ones((1, 16))
        assert np.array_equal(got, want)
        # e2m1 * e4m3 is exact in float32
        prod = e2m1[np.repeat(np.arange(16), 127)] * e4m3[np.tile(np.arange(127), 16)]
        assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)


def test_pack_unpack_roundtrip_and_nibble_order():
    c = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    p = n.pack_nibbles(c)
    assert p.tolist() == [[0x21, 0x43]]
    assert np.array_equal(n.unpack_nibbles(p), c)


def _row_bf16(rng, rows, K, scale=1.0):
    return n.bf16_round(rng.standard_normal((rows, K)) * scale)


def test_quantizer_error_bound_and_max_element():
    rng = np.random.default_rng(5)
    x = _row_bf16(rng, 64, 256)
    q, s, r = n.nvfp4_quantize_rows(x)
    deq = n.nvfp4_dequantize(q, s, r)
    sb = n.e4m3_decode(s).astype(np.float32)
    c = (sb * r[:, None]).astype(np.float64)
    # every element within half a grid step of its block's E2M1 grid
    ratio = x.reshape(64, 16, 16) / c[:, :, None]
    mag = n.e2m1_decode(n.unpack_nibbles(q) & 7).reshape(64, 16, 16)
    grid = n.e2m1_decode(np.arange(8))
    # each code is the nearest E2M1 grid point to x / (block scale * s_row)
    nearest = np.min(np.abs(np.abs(ratio)[..., None] - grid), axis=-1)
    assert np.all(np.abs(np.abs(ratio) - mag) <= nearest + 1e-6)
    assert np.allclose(deq.reshape(64, 16, 16), mag * np.sign(ratio) * c[:, :, None])
    # the row amax element lands on the top code (+-6)
    codes = n.unpack_nibbles(q)
    am = np.argmax(np.abs(x), axis=1)
    assert np.all((codes[np.arange(64), am] & 7) == 7)
    # s_row definition
    assert np.array_equal(r, (np.max(np.abs(x.astype(np.float32)), axis=1) / np.float32(2688)).astype(np.float32))


def test_quantizer_zero_row_and_sign_symmetry_and_pow2_invariance():
    rng = np.random.default_rng(6)
    z = np.zeros((1, 64))
    q, s, r = n.nvfp4_quantize_rows(z)
    assert np.all(q == 0) and np.all(s == 0) and r[0] == 1.0
    x = _row_bf16(rng, 8, 128)
    q1, s1, r1 = n.nvfp4_quantize_rows(x)
    q2, s2, r2 = n.nvfp4_quantize_rows(-x)
    c1, c2 = n.unpack_nibbles(q1), n.unpack_nibbles(q2)
    assert np.array_equal(s1, s2) and np.array_equal(r1, r2)
    assert np.array_equal(c1 & 7, c2 & 7)
    nz = (c1 & 7) != 0
    assert np.array_equal((c1 ^ c2)[nz], np.full(nz.sum(), 8, dtype=np.uint8))
    q3, s3, r3 = n.nvfp4_quantize_rows(x * 2.0 ** 5)
    assert np.array_equal(q3, q1) and np.array_equal(s3, s1)
    assert np.array_equal(r3, r1 * np.float32(32))


def test_quantizer_blocks_are_independent():
    rng = np.random.default_rng(7)
    x = _row_bf16(rng, 1, 128)
    x[0, 0] = 10.0                     # fix the row amax
    q1, s1, _ = n.nvfp4_quantize_rows(x)
    y = x.copy()
    y[0, 40] = 0.5 * y[0, 40]          # inside block 2 only
    q2, s2, _ = n.nvfp4_quantize_rows(y)
    c1, c2 = n.unpack_nibbles(q1), n.unpack_nibbles(q2)
    changed = np.nonzero((c1 != c2)[0])[0]
    assert set(changed.tolist()) <= set(range(32, 48))
    assert np.array_equal(np.delete(s1, 2, axis=1), np.delete(s2, 2, axis=1))
