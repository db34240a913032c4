"""Readings of the pages checked on the arithmetic alone (CPU).

The fused next-layer QKV: the pages apply RMSNorm and then the QKV
projection, and do not say where the bf16 rounding of the normalised input
falls.  The oracle (and the first-layer QKV on the GPU) project
h = bf16(x * r * gain), r the row's RMS factor; the fused next-layer QKV on
the GPU projects bf16(x * gain) and multiplies the float32 sum by r, so that
it can start on each 128-column tile of x as soon as that tile is final.  In
exact arithmetic the two are the same map.  These tests measure, in the
oracle's float64 arithmetic at the stack's shapes, what moving that one
rounding costs against the oracle: it stays inside the layer contract
(max |err| <= 2e-2 * RMS or one bf16 ulp of the element, cosine >= 0.9995),
and no element moves by more than one bf16 ulp of the largest output of its
row.
"""

import numpy as np
import pytest

import layer_harness as H
from oracle import layer as ol
from oracle.numerics import bf16_round


def _draw(seed, T=16, Hd=4096, N=6144):
    rng = np.random.default_rng(seed)
    x = bf16_round(rng.standard_normal((T, Hd)) * 1.7)
    gain = bf16_round(1.0 + 0.1 * rng.standard_normal(Hd))
    w = bf16_round(rng.standard_normal((N, Hd)) / np.sqrt(Hd))
    return x, gain, w


def _rms_factor_first(x, gain, w):
    n = bf16_round(ol.rmsnorm(x, gain))
    return bf16_round(n @ w.T)


def _rms_factor_after(x, gain, w):
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + ol.RMS_EPS)
    return bf16_round(r * (bf16_round(x * gain) @ w.T))


def test_rms_factor_first_is_the_oracle_qkv_projection():
    x, gain, w = _draw(0, Hd=512, N=768)
    q, k, v = ol.qkv_project(x, gain, w, 4, 1, 128)
    got = np.concatenate([q.reshape(16, -1), k.reshape(16, -1), v.reshape(16, -1)], axis=1)
    assert np.array_equal(got, _rms_factor_first(x, gain, w))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rms_factor_after_the_projection_stays_inside_the_contract(seed):
    x, gain, w = _draw(seed)
    ref = _rms_factor_first(x, gain, w)
    alt = _rms_factor_after(x, gain, w)
    H.assert_close("next-layer q/k/v", alt, ref)
    row_ulp = H.bf16_ulp(np.abs(ref).max(axis=1, keepdims=True))
    assert np.all(np.abs(alt - ref) <= row_ulp)
