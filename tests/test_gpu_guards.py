"""Checks that stand in for a memory checker (compute-sanitizer is closed on
this pool) and for the self-timing contract, all through the C ABI:

  * NaN-poisoned KV rows that no verify token may see (below the sliding
    window, and past ctx + T up to the end of the cache) leave every output
    finite and bit-identical to the run without poison: nothing reads them;
  * canary rows around x_out, q_out, the top-k outputs and the written cache
    rows are unchanged after a step: nothing writes outside its rows;
  * outputs are bit-identical with the kernel's self-timing stamps on and off
    (page "Muse Spark Open: 1,109 Tokens a Second Is a Kernel Change, Not a
    Model Change", section "What the 5.9 ms is still spent on": the timing
    leaves the results unchanged).
"""

import os

import numpy as np
import pytest
import torch

from moe_decode_layer_persistent_gb300 import synth
import layer_harness as H

pytestmark = pytest.mark.gpu

NAN_BF16 = torch.tensor(float("nan"), dtype=torch.bfloat16)
GUARD = 3            # canary rows on each side of an output
CANARY = -1152.0     # exactly representable in bf16 and float32


def _layer(binding, work, fuse, max_ctx):
    c = work["cfgs"][0]
    flags = binding.MK_FIRST_LAYER | (binding.MK_FUSE_NEXT_QKV if fuse else 0)
    return H.make_layer(binding, c, work["Ws"][0], flags, max_ctx,
                        next_W=work["next"] if fuse else None)


def _guarded(rows, cols, dtype, fill=CANARY):
    """A buffer of rows + 2 * GUARD rows filled with the canary; returns
    (whole buffer, view of the middle rows zeroed)."""
    buf = torch.full((rows + 2 * GUARD, cols), fill, dtype=dtype, device="cuda")
    mid = buf[GUARD:GUARD + rows]
    mid.zero_()
    return buf, mid


def _step(binding, layer, work, T, ctx, kc, vc, fuse, nkc=None, nvc=None):
    """One step with canary rows around every output; returns the outputs and
    asserts the canaries are intact."""
    c = work["cfgs"][0]
    H_, qd = c["hidden"], c["n_q_heads"] * c["head_dim"]
    moe = c["ffn"] == "moe"
    k = c.get("top_k", 1)
    xb, x_out = _guarded(T, H_, torch.bfloat16)
    qb, q_out = _guarded(T, qd, torch.bfloat16) if fuse else (None, None)
    ib, idx = _guarded(T, k, torch.int32, fill=-77) if moe else (None, None)
    wb, wts = _guarded(T, k, torch.float32) if moe else (None, None)
    io = binding.make_step_io(T, ctx, work["x_in"][:T].contiguous(), x_out, kc, vc,
                              next_k_cache=nkc, next_v_cache=nvc, q_out=q_out,
                              topk_idx_out=idx, topk_w_out=wts)
    binding.mk_decode_step(layer, io)
    torch.cuda.synchronize()
    assert binding.mk_layer_status(layer) == 0
    for name, b, fill in (("x_out", xb, CANARY), ("q_out", qb, CANARY), ("idx", ib, -77),
                          ("w", wb, CANARY)):
        if b is None:
            continue
        for part in (b[:GUARD], b[-GUARD:]):
            assert bool((part == fill).all()), "canary around %s overwritten" % name
    out = dict(x_out=x_out.clone(), k=kc.clone(), v=vc.clone())
    if fuse:
        out.update(q_out=q_out.clone(), nk=nkc.clone(), nv=nvc.clone())
    if moe:
        out.update(idx=idx.clone(), w=wts.clone())
    return out


def _poison(cache, lo, hi_from):
    """NaN in rows [0, lo) and [hi_from, end) of a cache (rows no verify token
    of this step may see)."""
    c = cache.clone()
    c[:lo] = NAN_BF16
    c[hi_from:] = NAN_BF16
    return c


@pytest.mark.parametrize("name,T,ctx", [("swa_layer", 16, 5000), ("global_layer_fused", 16, 3000),
                                        ("tiny_layer", 7, 90)])
def test_unseen_kv_rows_poisoned_with_nan_change_nothing(cuda_lib, name, T, ctx):
    wl = synth.WORKLOADS[name]
    work, _ = H.prepare(name, "host" if name == "tiny_layer" else "cuda", T=T, ctx=ctx, enforce=False)
    fuse = work["next"] is not None
    pad = 200                                   # cache rows past ctx + T
    kc0, vc0 = (torch.cat([t, torch.zeros((pad,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)])
                for t in work["caches"][0])
    max_ctx = kc0.shape[0]
    window = wl["window"]
    lo = max(0, ctx - window + 1) if window else 0
    layer = _layer(cuda_lib, work, fuse, max_ctx)
    try:
        nk0 = nv0 = None
        if fuse:
            nk0, nv0 = (torch.cat([t, torch.zeros((pad,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)])
                        for t in (work["next"]["k_cache"], work["next"]["v_cache"]))
        clean = _step(cuda_lib, layer, work, T, ctx, kc0.clone(), vc0.clone(), fuse,
                      nk0.clone() if fuse else None, nv0.clone() if fuse else None)
        kp, vp = _poison(kc0, lo, ctx + T), _poison(vc0, lo, ctx + T)
        # the next layer's caches: only rows ctx..ctx+T-1 belong to this step
        nkp = _poison(nk0, ctx, ctx + T) if fuse else None
        nvp = _poison(nv0, ctx, ctx + T) if fuse else None
        dirty = _step(cuda_lib, layer, work, T, ctx, kp, vp, fuse, nkp, nvp)
    finally:
        cuda_lib.mk_layer_destroy(layer)
    assert torch.isfinite(dirty["x_out"].float()).all()
    assert torch.equal(dirty["x_out"], clean["x_out"])
    # the rows the step writes, bit-identical; the poisoned rows untouched
    for key in ("k", "v"):
        assert torch.equal(dirty[key][ctx:ctx + T], clean[key][ctx:ctx + T])
        assert torch.isnan(dirty[key][ctx + T:].float()).all()
        assert torch.isnan(dirty[key][:lo].float()).all()
    if fuse:
        assert torch.equal(dirty["q_out"], clean["q_out"])
        for key in ("nk", "nv"):
            assert torch.equal(dirty[key][ctx:ctx + T], clean[key][ctx:ctx + T])
            assert torch.isnan(dirty[key][ctx + T:].float()).all()
            assert torch.isnan(dirty[key][:ctx].float()).all()
    if "idx" in clean:
        assert torch.equal(dirty["idx"], clean["idx"]) and torch.equal(dirty["w"], clean["w"])


@pytest.mark.parametrize("name,T,ctx", [("global_layer_fused", 16, 1000), ("tiny_layer", 5, 40)])
def test_cache_rows_outside_the_step_keep_their_canaries(cuda_lib, name, T, ctx):
    """Rows [0, ctx) keep their values and rows past ctx + T keep a canary, in
    this layer's caches and (fused) the next layer's; the output canaries are
    checked inside _step."""
    work, _ = H.prepare(name, "host" if name == "tiny_layer" else "cuda", T=T, ctx=ctx, enforce=False)
    fuse = work["next"] is not None
    pad = 64

    def padded(t):
        return torch.cat([t, torch.full((pad,) + tuple(t.shape[1:]), CANARY, dtype=t.dtype, device=t.device)])

    kc, vc = (padded(t) for t in work["caches"][0])
    before = (kc.clone(), vc.clone())
    nkc = nvc = None
    if fuse:
        nkc, nvc = (padded(t) for t in (work["next"]["k_cache"], work["next"]["v_cache"]))
        nbefore = (nkc.clone(), nvc.clone())
    layer = _layer(cuda_lib, work, fuse, kc.shape[0])
    try:
        _step(cuda_lib, layer, work, T, ctx, kc, vc, fuse, nkc, nvc)
    finally:
        cuda_lib.mk_layer_destroy(layer)
    for got, want in zip((kc, vc) + ((nkc, nvc) if fuse else ()), before + (nbefore if fuse else ())):
        assert torch.equal(got[:ctx], want[:ctx])
        assert torch.equal(got[ctx + T:], want[ctx + T:])
        assert not torch.equal(got[ctx:ctx + T], want[ctx:ctx + T])   # the step did write its rows


@pytest.mark.parametrize("name,T,ctx", [("swa_layer", 16, 8192), ("tiny_layer", 9, 70)])
def test_self_timing_leaves_outputs_bit_identical(cuda_lib, name, T, ctx):
    work, _ = H.prepare(name, "host" if name == "tiny_layer" else "cuda", T=T, ctx=ctx, enforce=False)
    fuse = work["next"] is not None
    outs = []
    for stamps in ("0", "1"):
        old = os.environ.get("MK_TIMESTAMPS")
        os.environ["MK_TIMESTAMPS"] = stamps
        try:
            layer = _layer(cuda_lib, work, fuse, work["caches"][0][0].shape[0])
        finally:
            if old is None:
                del os.environ["MK_TIMESTAMPS"]
            else:
                os.environ["MK_TIMESTAMPS"] = old
        try:
            kc, vc = (t.clone() for t in work["caches"][0])
            outs.append(_step(cuda_lib, layer, work, T, ctx, kc, vc, fuse))
            if stamps == "1":
                ts = cuda_lib.mk_get_timestamps(layer, cuda_lib.mk_layer_get_info(layer)["grid"])
                assert (ts[:, 9, 2] > ts[:, 9, 0]).all()       # the stamps were taken
        finally:
            cuda_lib.mk_layer_destroy(layer)
    for key in outs[0]:
        assert torch.equal(outs[0][key], outs[1][key]), key
