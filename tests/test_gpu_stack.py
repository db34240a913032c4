"""GPU parity of layer stacks (programmatic-dependent-launch chains) through
the C ABI: every layer is held to the single-layer contract.

For a stack of L layers:
  1. The layers run one launch at a time (mk_decode_step), each on the GPU's
     own outputs of the layer before (x, the fused next-layer q and the K/V
     rows that layer wrote).  Before each MoE layer runs, its router is
     redrawn on the oracle's h of THOSE inputs until every token's k-th and
     (k+1)-th logits are >= 1e-2 apart (the margin rule of the generator), so
     the expert sets are unique for the inputs the GPU sees.
  2. The same layers run as one stack (mk_stack_step): its outputs, every
     layer's cache rows and router indices must equal the one-at-a-time run
     bit for bit (the chaining adds no arithmetic).
  3. On a fixed subset of layers the oracle runs the layer on the GPU's inputs
     of that layer, and the GPU's outputs of the layer must meet the contract:
     expert sets exact (order within the float32 summation bound); x_out (and
     the first layer's own K/V rows) within max |err| <= 2e-2 RMS -- widened,
     for MoE layers, by the oracle's bound for one NVFP4 decision flip, as in
     the ragged single-layer tests -- and cosine >= 0.9995; the fused
     next-layer q and K/V rows within the same bound of the oracle's QKV
     projection of the GPU's own x_out (each stage on its own inputs).
"""

import numpy as np
import pytest
import torch

from moe_decode_layer_persistent_gb300 import synth
import layer_harness as H
import oracle_io as oio
from oracle import layer as ol
from oracle.numerics import bf16_round

pytestmark = pytest.mark.gpu


def _attention_half(cfg, W, x, kc, vc, ctx, q, first):
    """h of one layer from its inputs (the oracle's steps 1-4)."""
    T = x.shape[0]
    kc, vc = kc.copy(), vc.copy()
    if first:
        q, kn, vn = ol.qkv_project(x, W["attn_norm_w"], W["w_qkv"], cfg["n_q_heads"],
                                   cfg["n_kv_heads"], cfg["head_dim"])
        kc[ctx:ctx + T], vc[ctx:ctx + T] = kn, vn
    q = np.asarray(q).reshape(T, cfg["n_q_heads"], cfg["head_dim"])
    o = bf16_round(ol.attention(q, kc, vc, ctx, cfg["window"])).reshape(T, -1)
    x_mid = bf16_round(x + o @ W["w_o"].T)
    return bf16_round(ol.rmsnorm(x_mid, W["ffn_norm_w"]))


def _enforce_router_margin(work, l, h):
    """Redraw layer l's router (in place, so that a layer created on the
    tensor sees it) until the oracle's logits on h meet the margin."""
    c = work["cfgs"][l]
    W = work["Ws"][l]
    for draw in range(400):
        wr = synth.router_weight(work["wl"], work["seed"], l, draw, W["w_router"].device)
        logits, _, _ = ol.router(h, oio.np64(wr), c["top_k"])
        if np.all(oio.router_margin(logits, c["top_k"]) >= oio.MARGIN):
            W["w_router"].copy_(wr)
            return
    raise RuntimeError("no router draw met the margin at layer %d" % l)


def _check_stack(binding, work, subset):
    """Steps 1-3 of the module docstring; `subset` = layers checked against
    the oracle."""
    cfgs, Ws = work["cfgs"], work["Ws"]
    L = len(Ws)
    T, ctx = work["wl"]["T"], work["wl"]["ctx"]
    moe = work["wl"]["ffn"] == "moe"
    k = work["wl"].get("top_k", 1)
    max_ctx = work["caches"][0][0].shape[0]
    Hqd = cfgs[0]["n_q_heads"] * cfgs[0]["head_dim"]
    # 1. one launch per layer on the GPU's own outputs, margins on those inputs
    kcs = [c[0].clone() for c in work["caches"]]
    vcs = [c[1].clone() for c in work["caches"]]
    x = work["x_in"][:T].contiguous()
    q = None
    inputs, outputs, idx_chain = {}, {}, []
    layers = []
    try:
        for l in range(L):
            fuse = l + 1 < L
            if moe:
                Wl = oio.np_weights({n: Ws[l][n] for n in ("attn_norm_w", "w_qkv", "w_o", "ffn_norm_w")})
                h = _attention_half(oio.oracle_cfg(cfgs[l]), Wl, oio.np64(x), oio.np64(kcs[l]),
                                    oio.np64(vcs[l]), ctx, None if q is None else oio.np64(q), l == 0)
                _enforce_router_margin(work, l, h)
            flags = (binding.MK_FIRST_LAYER if l == 0 else 0) | (binding.MK_FUSE_NEXT_QKV if fuse else 0)
            lay = H.make_layer(binding, cfgs[l], Ws[l], flags, max_ctx, next_W=Ws[l + 1] if fuse else None)
            layers.append(lay)
            if l in subset:
                inputs[l] = dict(x=x.cpu(), q=None if q is None else q.cpu(),
                                 k=kcs[l].cpu(), v=vcs[l].cpu(),
                                 nk=kcs[l + 1].cpu() if fuse else None, nv=vcs[l + 1].cpu() if fuse else None)
            x_out = torch.zeros_like(x)
            q_out = torch.zeros((T, Hqd), dtype=torch.bfloat16, device="cuda") if fuse else None
            idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
            wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
            io = binding.make_step_io(T, ctx, x, x_out, kcs[l], vcs[l], q_in=q,
                                      next_k_cache=kcs[l + 1] if fuse else None,
                                      next_v_cache=vcs[l + 1] if fuse else None, q_out=q_out,
                                      topk_idx_out=idx if moe else None, topk_w_out=wts if moe else None)
            binding.mk_decode_step(lay, io)
            torch.cuda.synchronize()
            assert binding.mk_layer_status(lay) == 0, "layer %d" % l
            idx_chain.append(idx.clone())
            if l in subset:
                outputs[l] = dict(status=0, x_out=x_out.cpu(), k_cache=kcs[l].cpu(), v_cache=vcs[l].cpu(),
                                  idx=idx.cpu().numpy() if moe else None, w=wts.cpu().numpy() if moe else None)
                if fuse:
                    outputs[l].update(q_out=q_out.cpu(), next_k_cache=kcs[l + 1].cpu(),
                                      next_v_cache=vcs[l + 1].cpu())
            x, q = x_out, q_out
        # 2. the PDL-chained stack of the same layer objects, on fresh copies of
        # the caches
        stack = binding.mk_stack_create(layers)
        skc = [c[0].clone() for c in work["caches"]]
        svc = [c[1].clone() for c in work["caches"]]
        s_out = torch.zeros_like(x)
        s_idx = torch.full((L, T, k), -1, dtype=torch.int32, device="cuda") if moe else None
        binding.mk_stack_step(stack, binding.make_stack_io(T, ctx, work["x_in"][:T].contiguous(), s_out,
                                                           skc, svc, topk_idx_out=s_idx))
        torch.cuda.synchronize()
        st = binding.mk_stack_status(stack)
        binding.mk_stack_destroy(stack)
    finally:
        for lay in layers:
            binding.mk_layer_destroy(lay)
    assert st == 0
    assert torch.equal(s_out, x)
    for l in range(L):
        assert torch.equal(skc[l], kcs[l]) and torch.equal(svc[l], vcs[l]), "layer %d caches" % l
        if moe:
            assert torch.equal(s_idx[l], idx_chain[l]), "layer %d router" % l
    # 3. the oracle on the GPU's inputs of each layer of the subset, stage by
    # stage: the layer (x_out, routing; the first layer's own K/V rows) on the
    # GPU's inputs, and the fused next-layer QKV (q, K/V rows) on the GPU's
    # own x_out, so that an admissible difference in x_out is not counted
    # again in the next layer's q
    failures = []
    for l in sorted(subset):
        fuse = l + 1 < L
        i = inputs[l]
        Wl = oio.np_weights(Ws[l])
        r = ol.layer_forward(oio.oracle_cfg(cfgs[l]), Wl, oio.np64(i["x"]), oio.np64(i["k"]), oio.np64(i["v"]),
                             ctx, q_in=None if i["q"] is None else oio.np64(i["q"]), first_layer=(l == 0))
        g = outputs[l]
        extra = 0.0
        if moe:
            r["router_abs"] = H.router_abs(r, Wl["w_router"])
            # NVFP4 decisions next to a rounding boundary (the oracle's bound,
            # as in the ragged single-layer tests)
            extra = 3.0 * oio.flip_tolerance_fast(cfgs[l], Wl, r)[:, None]
        if fuse:
            nW = oio.np_weights({n: Ws[l + 1][n] for n in ("attn_norm_w", "w_qkv")})
            qn, kn, vn = ol.qkv_project(g["x_out"].double().numpy(), nW["attn_norm_w"], nW["w_qkv"],
                                        cfgs[l]["n_q_heads"], cfgs[l]["n_kv_heads"], cfgs[l]["head_dim"])
            r.update(q_next=qn, k_next=kn, v_next=vn)
        try:
            H.compare_single(g, r, T, ctx, fuse_next=fuse, moe=moe, x_extra=extra)
        except AssertionError as e:
            failures.append("layer %d: %s" % (l, e))
    assert not failures, "\n".join(failures)


def test_dense_draft_stack(cuda_lib):
    """5 dense GQA layers (ctx 4096, global), every layer against the oracle."""
    work = synth.make_workload("dense_draft_stack", device="cuda")
    _check_stack(cuda_lib, work, subset=set(range(5)))


def test_tiny_stack_mixed_windows(cuda_lib):
    """4 tiny MoE layers with windows 32, global, 16, global; every layer."""
    wl = dict(synth.WORKLOADS["tiny_layer"], layers=4, T=8, ctx=90)
    work = synth.make_workload(wl, device="cpu")
    for l, win in enumerate((32, 0, 16, 0)):
        work["cfgs"][l] = dict(work["cfgs"][l], window=win)
    for key in ("Ws", "caches", "x_in"):
        work[key] = H.to_device(work[key], "cuda")
    _check_stack(cuda_lib, work, subset=set(range(4)))


def test_moe_stack_62_layers(cuda_lib):
    """The full 62-layer MoE stack (46 sliding-window / 16 global layers, ctx
    16384): all 62 layers chained bit for bit against one-at-a-time launches,
    and against the oracle on the first layers (prologue, both window kinds),
    a middle pair, and the tail 59 (global), 60 (sliding window) and 61
    (global, the last layer: no fused next QKV)."""
    work = synth.make_workload("moe_stack", device="cuda")
    assert [c["window"] for c in work["cfgs"]].count(0) == 16
    _check_stack(cuda_lib, work, subset={0, 1, 3, 30, 31, 59, 60, 61})


def _run_stack(binding, work, extra_flags):
    """One PDL-chained stack step on fresh copies of the caches; returns the
    output, every layer's caches and router indices."""
    cfgs, Ws = work["cfgs"], work["Ws"]
    L = len(Ws)
    T, ctx = work["wl"]["T"], work["wl"]["ctx"]
    k = work["wl"].get("top_k", 1)
    max_ctx = work["caches"][0][0].shape[0]
    layers = []
    try:
        for l in range(L):
            fuse = l + 1 < L
            flags = (binding.MK_FIRST_LAYER if l == 0 else 0) | (binding.MK_FUSE_NEXT_QKV if fuse else 0)
            if fuse:
                flags |= extra_flags
            layers.append(H.make_layer(binding, cfgs[l], Ws[l], flags, max_ctx,
                                       next_W=Ws[l + 1] if fuse else None))
        stack = binding.mk_stack_create(layers)
        kcs = [c[0].clone() for c in work["caches"]]
        vcs = [c[1].clone() for c in work["caches"]]
        out = torch.zeros_like(work["x_in"][:T])
        idx = torch.full((L, T, k), -1, dtype=torch.int32, device="cuda")
        binding.mk_stack_step(stack, binding.make_stack_io(T, ctx, work["x_in"][:T].contiguous(), out,
                                                           kcs, vcs, topk_idx_out=idx))
        torch.cuda.synchronize()
        st = binding.mk_stack_status(stack)
        binding.mk_stack_destroy(stack)
    finally:
        for lay in layers:
            binding.mk_layer_destroy(lay)
    assert st == 0
    return out, kcs, vcs, idx


def test_next_layer_kv_prefetch_changes_no_output(cuda_lib):
    """MK_PREFETCH_NEXT_KV only fetches the next layer's old K/V rows into L2:
    a stack with it (4 tiny MoE layers, windows 32, global, 16, global, so both
    kinds of visible range are fetched) gives the same output, caches and
    router indices, bit for bit, as the stack without it."""
    wl = dict(synth.WORKLOADS["tiny_layer"], layers=4, T=8, ctx=90)
    work = synth.make_workload(wl, device="cpu")
    for l, win in enumerate((32, 0, 16, 0)):
        work["cfgs"][l] = dict(work["cfgs"][l], window=win)
    for key in ("Ws", "caches", "x_in"):
        work[key] = H.to_device(work[key], "cuda")
    base = _run_stack(cuda_lib, work, 0)
    pref = _run_stack(cuda_lib, work, cuda_lib.MK_PREFETCH_NEXT_KV)
    assert torch.equal(base[0], pref[0])
    for l in range(4):
        assert torch.equal(base[1][l], pref[1][l]) and torch.equal(base[2][l], pref[2][l]), "layer %d" % l
    assert torch.equal(base[3], pref[3])
