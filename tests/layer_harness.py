"""Shared harness of the GPU parity tests: run one layer (or a stack) through
the C ABI on seeded synthetic inputs, run the oracle on the same inputs, and
compare with the tolerances of the layer's contract:
  router expert indices bit-exact;
  x_out, written K/V rows and next-layer q: max |err| <= 2e-2 * RMS(ref) and
  cosine >= 0.9995.
"""

import numpy as np
import torch

from moe_decode_layer_persistent_gb300 import synth
import oracle_io as oio
from oracle import layer as ol

ABS_TOL = 2e-2
COS_TOL = 0.9995


def metrics(got, ref):
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    rms = float(np.sqrt(np.mean(ref * ref)))
    maxabs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    den = float(np.linalg.norm(got) * np.linalg.norm(ref))
    cos = float(np.dot(got, ref) / den) if den > 0 else (1.0 if maxabs == 0 else 0.0)
    return dict(rms=rms, maxabs=maxabs, rel=maxabs / rms if rms > 0 else maxabs, cos=cos)


def bf16_ulp(x):
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.frexp(np.where(x > 0, x, 1.0))[1]
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def assert_close(name, got, ref, extra_abs=0.0):
    """max |got - ref| <= 2e-2 * RMS(ref) and cosine >= 0.9995.

    Both sides store bfloat16, so two correct evaluations can differ by one
    unit in the last place of an element; where that unit exceeds 2e-2 * RMS
    (elements above ~4 * RMS), the element's own ulp is the bound.
    `extra_abs` widens the bound by an amount derived from the oracle (see
    flip_tolerance)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = metrics(got, ref)
    assert np.all(np.isfinite(got)), name + ": non-finite"
    bound = np.maximum(ABS_TOL * m["rms"], bf16_ulp(ref)) + extra_abs
    over = np.abs(got - ref) > bound
    m["n_over"] = int(over.sum())
    assert not over.any() and m["cos"] >= COS_TOL, "%s: %s" % (name, m)
    return m


def weights_for_lib(W):
    """The weight dict as the C ABI expects it (device tensors)."""
    return dict(W)


def make_layer(binding, wl, W, flags, max_ctx, next_W=None, window=None, timeout_ns=0):
    cfg = binding.make_config(wl, flags=flags, max_ctx=max_ctx, window=window,
                              timeout_ns=timeout_ns)
    wd = weights_for_lib(W)
    if next_W is not None:
        wd["next_attn_norm_w"] = next_W["attn_norm_w"]
        wd["next_w_qkv"] = next_W["w_qkv"]
    return binding.mk_layer_create(cfg, wd)


def run_single_layer(binding, work, T=None, ctx=None, fuse_next=False, first_layer=True,
                     q_in=None, renorm=False, stream=None, keep_layer=False, tree_mask=None):
    """One mk_decode_step on device tensors of `work` (a synth.make_workload
    result on cuda).  Returns host copies of every output."""
    wl = work["wl"]
    c = work["cfgs"][0]
    W = work["Ws"][0]
    T = wl["T"] if T is None else T
    ctx = wl["ctx"] if ctx is None else ctx
    kc, vc = (t.clone() for t in work["caches"][0])
    max_ctx = kc.shape[0]
    flags = (binding.MK_FIRST_LAYER if first_layer else 0) | \
        (binding.MK_FUSE_NEXT_QKV if fuse_next else 0) | (binding.MK_TOPK_RENORM if renorm else 0)
    nxt = work["next"] if fuse_next else None
    layer = make_layer(binding, c, W, flags, max_ctx, next_W=nxt)
    x_in = work["x_in"][:T].contiguous()
    x_out = torch.zeros_like(x_in)
    dev = x_in.device
    k = c.get("top_k", 0)
    idx = torch.full((T, max(k, 1)), -1, dtype=torch.int32, device=dev)
    wts = torch.zeros((T, max(k, 1)), dtype=torch.float32, device=dev)
    q_out = nkc = nvc = None
    if fuse_next:
        nkc, nvc = (t.clone() for t in (nxt["k_cache"], nxt["v_cache"]))
        q_out = torch.zeros((T, c["n_q_heads"] * c["head_dim"]), dtype=torch.bfloat16, device=dev)
    io = binding.make_step_io(T, ctx, x_in, x_out, kc, vc, q_in=q_in, next_k_cache=nkc,
                              next_v_cache=nvc, q_out=q_out,
                              topk_idx_out=idx if k else None, topk_w_out=wts if k else None,
                              tree_mask=tree_mask)
    binding.mk_decode_step(layer, io, stream)
    torch.cuda.synchronize()
    st = binding.mk_layer_status(layer)
    out = dict(status=st, x_out=x_out.cpu(), k_cache=kc.cpu(), v_cache=vc.cpu(),
               idx=idx.cpu().numpy() if k else None, w=wts.cpu().numpy() if k else None)
    if fuse_next:
        out.update(q_out=q_out.cpu(), next_k_cache=nkc.cpu(), next_v_cache=nvc.cpu())
    if keep_layer:
        out["layer"] = layer
    else:
        binding.mk_layer_destroy(layer)
    return out


def oracle_single_layer(work, T=None, ctx=None, fuse_next=False, Wn=None, renorm=False, tree=None):
    wl = work["wl"]
    c = work["cfgs"][0]
    T = wl["T"] if T is None else T
    ctx = wl["ctx"] if ctx is None else ctx
    Wn = oio.np_weights(work["Ws"][0]) if Wn is None else Wn
    kc, vc = (oio.np64(t) for t in work["caches"][0])
    nxt = None
    nkc = nvc = None
    if fuse_next:
        nxt = oio.np_weights({k: v for k, v in work["next"].items() if k in ("attn_norm_w", "w_qkv")})
        nkc, nvc = oio.np64(work["next"]["k_cache"]), oio.np64(work["next"]["v_cache"])
    r = ol.layer_forward(oio.oracle_cfg(c), Wn, oio.np64(work["x_in"][:T]), kc, vc, ctx,
                         next_W=nxt, next_k_cache=nkc, next_v_cache=nvc, renorm=renorm, tree=tree)
    if "w_router" in Wn and "logits" in r:
        r["router_abs"] = router_abs(r, Wn["w_router"])
    return r


# Rounding of the GPU's float32 router logits: the products h_i w_i are exact
# in float32 (bf16 x bf16), and every path of the GPU's summation tree over
# K = hidden inputs (the tensor core's K-steps within a 512-input split-K
# unit, the four MMA lanes' partials, then the split-K partials) holds at most
# 8 + 2 + 8 sequential roundings plus the tensor core's own: at most 32, so
# |logit_gpu - logit_exact| <= 32 u sum_i |h_i w_i| (u = 2^-24, first order).
# The oracle's float32 logit is within u |logit| of the exact one.
ORDER_ROUNDINGS = 32
U32 = 2.0 ** -24


def router_abs(ref, w_router):
    """sum_i |h_ti W_r[e, i]| per token and expert, from the oracle's h."""
    return np.abs(np.asarray(ref["h"], dtype=np.float64)) @ np.abs(np.asarray(w_router, dtype=np.float64)).T


def check_router(g_idx, g_w, r_idx, r_w, r_logits, abs_sum):
    """Router contract: the chosen expert SET of every token bit-exact (the
    margin between the k-th and (k+1)-th logit makes it unique).  The order
    inside the set is unique only where the chosen logits differ by more than
    the logits' rounding, so consecutive experts a, b of the GPU's order must
    satisfy logit(a) >= logit(b) - (e_a + e_b) in the oracle's logits, with
    e = ORDER_ROUNDINGS u sum_i |h_i w_i| + u |logit| (the float32 rounding
    bound above; abs_sum = router_abs).  The weights, matched by expert,
    within the contract bound."""
    g_idx = np.asarray(g_idx)
    assert np.array_equal(np.sort(g_idx, axis=1), np.sort(r_idx, axis=1)), (g_idx, r_idx)
    gi = g_idx.astype(np.int64)
    lg = np.take_along_axis(np.asarray(r_logits, dtype=np.float64), gi, axis=1)
    err = ORDER_ROUNDINGS * U32 * np.take_along_axis(np.asarray(abs_sum, dtype=np.float64), gi, axis=1) \
        + U32 * np.abs(lg)
    slack = err[:, :-1] + err[:, 1:]
    assert np.all(np.diff(lg, axis=1) <= slack), "router order"
    pos = np.argsort(g_idx, axis=1)
    rpos = np.argsort(r_idx, axis=1)
    gw = np.take_along_axis(np.asarray(g_w), pos, axis=1)
    rw = np.take_along_axis(np.asarray(r_w), rpos, axis=1)
    return assert_close("w", gw, rw)


def compare_single(gpu, ref, T, ctx, fuse_next=False, moe=True, x_extra=0.0):
    """Asserts the contract; returns the metrics of every compared tensor.
    x_extra: per-token widening of the x_out bound (flip_tolerance)."""
    res = {}
    assert gpu["status"] == 0, "device status %d" % gpu["status"]
    if moe:
        res["w"] = check_router(gpu["idx"], gpu["w"], ref["idx"], ref["w"], ref["logits"],
                                ref["router_abs"])
    res["x_out"] = assert_close("x_out", gpu["x_out"].double().numpy(), ref["x_out"], x_extra)
    res["k_rows"] = assert_close("k_rows", gpu["k_cache"][ctx:ctx + T].double().numpy(),
                                 ref["k_cache"][ctx:ctx + T])
    res["v_rows"] = assert_close("v_rows", gpu["v_cache"][ctx:ctx + T].double().numpy(),
                                 ref["v_cache"][ctx:ctx + T])
    # rows outside [ctx, ctx+T) untouched
    assert np.array_equal(gpu["k_cache"][:ctx].double().numpy(), ref["k_cache"][:ctx])
    if fuse_next:
        res["q_out"] = assert_close("q_out", gpu["q_out"].double().numpy(),
                                    ref["q_next"].reshape(T, -1))
        res["next_k"] = assert_close("next_k", gpu["next_k_cache"][ctx:ctx + T].double().numpy(),
                                     ref["k_next"])
        res["next_v"] = assert_close("next_v", gpu["next_v_cache"][ctx:ctx + T].double().numpy(),
                                     ref["v_next"])
    return res


def to_device(obj, device):
    if isinstance(obj, torch.Tensor):
        return obj.to(device)
    if isinstance(obj, dict):
        return {k: to_device(v, device) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return type(obj)(to_device(v, device) for v in obj)
    return obj


def prepare(work_name, device, T=None, ctx=None, layers=None, enforce=True, seed=None):
    """Synthetic workload on `device`; "host" generates on the CPU generator
    and moves the tensors to the GPU (small workloads: same values as the CPU
    tests see)."""
    gen_dev = "cpu" if device == "host" else device
    work = synth.make_workload(work_name, device=gen_dev, T=T, ctx=ctx, layers=layers, seed=seed)
    if device == "host":
        for key in ("Ws", "caches", "x_in", "next"):
            work[key] = to_device(work[key], "cuda")
    Wn = None
    if enforce and work["wl"]["ffn"] == "moe" and work["wl"]["layers"] == 1:
        Wn, _ = oio.enforce_margin_single(work)
    return work, Wn
