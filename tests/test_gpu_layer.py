"""GPU parity of the persistent decode layer against the oracle (all through
the C ABI), on seeded synthetic inputs of the five workloads and of ragged
and edge-case sizes."""

import numpy as np
import pytest
import torch

from moe_decode_layer_persistent_gb300 import synth
import layer_harness as H
import oracle_io as oio
from oracle import layer as ol

pytestmark = pytest.mark.gpu


def _single(binding, name, dev, T=None, ctx=None, fuse=False, renorm=False, flips=False, **kw):
    """One layer on the GPU vs the oracle.  flips: widen the x_out bound of
    each token by three times the largest change one admissible NVFP4
    activation decision makes there (oracle-derived, see
    oracle_io.flip_tolerance_fast): for ragged/edge sizes, where a handful of
    one-ulp differences in the expert inputs select the other NVFP4 code."""
    work, Wn = H.prepare(name, dev, T=T, ctx=ctx, **kw)
    g = H.run_single_layer(binding, work, fuse_next=fuse, renorm=renorm)
    r = H.oracle_single_layer(work, fuse_next=fuse, Wn=Wn, renorm=renorm)
    wl = work["wl"]
    extra = 0.0
    if flips:
        extra = 3.0 * oio.flip_tolerance_fast(work["cfgs"][0], Wn, r)[:, None]
    return H.compare_single(g, r, wl["T"], wl["ctx"], fuse_next=fuse, moe=wl["ffn"] == "moe",
                            x_extra=extra)


def test_tiny_layer(cuda_lib):
    """1 token, 128 past positions, 16 experts top-2, head_dim 64."""
    _single(cuda_lib, "tiny_layer", "host")


@pytest.mark.parametrize("T,ctx", [(16, 100), (3, 0), (5, 1), (16, 128), (7, 257)])
def test_tiny_shapes_ragged(cuda_lib, T, ctx):
    _single(cuda_lib, "tiny_layer", "host", T=T, ctx=ctx, flips=True)


def test_tiny_renormalised_topk(cuda_lib):
    _single(cuda_lib, "tiny_layer", "host", T=4, ctx=50, renorm=True, flips=True)


def test_tiny_odd_down_tile_count(cuda_lib):
    """pooled_dim 384: three 128-row down tiles per expert, so the down phase
    has a unit of two tiles and a unit of one; and a gate/up K of 384 (one
    full and one half NVFP4 K-block)."""
    wl = dict(synth.WORKLOADS["tiny_layer"], pooled_dim=384, T=8, ctx=100)
    _single(cuda_lib, wl, "host", flips=True)


def test_swa_layer(cuda_lib):
    """16 verify tokens, context 8192, window 2048, 256 experts top-8."""
    _single(cuda_lib, "swa_layer", "cuda")


@pytest.mark.parametrize("T,ctx", [(1, 8192), (5, 0), (16, 1), (9, 2047), (16, 2100)])
def test_swa_shapes_ragged(cuda_lib, T, ctx):
    """Ragged token counts and contexts at the full expert shapes, including an
    empty history, windows cut at the first position and the window edge."""
    _single(cuda_lib, "swa_layer", "cuda", T=T, ctx=ctx, flips=True)


def test_layer_with_q_in(cuda_lib):
    """A layer that is not the first of a chain: q and rows ctx..ctx+T-1 of the
    caches come from the previous launch (here: drawn)."""
    work = synth.make_workload("swa_layer", device="cuda", ctx=3000)
    T, ctx = 16, 3000
    c = work["cfgs"][0]
    q_in = synth.randn((T, c["n_q_heads"] * c["head_dim"]), work["seed"], 7, "q_in", "cuda").bfloat16()
    for cache, nm in zip(work["caches"][0], ("k_new", "v_new")):
        cache[ctx:ctx + T] = synth.randn((T, c["n_kv_heads"], c["head_dim"]), work["seed"], 7, nm,
                                         "cuda").bfloat16()
    Wn, _ = oio.enforce_margin_single(work, q_np=oio.np64(q_in).reshape(T, c["n_q_heads"], -1),
                                      first_layer=False)
    g = H.run_single_layer(cuda_lib, work, first_layer=False, q_in=q_in)
    kc, vc = (oio.np64(t) for t in work["caches"][0])
    r = ol.layer_forward(oio.oracle_cfg(c), Wn, oio.np64(work["x_in"]), kc, vc, ctx,
                         q_in=oio.np64(q_in), first_layer=False)
    r["router_abs"] = H.router_abs(r, Wn["w_router"])
    H.compare_single(g, r, T, ctx)


def test_swa_layer_short_context_equals_global(cuda_lib):
    """ctx + T <= window: the sliding-window layer equals the global one."""
    work, Wn = H.prepare("swa_layer", "cuda", ctx=2000)
    g_swa = H.run_single_layer(cuda_lib, work)
    work["cfgs"][0] = dict(work["cfgs"][0], window=0)
    g_glob = H.run_single_layer(cuda_lib, work)
    assert torch.equal(g_swa["x_out"], g_glob["x_out"])


def test_global_layer_fused_next_qkv(cuda_lib):
    """Context 32768, global attention, fused next-layer QKV + KV write."""
    _single(cuda_lib, "global_layer_fused", "cuda", fuse=True)


def test_dense_layer(cuda_lib):
    _single(cuda_lib, "dense_draft_stack", "cuda", layers=1)


def test_repeated_steps_and_determinism(cuda_lib):
    work, Wn = H.prepare("tiny_layer", "host", T=16, ctx=60)
    c = work["cfgs"][0]
    kc, vc = (t.clone() for t in work["caches"][0])
    layer = H.make_layer(cuda_lib, c, work["Ws"][0], cuda_lib.MK_FIRST_LAYER, kc.shape[0])
    outs = []
    for _ in range(3):
        x_out = torch.zeros_like(work["x_in"])
        io = cuda_lib.make_step_io(16, 60, work["x_in"], x_out, kc, vc)
        cuda_lib.mk_decode_step(layer, io)
        torch.cuda.synchronize()
        outs.append(x_out.clone())
    assert cuda_lib.mk_layer_status(layer) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    cuda_lib.mk_layer_destroy(layer)


def _predicted(idx_prev, n, E):
    """The previous step's n most-used experts, an equal count going to the
    lower index (experts with no token are never predicted)."""
    cnt = np.bincount(np.asarray(idx_prev).ravel(), minlength=E)
    order = sorted(range(E), key=lambda e: (-cnt[e], e))
    return [e for e in order[:n] if cnt[e] > 0]


def test_expert_prefetch_statistics(cuda_lib):
    """Each step prefetches the previous step's most-used experts; the layer
    counts steps, predicted, active and hit experts.  The host recomputes the
    prediction from the previous step's top-k indices."""
    N = 5
    work, Wn = H.prepare("tiny_layer", "host", T=16, ctx=60)
    other = synth.make_workload("tiny_layer", device="cpu", T=16, ctx=60, seed=synth.SEED_BASE + 77)
    c = work["cfgs"][0]
    E, k = c["n_experts"], c["top_k"]
    kc, vc = (t.clone() for t in work["caches"][0])
    cfg = cuda_lib.make_config(c, flags=cuda_lib.MK_FIRST_LAYER, max_ctx=kc.shape[0], prefetch_experts=N)
    layer = cuda_lib.mk_layer_create(cfg, work["Ws"][0])
    xs = [work["x_in"], work["x_in"], other["x_in"][:16].to("cuda")]
    idxs = []
    for x in xs:
        x_out = torch.zeros_like(x)
        idx = torch.full((16, k), -1, dtype=torch.int32, device="cuda")
        io = cuda_lib.make_step_io(16, 60, x.contiguous(), x_out, kc, vc, topk_idx_out=idx)
        cuda_lib.mk_decode_step(layer, io)
        torch.cuda.synchronize()
        idxs.append(idx.cpu().numpy())
    assert cuda_lib.mk_layer_status(layer) == 0
    st = cuda_lib.mk_layer_prefetch_stats(layer)
    cuda_lib.mk_layer_destroy(layer)
    want = dict(steps=3, predicted=0, active=0, hits=0)
    for s, idx in enumerate(idxs):
        active = set(idx.ravel().tolist())
        want["active"] += len(active)
        if s > 0:
            pred = _predicted(idxs[s - 1], N, E)
            want["predicted"] += len(pred)
            want["hits"] += len(active & set(pred))
    assert st == want, (st, want)
    assert st["hits"] >= len(_predicted(idxs[0], N, E))  # step 2 repeats step 1's routing


def test_step_rejects_bad_arguments_before_launch(cuda_lib):
    """Malformed steps are refused on the host (MK_ERR_INVALID_ARG) before
    anything is launched: a context whose end overflows, misaligned top-k
    outputs, token counts outside 1..max_tokens, output aliasing input."""
    work, _ = H.prepare("tiny_layer", "host", T=4, ctx=30, enforce=False)
    c = work["cfgs"][0]
    kc, vc = (t.clone() for t in work["caches"][0])
    layer = H.make_layer(cuda_lib, c, work["Ws"][0], cuda_lib.MK_FIRST_LAYER, kc.shape[0])
    x = work["x_in"][:4].contiguous()
    y = torch.zeros_like(x)
    idx = torch.zeros((4, c["top_k"] + 1), dtype=torch.int32, device="cuda")
    bad = [cuda_lib.make_step_io(4, 2**31 - 1, x, y, kc, vc),
           cuda_lib.make_step_io(4, 30, x, y, kc, vc, topk_idx_out=idx.data_ptr() + 2),
           cuda_lib.make_step_io(0, 30, x, y, kc, vc),
           cuda_lib.make_step_io(17, 30, x, y, kc, vc),
           cuda_lib.make_step_io(4, 30, x, x, kc, vc)]
    try:
        for io in bad:
            with pytest.raises(cuda_lib.MkError) as e:
                cuda_lib.mk_decode_step(layer, io)
            assert e.value.status == 1
        torch.cuda.synchronize()
        assert cuda_lib.mk_layer_status(layer) == 0
    finally:
        cuda_lib.mk_layer_destroy(layer)


def test_bounded_wait_reports_timeout_and_recovers(cuda_lib):
    """A wait limit of 1 ns makes the first wait that is not already satisfied
    give up: the kernel returns, the status reads MK_ERR_TIMEOUT, the context
    stays usable, and after clearing the status the layer runs normally."""
    work, Wn = H.prepare("tiny_layer", "host", T=4, ctx=30)
    c = work["cfgs"][0]
    kc, vc = (t.clone() for t in work["caches"][0])
    layer = H.make_layer(cuda_lib, c, work["Ws"][0], cuda_lib.MK_FIRST_LAYER, kc.shape[0],
                         timeout_ns=1)
    x_out = torch.zeros_like(work["x_in"])
    io = cuda_lib.make_step_io(4, 30, work["x_in"], x_out, kc, vc)
    cuda_lib.mk_decode_step(layer, io)
    torch.cuda.synchronize()
    assert cuda_lib.mk_layer_status(layer) == 5
    cuda_lib.mk_layer_destroy(layer)
    g = H.run_single_layer(cuda_lib, work)
    r = H.oracle_single_layer(work, Wn=Wn)
    H.compare_single(g, r, 4, 30)


# ------------------------------------------------------------ token trees

# 16 verify tokens as a tree (parent indices, -1 = a root after the prefix):
# three branches of different depths, siblings at several levels.
TREE_PARENTS = [-1, 0, 0, 0, 1, 1, 2, 4, 4, 5, 6, 7, 3, 12, 9, 13]


def tree_masks(parents):
    m = []
    for i, p in enumerate(parents):
        m.append((1 << i) | (m[p] if p >= 0 else 0))
    return m


def _tree_single(binding, name, dev, T, ctx, tree, flips=False):
    work, Wn = H.prepare(name, dev, T=T, ctx=ctx, enforce=False)
    c = work["cfgs"][0]
    # margin on the tree's router input (the oracle decides)
    if c["ffn"] == "moe":
        Wn, _ = oio.enforce_margin_single(work, tree=tree)
    g = H.run_single_layer(binding, work, tree_mask=tree)
    r = H.oracle_single_layer(work, Wn=Wn, tree=tree)
    extra = 3.0 * oio.flip_tolerance_fast(c, Wn, r)[:, None] if flips else 0.0
    return H.compare_single(g, r, T, ctx, moe=c["ffn"] == "moe", x_extra=extra)


def test_tree_mask_of_the_chain_is_the_default(cuda_lib):
    """The causal chain passed as an explicit tree gives the same bits as no
    mask."""
    work, _ = H.prepare("swa_layer", "cuda", ctx=3000, enforce=False)
    a = H.run_single_layer(cuda_lib, work)
    b = H.run_single_layer(cuda_lib, work, tree_mask=tree_masks(list(range(-1, 15))))
    for key in ("x_out", "k_cache", "v_cache"):
        assert torch.equal(a[key], b[key]), key


def test_tree_verification_swa_layer(cuda_lib):
    """Token-tree verification at the full shapes: 16 tokens in a tree, context
    8192, window 2048, against the oracle's tree attention."""
    _tree_single(cuda_lib, "swa_layer", "cuda", 16, 8192, tree_masks(TREE_PARENTS))


def test_tree_verification_tiny_short_window(cuda_lib):
    """A tree whose depth reaches past a short window (window 4): ancestors more
    than 3 levels up are cut off like prefix positions."""
    work_parents = [-1, 0, 1, 2, 3, 4, 1, 6]       # a chain of depth 5 and a side branch
    wl = dict(synth.WORKLOADS["tiny_layer"], window=4)
    work, _ = H.prepare(wl, "host", T=8, ctx=30, enforce=False)
    Wn, _ = oio.enforce_margin_single(work, tree=tree_masks(work_parents))
    g = H.run_single_layer(cuda_lib, work, tree_mask=tree_masks(work_parents))
    r = H.oracle_single_layer(work, Wn=Wn, tree=tree_masks(work_parents))
    extra = 3.0 * oio.flip_tolerance_fast(work["cfgs"][0], Wn, r)[:, None]
    H.compare_single(g, r, 8, 30, x_extra=extra)


def test_tree_masks_that_are_not_trees_are_refused(cuda_lib):
    work, _ = H.prepare("tiny_layer", "host", T=4, ctx=30, enforce=False)
    c = work["cfgs"][0]
    kc, vc = (t.clone() for t in work["caches"][0])
    layer = H.make_layer(cuda_lib, c, work["Ws"][0], cuda_lib.MK_FIRST_LAYER, kc.shape[0])
    x = work["x_in"][:4].contiguous()
    y = torch.zeros_like(x)
    bad = [[1, 3, 5, 3],       # token 3 misses itself
           [1, 3, 7, 0x18],    # token 3 holds a later token (bit 4)
           [1, 3, 6, 13],      # token 2 lists 1 but not 1's ancestor 0
           [3, 3, 7, 15]]      # token 0 holds token 1
    try:
        for m in bad:
            with pytest.raises(cuda_lib.MkError) as e:
                cuda_lib.mk_decode_step(layer, cuda_lib.make_step_io(4, 30, x, y, kc, vc, tree_mask=m))
            assert e.value.status == 1, m
        torch.cuda.synchronize()
        assert cuda_lib.mk_layer_status(layer) == 0
    finally:
        cuda_lib.mk_layer_destroy(layer)
