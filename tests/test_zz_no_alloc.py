"""The allocation-free decode step.

Callers that cannot allocate device memory (their device memory belongs to
another allocator or pool, or they must not grow their footprint after
start-up) run a layer step through mk_decode_step_noalloc, whose library
buffers live in the library's fixed static device array.  Each case runs it
twice in a row and checks both results against the regular entry point
(mk_layer_create + mk_decode_step) on the same inputs, and against the
oracle, with the parity tolerances of the other tests.  The cases cover the
MoE and dense layers, the fused next-layer QKV, and a context whose
attention split reaches the allocation-free path's cap of 32 chunks per KV
head.  Kept in a file of its own, collected last.
"""

import pytest
import torch

from moe_decode_layer_persistent_gb300 import synth
import layer_harness as H
import oracle_io as oio

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_layer"]
CASES = {
    "moe": (dict(TINY), 8, 100),
    "dense": (dict(TINY, ffn="dense", dense_inter=256), 8, 100),
    "moe_fused_next_qkv": (dict(TINY, fuse_next=True), 8, 100),
    # 2016 visible positions over 32 chunks of 64: the split's cap
    "moe_attention_split_cap": (dict(TINY), 16, 2000),
}


def _outputs(binding, work, T, ctx, noalloc):
    """One step through either entry point; host copies of every output."""
    c = work["cfgs"][0]
    W = dict(work["Ws"][0])
    fuse = work["next"] is not None
    moe = c["ffn"] == "moe"
    kc, vc = (t.clone() for t in work["caches"][0])
    x_out = torch.zeros_like(work["x_in"][:T])
    k = c.get("top_k", 1) if moe else 1
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    q_out = nkc = nvc = None
    if fuse:
        W["next_attn_norm_w"], W["next_w_qkv"] = work["next"]["attn_norm_w"], work["next"]["w_qkv"]
        nkc, nvc = (t.clone() for t in (work["next"]["k_cache"], work["next"]["v_cache"]))
        q_out = torch.zeros((T, c["n_q_heads"] * c["head_dim"]), dtype=torch.bfloat16, device="cuda")
    io = binding.make_step_io(T, ctx, work["x_in"][:T].contiguous(), x_out, kc, vc,
                              next_k_cache=nkc, next_v_cache=nvc, q_out=q_out,
                              topk_idx_out=idx if moe else None, topk_w_out=wts if moe else None)
    flags = binding.MK_FIRST_LAYER | (binding.MK_FUSE_NEXT_QKV if fuse else 0)
    cfg = binding.make_config(c, flags=flags, max_ctx=kc.shape[0])
    status = 0
    if noalloc:
        binding.mk_decode_step_noalloc(cfg, W, io)
        torch.cuda.synchronize()
    else:
        layer = binding.mk_layer_create(cfg, W)
        binding.mk_decode_step(layer, io)
        torch.cuda.synchronize()
        status = binding.mk_layer_status(layer)
        binding.mk_layer_destroy(layer)
    out = dict(status=status, x_out=x_out.cpu(), k_cache=kc.cpu(), v_cache=vc.cpu(),
               idx=idx.cpu().numpy() if moe else None, w=wts.cpu().numpy() if moe else None)
    if fuse:
        out.update(q_out=q_out.cpu(), next_k_cache=nkc.cpu(), next_v_cache=nvc.cpu())
    return out


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_step_matches_regular_step_and_oracle_twice(cuda_lib, case):
    wl, T, ctx = CASES[case]
    work, Wn = H.prepare(wl, "host", T=T, ctx=ctx)
    fuse = work["next"] is not None
    moe = wl["ffn"] == "moe"
    ref = _outputs(cuda_lib, work, T, ctx, noalloc=False)
    assert ref["status"] == 0
    r = H.oracle_single_layer(work, fuse_next=fuse, Wn=Wn)
    # ragged tiny shapes: x_out may differ where one NVFP4 decision flips
    # (a bound derived from the oracle, as in the other tiny-shape tests)
    extra = 3.0 * oio.flip_tolerance_fast(work["cfgs"][0], Wn, r)[:, None] if moe else 0.0
    names = ["x_out", "k_cache", "v_cache"] + (["q_out", "next_k_cache", "next_v_cache"] if fuse else [])
    for _ in range(2):
        got = _outputs(cuda_lib, work, T, ctx, noalloc=True)
        if moe:
            assert (got["idx"] == ref["idx"]).all()                 # router indices
        for name in names:
            H.assert_close(name, got[name].double().numpy(), ref[name].double().numpy())
        H.compare_single(got, r, T, ctx, fuse_next=fuse, moe=moe, x_extra=extra)


def test_noalloc_rejects_layers_beyond_the_scratch(cuda_lib):
    wl = synth.WORKLOADS["swa_layer"]
    cfg = cuda_lib.make_config(wl, flags=cuda_lib.MK_FIRST_LAYER, max_ctx=64)
    # shapes are checked before any weight is touched: pointers only need to be aligned
    fake = {n: 0x10000 for n in cuda_lib._WEIGHT_FIELDS}
    io = cuda_lib.make_step_io(16, 0, 0x20000, 0x30000, 0x40000, 0x50000)
    with pytest.raises(cuda_lib.MkError) as e:
        cuda_lib.mk_decode_step_noalloc(cfg, fake, io)
    assert e.value.status == 2
