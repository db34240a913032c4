"""The allocation-free decode step.

Callers that cannot allocate device memory (their device memory belongs to
another allocator or pool, or they must not grow their footprint after
start-up) run a layer step through mk_decode_step_noalloc, whose library
buffers live in the library's fixed static device array.  This test runs it
twice in a row and checks both results against the regular entry point
(mk_layer_create + mk_decode_step) on the same inputs, with the parity
tolerance of the other tests.  Kept in a file of its own, collected last.
"""

import pytest
import torch

import layer_harness as H

pytestmark = pytest.mark.gpu


def _outputs(binding, work, T, ctx, noalloc):
    c = work["cfgs"][0]
    kc, vc = (t.clone() for t in work["caches"][0])
    x_out = torch.zeros_like(work["x_in"][:T])
    idx = torch.full((T, c["top_k"]), -1, dtype=torch.int32, device="cuda")
    io = binding.make_step_io(T, ctx, work["x_in"][:T].contiguous(), x_out, kc, vc,
                              topk_idx_out=idx)
    cfg = binding.make_config(c, flags=binding.MK_FIRST_LAYER, max_ctx=kc.shape[0])
    if noalloc:
        binding.mk_decode_step_noalloc(cfg, dict(work["Ws"][0]), io)
        torch.cuda.synchronize()
    else:
        layer = binding.mk_layer_create(cfg, dict(work["Ws"][0]))
        binding.mk_decode_step(layer, io)
        torch.cuda.synchronize()
        assert binding.mk_layer_status(layer) == 0
        binding.mk_layer_destroy(layer)
    return x_out.cpu(), kc.cpu(), vc.cpu(), idx.cpu()


def test_noalloc_step_matches_regular_step_twice(cuda_lib):
    work, _ = H.prepare("tiny_layer", "host", T=8, ctx=100)
    ref = _outputs(cuda_lib, work, 8, 100, noalloc=False)
    for _ in range(2):
        got = _outputs(cuda_lib, work, 8, 100, noalloc=True)
        assert torch.equal(got[3], ref[3])                      # router indices
        for g, r, name in zip(got[:3], ref[:3], ("x_out", "k_cache", "v_cache")):
            H.assert_close(name, g.double().numpy(), r.double().numpy())


def test_noalloc_rejects_layers_beyond_the_scratch(cuda_lib):
    work = {"wl": None}
    from moe_decode_layer_persistent_gb300 import synth
    wl = synth.WORKLOADS["swa_layer"]
    cfg = cuda_lib.make_config(wl, flags=cuda_lib.MK_FIRST_LAYER, max_ctx=64)
    # shapes are checked before any weight is touched: pointers only need to be aligned
    fake = {n: 0x10000 for n in cuda_lib._WEIGHT_FIELDS}
    io = cuda_lib.make_step_io(16, 0, 0x20000, 0x30000, 0x40000, 0x50000)
    with pytest.raises(cuda_lib.MkError) as e:
        cuda_lib.mk_decode_step_noalloc(cfg, fake, io)
    assert e.value.status == 2
    del work
