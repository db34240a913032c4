"""GPU checks of the layer's building blocks against the oracle: the NVFP4
quantiser (bit-exact) and one TMA + tcgen05 MMA tile (bf16 and block-scaled
NVFP4), through the library's self-test entry points."""

import numpy as np
import pytest
import torch

from oracle import numerics as n

pytestmark = pytest.mark.gpu


def _bf16_rows(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g) * torch.exp(torch.randn(rows, 1, generator=g))
    x = x.bfloat16()
    # edge rows: all zero, tiny values, exact RNE ties on the E2M1 grid
    x[0] = 0
    if rows > 2:
        x[1] = (torch.randn(K, generator=g) * 1e-30).bfloat16()
        ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * (K // 8)).bfloat16()
        x[2] = ties * torch.where(torch.arange(K) % 3 == 0, -1.0, 1.0).bfloat16()
    return x


@pytest.mark.parametrize("K", [128, 1024, 2048])
def test_quantizer_bit_exact(cuda_lib, K):
    x = _bf16_rows(64, K, K)
    xd = x.cuda()
    codes = torch.zeros(64, K // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(64, K // 16, dtype=torch.uint8, device="cuda")
    s_row = torch.zeros(64, dtype=torch.float32, device="cuda")
    cuda_lib.mk_selftest_quantize(xd, codes, scales, s_row)
    q, s, r = n.nvfp4_quantize_rows(x.double().numpy())
    assert np.array_equal(s_row.cpu().numpy(), r)
    assert np.array_equal(scales.cpu().numpy(), s)
    assert np.array_equal(codes.cpu().numpy(), q)


@pytest.mark.parametrize("K", [64, 256, 512])
def test_mma_tile_bf16(cuda_lib, K):
    g = torch.Generator().manual_seed(K)
    a = torch.randn(128, K, generator=g).bfloat16()
    b = torch.randn(16, K, generator=g).bfloat16()
    out = torch.zeros(16, 128, dtype=torch.float32, device="cuda")
    cuda_lib.mk_selftest_mma(0, a.cuda(), None, b.cuda(), None, K, out)
    want = b.double().numpy() @ a.double().numpy().T
    got = out.cpu().double().numpy()
    assert np.allclose(got, want, rtol=1e-5, atol=1e-4 * np.abs(want).max())


def _fp4_operand(rows, K, seed, scale_mode):
    g = torch.Generator().manual_seed(seed)
    codes = torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.uint8)
    if scale_mode == "one":
        scales = torch.full((rows, K // 16), 0x38, dtype=torch.uint8)        # 1.0
    else:
        scales = torch.randint(0x28, 0x48, (rows, K // 16), generator=g, dtype=torch.uint8)
    return codes, scales


@pytest.mark.parametrize("K,mode", [(256, "one"), (1024, "one"), (256, "rand_a"),
                                    (256, "rand"), (1024, "rand"), (128, "rand"), (64, "rand")])
def test_mma_tile_nvfp4(cuda_lib, K, mode):
    ac, as_ = _fp4_operand(128, K, 1 + K, "one" if mode == "one" else "rand")
    bc, bs = _fp4_operand(16, K, 2 + K, "rand" if mode == "rand" else "one")
    out = torch.zeros(16, 128, dtype=torch.float32, device="cuda")
    cuda_lib.mk_selftest_mma(1, ac.cuda(), as_.cuda(), bc.cuda(), bs.cuda(), K, out)
    A = n.nvfp4_dequantize(ac.numpy(), as_.numpy(), np.float32(1))
    B = n.nvfp4_dequantize(bc.numpy(), bs.numpy(), np.float32(1))
    want = B @ A.T
    got = out.cpu().double().numpy()
    assert np.allclose(got, want, rtol=1e-5, atol=1e-5 * np.abs(want).max())


def test_sync_microbenchmark(cuda_lib):
    """Intra-GPU synchronisation costs (one flag hop between two SMs, one hop
    of a value that is its own signal, one acquire poll, one idle fence) are
    measured without any poll giving up, and fall in a plausible range."""
    got = {m: cuda_lib.mk_selftest_sync(m, 2000) for m in cuda_lib.SYNC_MODES}
    for m, ns in got.items():
        assert 1.0 < ns < 1e5, (m, ns)
    assert got["acquire_poll"] < got["flag_hop"], got

