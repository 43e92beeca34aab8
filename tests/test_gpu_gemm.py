"""The batched prefill's tensor-core GEMM (tcgen05.mma with TMA-staged
operands, FP32 accumulators in TMEM) against an FP64 product on the same FP16
inputs, through its plain-store epilogue (needs a GB300)."""
import ctypes as C

import numpy as np
import pytest
import torch

from conftest import cuda_available

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    L = pm.lib()
    L.lfg_gemm_test.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                C.c_void_p, C.c_void_p, C.c_void_p]
    L.lfg_gemm_test.restype = C.c_int
    return L


def _split(x):
    hi = x.to(torch.float16)
    lo = (x - hi.to(torch.float32)).to(torch.float16)
    return hi, lo


@pytest.mark.parametrize("M,N,K,bn,splits", [(1, 128, 64, 128, 1), (100, 256, 192, 128, 1), (128, 384, 2560, 128, 1),
                                             (300, 512, 2560, 256, 1), (257, 256, 8192, 256, 1),
                                             (1024, 3840, 2560, 128, 1), (511, 2560, 2560, 256, 3),
                                             (511, 2560, 8192, 128, 2), (130, 256, 1024, 256, 16)])
def test_split_fp16_gemm_matches_fp64(lib, M, N, K, bn, splits):
    """Ragged row counts (TMA zero-fills the rows past M), several K stages
    round the shared-memory ring, both tile widths, and split-K with the
    partials summed in split order by the last CTA of each tile."""
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K)
    x = torch.randn(M, K, device="cuda", generator=g)
    w = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.float16)
    xh, xl = _split(x)
    y = torch.full((M, N), float("nan"), device="cuda")
    tiles = (N // bn) * ((M + 127) // 128)
    part = torch.empty(tiles * splits * 128 * bn, device="cuda")
    cnt = torch.zeros(tiles, dtype=torch.int32, device="cuda")
    rc = lib.lfg_gemm_test(xh.data_ptr(), xl.data_ptr(), w.data_ptr(), M, N, K, bn, splits, part.data_ptr(),
                           cnt.data_ptr(), y.data_ptr())
    assert rc == 0
    assert int(cnt.abs().sum()) == 0, "tile counters must be left at zero"
    ref = (xh.double() + xl.double()) @ w.double().T
    bound = (x.abs().double() @ w.abs().double().T) * (K * 2.0 ** -23) + 1e-30
    err = (y.double() - ref).abs()
    assert torch.isfinite(y).all()
    assert bool((err <= bound).all()), f"max err {err.max().item():.3g}, worst ratio {(err / bound).max().item():.3g}"
    if splits > 1:
        # the partials are added in split order whichever CTA finishes last: same bits every run
        y2 = torch.full_like(y, float("nan"))
        assert lib.lfg_gemm_test(xh.data_ptr(), xl.data_ptr(), w.data_ptr(), M, N, K, bn, splits, part.data_ptr(),
                                 cnt.data_ptr(), y2.data_ptr()) == 0
        assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    # the split keeps about 22 bits of x: the product equals the FP32-input product closely
    exact = x.double() @ w.double().T
    assert (y.double() - exact).abs().max().item() <= 1e-4 * exact.abs().max().item()
