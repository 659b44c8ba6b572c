"""rg_out_prod_noalloc: the entry point for callers that cannot allocate.

It must give what rg_out_prod gives (same kernels, scratch in a fixed device
array instead of allocated memory) on consecutive calls that reuse the shared
scratch, and must refuse a problem whose scratch would not fit, without
touching dX.  This file is collected last, so that a run that stops at its
first failure has already run every other test; it also passes when run on
its own in a fresh process (the first call on the device sets up the
scratch's address).
"""
import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _case(wtype, N, K, T, seed, beta):
    W = inputs.gen_weight(wtype, N, K, seed=seed, stream=1)
    dY = inputs.normal_f32(seed, 2, T * N, 1e-3).reshape(T, N)
    dX0 = inputs.normal_f32(seed, 3, T * K, 1e-3).reshape(T, K)
    return W, dY, dX0


def test_noalloc_matches_rg_out_prod_on_consecutive_calls(rg):
    dev = torch.device("cuda:0")
    s = torch.cuda.current_stream()
    # two calls in a row with different shapes: the second reuses the scratch
    # the first left behind (a ragged single-CTA-tile case, then pair tiles)
    cases = [(inputs.Q4_K, 1000, 768, 520, 21, 0.0), (inputs.Q8_0, 4096, 4096, 1300, 22, 1.0)]
    outs = []
    for wtype, N, K, T, seed, beta in cases:
        W, dY, dX0 = _case(wtype, N, K, T, seed, beta)
        Wt, dYt = torch.from_numpy(W).to(dev), torch.from_numpy(dY).to(dev)
        a = torch.from_numpy(dX0).to(dev)
        b = torch.from_numpy(dX0).to(dev)
        rg.check(rg.rg_out_prod(wtype, Wt, N, K, dYt, T, a, beta, s), "rg_out_prod")
        rg.check(rg.rg_out_prod_noalloc(wtype, Wt, N, K, dYt, T, b, beta, s), "rg_out_prod_noalloc")
        rg.check(rg.rg_check(s), "rg_check")
        outs.append((wtype, N, K, T, beta, W, dY, dX0, a.cpu().numpy(), b.cpu().numpy()))
    for wtype, N, K, T, beta, W, dY, dX0, ref_gpu, got in outs:
        Wd = oracle.dequant(wtype, W, N, K)
        bnd = oracle.abs_bound(dY, Wd)
        lim = 5e-3 * bnd + 1e-7 + np.abs(beta * dX0) * 2.0 ** -24
        assert np.all(np.abs(got.astype(np.float64) - ref_gpu) <= lim)
        ref = oracle.out_prod(wtype, W, N, K, dY, T, dX0, beta, Wd=Wd)
        assert np.all(np.abs(got.astype(np.float64) - ref) <= lim)


def test_noalloc_small_t_matches_rg_out_prod_on_consecutive_calls(rg):
    """The small-T variant through the fixed scratch: one dY row over a
    14336-row Q4_K weight (rows split over CTAs, whose partial sums sit in the
    scratch before the reduction adds them), then four rows through the
    warp-level MMA consumer, which again leaves partial sums there."""
    dev = torch.device("cuda:0")
    s = torch.cuda.current_stream()
    cases = [(inputs.Q4_K, 14336, 4096, 1, 23, 0.0), (inputs.Q4_K, 4096, 4096, 4, 24, 1.0)]
    outs = []
    for wtype, N, K, T, seed, beta in cases:
        assert rg.rg_select_variant(wtype, N, K, T) == rg.RG_VARIANT_SMALLT
        info = rg.rg_plan_info()
        rg.check(rg.rg_plan(0, wtype, N, K, T, info), "rg_plan")
        assert info.n_splits > 1 and 0 < info.workspace_bytes <= rg.RG_NOALLOC_SCRATCH_BYTES
        W, dY, dX0 = _case(wtype, N, K, T, seed, beta)
        Wt, dYt = torch.from_numpy(W).to(dev), torch.from_numpy(dY).to(dev)
        a = torch.from_numpy(dX0).to(dev)
        b = torch.from_numpy(dX0).to(dev)
        rg.check(rg.rg_out_prod(wtype, Wt, N, K, dYt, T, a, beta, s), "rg_out_prod")
        rg.check(rg.rg_out_prod_noalloc(wtype, Wt, N, K, dYt, T, b, beta, s), "rg_out_prod_noalloc")
        rg.check(rg.rg_check(s), "rg_check")
        outs.append((wtype, N, K, T, beta, W, dY, dX0, a.cpu().numpy(), b.cpu().numpy()))
    for wtype, N, K, T, beta, W, dY, dX0, ref_gpu, got in outs:
        # same kernels, same plan: the same fixed-order sums
        assert np.array_equal(got, ref_gpu)
        Wd = oracle.dequant(wtype, W, N, K)
        lim = 5e-3 * oracle.abs_bound(dY, Wd) + 1e-7 + np.abs(beta * dX0) * 2.0 ** -24
        ref = oracle.out_prod(wtype, W, N, K, dY, T, dX0, beta, Wd=Wd)
        assert np.all(np.abs(got.astype(np.float64) - ref) <= lim)


def test_noalloc_rejects_oversized_scratch_without_launching(rg):
    dev = torch.device("cuda:0")
    s = torch.cuda.current_stream()
    N, K, T = 4096, 256, 8192          # 8192 * 4096 * 2 B = 64 MiB > 32 MiB of scratch
    assert T * N * 2 > rg.RG_NOALLOC_SCRATCH_BYTES
    W = torch.zeros(N * inputs.row_bytes(inputs.Q8_0, K), dtype=torch.uint8, device=dev)
    dY = torch.zeros((T, N), device=dev)
    dX = torch.full((T, K), 7.0, device=dev)
    assert rg.rg_out_prod_noalloc(inputs.Q8_0, W, N, K, dY, T, dX, 0.0, s) == rg.RG_ERR_ARG
    rg.check(rg.rg_check(s))
    assert bool(torch.all(dX == 7.0))
