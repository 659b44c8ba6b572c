"""Outputs with more than 2^31 elements: every index past the 32-bit range
(dX of the OUT_PROD, Y of the forward, rg_dequant's F32 output) is written
where it belongs.  Each case holds about 9 GB on the device at most; the
checks read back sampled rows, among them the last."""
import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

BIG = 1 << 31


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _rows(T):
    rng = np.random.default_rng(7)
    return np.unique(np.concatenate([[0, T // 2, T - 1], rng.integers(0, T, 13)]))


def test_out_prod_dx_past_2_31_elements(rg):
    """dX [131072, 16384] F32 (2^31 elements, 8 GiB) through the tensor-core
    path: sampled whole rows of dX, the last among them, against the oracle."""
    wtype, N, K, T = inputs.Q8_0, 256, 16384, 131072
    assert T * K >= BIG
    W = inputs.gen_weight(wtype, N, K, seed=120, stream=1)
    dY = inputs.normal_f32(120, 2, T * N, 1e-3).reshape(T, N)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    dX = torch.full((T, K), float("nan"), device=dev)
    rg.check(rg.rg_out_prod(wtype, torch.from_numpy(W).to(dev), N, K, torch.from_numpy(dY).to(dev), T, dX,
                            0.0, s), "rg_out_prod")
    rg.check(rg.rg_check(s))
    ts = _rows(T)
    got = dX[torch.from_numpy(ts).to(dev)].cpu().numpy().astype(np.float64)  # [len(ts), K]
    del dX
    torch.cuda.empty_cache()
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY[ts], len(ts), Wd=Wd)
    bnd = oracle.abs_bound(dY[ts], Wd)
    err = np.abs(got - ref)
    assert np.all(err <= 5e-3 * bnd + 1e-7), float((err / (bnd + 1e-30)).max())


def test_mul_mat_y_past_2_31_elements(rg):
    """Y [131072, 16384] F32 of the forward (tensor-core route): sampled
    whole rows of Y, the last among them, against the oracle."""
    wtype, N, K, T = inputs.Q4_K, 16384, 256, 131072
    assert T * N >= BIG
    W = inputs.gen_weight(wtype, N, K, seed=121, stream=1)
    X = inputs.normal_f32(121, 2, T * K, 1e-2).reshape(T, K)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Y = torch.full((T, N), float("nan"), device=dev)
    rg.check(rg.rg_mul_mat(wtype, torch.from_numpy(W).to(dev), N, K, torch.from_numpy(X).to(dev), T, Y, 0.0, s),
             "rg_mul_mat")
    rg.check(rg.rg_check(s))
    ts = _rows(T)
    got = Y[torch.from_numpy(ts).to(dev)].cpu().numpy().astype(np.float64)
    del Y
    torch.cuda.empty_cache()
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.mul_mat(wtype, W, N, K, X[ts], len(ts), Wd=Wd)
    bnd = oracle.mul_mat_bound(X[ts], Wd)
    err = np.abs(got - ref)
    assert np.all(err <= 5e-3 * bnd + 1e-7), float((err / (bnd + 1e-30)).max())


def test_dequant_output_past_2_31_elements(rg):
    """rg_dequant of a Q4_0 weight [131072, 16384] (2^31 values, 8 GiB of
    F32): the weight repeats one 64-row pattern, so every sampled row, the
    last among them, must equal the pattern's bit-exact decode."""
    wtype, K, P = inputs.Q4_0, 16384, 64
    N = 131072
    assert N * K >= BIG
    pat = inputs.gen_weight(wtype, P, K, seed=122, stream=1)
    rb = inputs.row_bytes(wtype, K)
    W = np.tile(pat.reshape(P, rb), (N // P, 1))
    dev = torch.device("cuda:0")
    out = torch.empty((N, K), device=dev)
    rg.check(rg.rg_dequant(wtype, torch.from_numpy(W).to(dev), N, K, out), "rg_dequant")
    ns = _rows(N)
    got = out[torch.from_numpy(ns).to(dev)].cpu().numpy()
    del out
    torch.cuda.empty_cache()
    want = oracle.dequant(wtype, pat, P, K)[ns % P]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
