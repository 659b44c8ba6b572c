"""Seeded random cases through the C ABI against the oracle: weight type,
N, K, T, beta, variant and entry point (rg_out_prod_variant or rg_mul_mat)
drawn per case, so that combinations the hand-picked tests do not name are
still checked.  A case the library rejects for its documented shape rules
(rg_plan's status) is skipped; every other case must come back inside the
bound: |out - ref| <= tol * B + 1e-7 + 2^-23 |beta * out0|, tol 5e-3 (1e-5
for the SIMT variant), B the sum of absolute products."""
import ctypes

import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
needs_gpu = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

N_CASES = 160
ALIGN = {inputs.Q6_K: 2048, inputs.Q3_K: 2048, inputs.Q2_K: 1024, inputs.MXFP4: 512}
HALF = (inputs.F16, inputs.BF16, inputs.F32)


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def draw_case(i: int) -> dict:
    """Case i's parameters (its own generator: one case does not shift another)."""
    rng = np.random.default_rng([7919, i])
    wt = int(rng.choice(inputs.ALL_TYPES))
    fwd = bool(rng.random() < 0.2)
    variant = int(rng.choice([0, 0, 0, 1, 2, 3, 4, 5]))
    r = rng.random()
    T = int(rng.integers(1, 9)) if r < 0.3 else int(rng.integers(9, 65)) if r < 0.55 else int(rng.integers(65, 700))
    N = int(rng.integers(1, 2600))
    kmul = 8 if wt in HALF else 256
    K = int(rng.integers(1, 7)) * 256 if rng.random() < 0.7 else int(rng.integers(1, 20)) * kmul
    if wt in ALIGN and variant != 3 and rng.random() < 0.7:
        K = -(-K // ALIGN[wt]) * ALIGN[wt]
    beta = float(rng.choice([0.0, 0.0, 1.0, 0.5, -2.0]))
    if fwd:
        N = max(8, N // 8 * 8)
    if T * N * K > 3e8:
        T = max(1, int(3e8 // (N * K)))
    return dict(wt=wt, fwd=fwd, variant=variant, N=N, K=K, T=T, beta=beta, seed=2000 + i)


def test_cases_cover_every_type_variant_and_both_ops():
    """(host only) the draws reach every weight type, every variant, the
    forward, one to four rows and every beta."""
    cases = [draw_case(i) for i in range(N_CASES)]
    assert {c["wt"] for c in cases} == set(inputs.ALL_TYPES)
    assert {c["variant"] for c in cases if not c["fwd"]} == {0, 1, 2, 3, 4, 5}
    assert any(c["fwd"] for c in cases) and any(c["T"] <= 4 for c in cases)
    assert {c["beta"] for c in cases} == {0.0, 1.0, 0.5, -2.0}


@needs_gpu[0]
@needs_gpu[1]
@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(rg, i):
    c = draw_case(i)
    wt, N, K, T, beta, seed = c["wt"], c["N"], c["K"], c["T"], c["beta"], c["seed"]
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    W = inputs.gen_weight(wt, N, K, seed=seed, stream=1)
    Wd = oracle.dequant(wt, W, N, K)
    Wt = torch.from_numpy(np.ascontiguousarray(W)).to(dev)
    if c["fwd"]:
        X = inputs.normal_f32(seed, 2, T * K, 1e-2).reshape(T, K)
        Y0 = inputs.normal_f32(seed, 3, T * N, 1e-3).reshape(T, N)
        Y = torch.from_numpy(Y0).to(dev) if beta else torch.full((T, N), float("nan"), device=dev)
        st = rg.rg_mul_mat(wt, Wt, N, K, torch.from_numpy(X).to(dev), T, Y, beta, s)
        if st == rg.RG_ERR_SHAPE:
            pytest.skip(f"rejected by the shape rules: {c}")
        rg.check(st, f"rg_mul_mat {c}")
        rg.check(rg.rg_check(s), f"rg_check {c}")
        got = Y.cpu().numpy().astype(np.float64)
        ref = oracle.mul_mat(wt, W, N, K, X, T, Y0, beta, Wd=Wd)
        bnd, tol, old = oracle.mul_mat_bound(X, Wd), 5e-3, Y0
    else:
        info = rg.rg_plan_info()
        st = rg.load().rg_plan(c["variant"], wt, N, K, T, ctypes.byref(info))
        if st == rg.RG_ERR_SHAPE:
            pytest.skip(f"rejected by the shape rules: {c}")
        rg.check(st, f"rg_plan {c}")
        dY = inputs.normal_f32(seed, 2, T * N, 1e-3).reshape(T, N)
        dX0 = inputs.normal_f32(seed, 3, T * K, 1e-3).reshape(T, K)
        dX = torch.from_numpy(dX0).to(dev) if beta else torch.full((T, K), float("nan"), device=dev)
        rg.check(rg.rg_out_prod_variant(c["variant"], wt, Wt, N, K, torch.from_numpy(dY).to(dev), T, dX,
                                        beta, s), f"rg_out_prod_variant {c}")
        rg.check(rg.rg_check(s), f"rg_check {c}")
        got = dX.cpu().numpy().astype(np.float64)
        ref = oracle.out_prod(wt, W, N, K, dY, T, dX0, beta, Wd=Wd)
        bnd, tol, old = oracle.abs_bound(dY, Wd), (1e-5 if info.variant == rg.RG_VARIANT_SIMT32 else 5e-3), dX0
    lim = tol * bnd + 1e-7 + (np.abs(beta * old.astype(np.float64)) * 2.0 ** -23 if beta else 0.0)
    err = np.abs(got - ref)
    bad = ~(err <= lim)
    assert not bad.any(), (c, int(bad.sum()), float(np.nanmax(err / (bnd + 1e-30))))
