"""rg_out_prod_lora, the input gradient through the resident weight plus a
low-rank adapter, against the oracle.

Bounds (the adapter term's derived from its roundings):
  * tensor-core variants: |dX - ref| <= 5e-3 * B_base + 1e-2 * B_lora + 1e-7,
    where dY, B, U = dY . B and scale * A are each rounded to 16 bits once;
  * small-T and SIMT variants (adapter term in F32): the base bound of the
    variant plus 1e-5 * B_lora;
with B_base = sum_n |dY||deq W| and B_lora = |scale| sum_j (sum_n |dY||B|)|A|.
"""
import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

BASE_TOL = {1: 5e-3, 2: 5e-3, 3: 1e-5, 4: 5e-3, 5: 5e-3}
LORA_TOL = {1: 1e-2, 2: 1e-5, 3: 1e-5, 4: 1e-2, 5: 1e-2}


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _inputs(wtype, N, K, T, R, seed):
    W = inputs.gen_weight(wtype, N, K, seed=seed, stream=1)
    dY = inputs.normal_f32(seed, 2, T * N, 1.0).reshape(T, N)
    A = inputs.normal_f32(seed, 3, R * K, 0.05).reshape(R, K)
    B = inputs.normal_f32(seed, 4, N * R, 0.05).reshape(N, R)
    return W, dY, A, B


def _run(rg, variant, wtype, W, N, K, dY, T, A, B, R, scale, dX0=None, beta=0.0, fill=float("nan")):
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    dX = t(dX0) if dX0 is not None else torch.full((T, K), fill, device=dev)
    Ad = t(A) if R > 0 else torch.zeros(4, device=dev)
    Bd = t(B) if R > 0 else torch.zeros(4, device=dev)
    rg.check(rg.rg_out_prod_lora(variant, wtype, t(W), N, K, t(dY), T, dX, beta, Ad, Bd, R, scale, s),
             "rg_out_prod_lora")
    rg.check(rg.rg_check(s))
    return dX.cpu().numpy()


def _check(got, ref, bnd_base, bnd_lora, variant, what=""):
    err = np.abs(got.astype(np.float64) - ref)
    lim = BASE_TOL[variant] * bnd_base + LORA_TOL[variant] * bnd_lora + 1e-7
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside the bound; first "
                             f"{idx.tolist()}, err {err[bad][:5]}, lim {lim[bad][:5]}")


def _kfit(wtype, K, variant):
    a = {inputs.Q6_K: 2048, inputs.Q3_K: 2048, inputs.Q2_K: 1024, inputs.MXFP4: 512}.get(wtype)
    if a and variant != 3:
        return (K + a - 1) // a * a
    return K


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0, inputs.Q5_0, inputs.Q6_K, inputs.F16,
                                   inputs.BF16, inputs.F32, inputs.Q2_K, inputs.Q3_K, inputs.MXFP4])
@pytest.mark.parametrize("shape", [(200, 512, 300, 16), (64, 256, 1, 7), (1000, 768, 130, 100),
                                   (72, 1024, 33, 1), (201, 512, 77, 32), (130, 256, 40, 33),
                                   (96, 512, 50, 9)])
def test_lora_parity(rg, variant, wtype, shape):
    N, K, T, R = shape
    K = _kfit(wtype, K, variant)
    W, dY, A, B = _inputs(wtype, N, K, T, R, seed=101)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod_lora(wtype, W, N, K, dY, T, A, B, R, 2.0, Wd=Wd)
    got = _run(rg, variant, wtype, W, N, K, dY, T, A, B, R, 2.0)
    _check(got, ref, oracle.abs_bound(dY, Wd), oracle.lora_bound(dY, A, B, 2.0), variant,
           f"variant {variant} type {wtype} {shape}")


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_lora_rank_zero_is_out_prod(rg, variant):
    N, K, T = 192, 512, 70
    W, dY, _, _ = _inputs(inputs.Q4_K, N, K, T, 1, seed=102)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Wt, dYt = torch.from_numpy(W).to(dev), torch.from_numpy(dY).to(dev)
    want = torch.full((T, K), float("nan"), device=dev)
    rg.check(rg.rg_out_prod_variant(variant, inputs.Q4_K, Wt, N, K, dYt, T, want, 0.0, s))
    got = _run(rg, variant, inputs.Q4_K, W, N, K, dY, T, None, None, 0, 3.0)
    assert np.array_equal(got, want.cpu().numpy())


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_lora_beta_and_negative_scale(rg, variant):
    N, K, T, R = 130, 512, 45, 24
    W, dY, A, B = _inputs(inputs.Q8_0, N, K, T, R, seed=103)
    dX0 = inputs.normal_f32(103, 5, T * K, 1.0).reshape(T, K)
    Wd = oracle.dequant(inputs.Q8_0, W, N, K)
    ref = oracle.out_prod_lora(inputs.Q8_0, W, N, K, dY, T, A, B, R, -0.5, dX0, 0.75, Wd=Wd)
    got = _run(rg, variant, inputs.Q8_0, W, N, K, dY, T, A, B, R, -0.5, dX0, 0.75)
    base = oracle.abs_bound(dY, Wd) + np.abs(0.75 * dX0) * 2.0 ** -24 / BASE_TOL[variant]
    _check(got, ref, base, oracle.lora_bound(dY, A, B, -0.5), variant)


def test_lora_zero_adapter_adds_nothing(rg):
    """A = 0: the adapter's chunk contributes exact zeros, so the tensor-core
    result equals the base product's bit for bit."""
    N, K, T, R = 256, 2048, 2048, 32
    info = rg.rg_plan_info()
    for n in (N, N + 64):  # the same (unsplit) order of chunks with and without the adapter
        rg.check(rg.rg_plan(1, inputs.Q4_0, n, K, T, info))
        assert info.n_splits == 1
    W, dY, _, B = _inputs(inputs.Q4_0, N, K, T, R, seed=104)
    A = np.zeros((R, K), np.float32)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    want = torch.empty((T, K), device=dev)
    rg.check(rg.rg_out_prod_variant(1, inputs.Q4_0, torch.from_numpy(W).to(dev), N, K,
                                    torch.from_numpy(dY).to(dev), T, want, 0.0, s))
    got = _run(rg, 1, inputs.Q4_0, W, N, K, dY, T, A, B, R, 1.0)
    assert np.array_equal(got, want.cpu().numpy())


def test_lora_split_contraction(rg):
    """Few outputs and a long contraction: the base product (and U) split the
    contraction over CTAs; the adapter's chunk lands in the last split."""
    N, K, T, R = 4096, 256, 64, 48
    W, dY, A, B = _inputs(inputs.Q4_K, N, K, T, R, seed=105)
    info = rg.rg_plan_info()
    rg.check(rg.rg_plan(1, inputs.Q4_K, N, K, T, info))
    assert info.n_splits > 1
    Wd = oracle.dequant(inputs.Q4_K, W, N, K)
    ref = oracle.out_prod_lora(inputs.Q4_K, W, N, K, dY, T, A, B, R, 1.0, Wd=Wd)
    got = _run(rg, 1, inputs.Q4_K, W, N, K, dY, T, A, B, R, 1.0)
    _check(got, ref, oracle.abs_bound(dY, Wd), oracle.lora_bound(dY, A, B, 1.0), 1)


@pytest.mark.parametrize("R", [16, 32, 64])
def test_lora_layer_size_sampled(rg, R):
    """The gate projection of a 7B layer (N = 14336 rows of K = 4096 Q4_K
    values) at T = 8192 with a rank-R adapter, in the launch configuration
    the bench times; 4096 sampled outputs against the oracle one by one."""
    N, K, T = 14336, 4096, 8192
    W, dY, A, B = _inputs(inputs.Q4_K, N, K, T, R, seed=106)
    got = _run(rg, 0, inputs.Q4_K, W, N, K, dY, T, A, B, R, 0.5)
    rng = np.random.default_rng(106)
    ts, ks = rng.integers(0, T, 4096), rng.integers(0, K, 4096)
    ts[:2], ks[:2] = [T - 1, 0], [K - 1, 0]
    Wd = oracle.dequant(inputs.Q4_K, W, N, K)
    ref, bnd = oracle.out_prod_at(Wd, dY, ts, ks)
    lv, lb = oracle.lora_at(dY, A, B, 0.5, ts, ks)
    err = np.abs(got[ts, ks].astype(np.float64) - (ref + lv))
    assert np.all(err <= 5e-3 * bnd + 1e-2 * lb + 1e-7), float(err.max())


@pytest.mark.parametrize("variant", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0, inputs.F16, inputs.BF16, inputs.F32])
@pytest.mark.parametrize("shape", [(200, 512, 300, 16), (64, 256, 2, 70), (640, 256, 129, 3)])
def test_lora_adapter_term_alone(rg, variant, wtype, shape):
    """An all-zero W (every block's scales zero) removes the base term, so the
    adapter's term is checked against its own bound alone."""
    N, K, T, R = shape
    _, dY, A, B = _inputs(wtype, N, K, T, R, seed=107)
    W = np.zeros(N * inputs.row_bytes(wtype, K), np.uint8)
    ref = oracle.out_prod_lora(wtype, W, N, K, dY, T, A, B, R, 1.5)
    assert np.abs(ref).max() > 0.1   # the term is far above the 1e-7 floor
    got = _run(rg, variant, wtype, W, N, K, dY, T, A, B, R, 1.5)
    _check(got, ref, np.zeros_like(ref), oracle.lora_bound(dY, A, B, 1.5), variant,
           f"variant {variant} type {wtype} {shape}")
