"""rg_mul_mat, the forward Y = X . deq(W)^T, against the oracle."""
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


def _run(rg, wtype, W, N, K, X, T, Y0=None, beta=0.0):
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Y = torch.from_numpy(Y0).to(dev) if Y0 is not None else torch.full((T, N), float("nan"), device=dev)
    rg.check(rg.rg_mul_mat(wtype, torch.from_numpy(W).to(dev), N, K, torch.from_numpy(X).to(dev), T, Y,
                           beta, s), "rg_mul_mat")
    rg.check(rg.rg_check(s))
    return Y.cpu().numpy()


@pytest.mark.parametrize("wtype", inputs.ALL_TYPES)
@pytest.mark.parametrize("shape", [(208, 512, 300), (64, 256, 1), (1000, 768, 130), (72, 1024, 33),
                                   (136, 2048, 290)])
def test_mul_mat_parity(rg, wtype, shape):
    """Every weight type on ragged shapes (rows against the 128-row units,
    T against the 256-row tiles, K from one 256-value tile up); K that the
    type's rows do not align to runs the transient-copy route, the rest the
    fused decoder."""
    N, K, T = shape
    W = inputs.gen_weight(wtype, N, K, seed=91, stream=1)
    X = inputs.normal_f32(91, 2, T * K, 1e-2).reshape(T, K)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.mul_mat(wtype, W, N, K, X, T, Wd=Wd)
    bnd = oracle.mul_mat_bound(X, Wd)
    got = _run(rg, wtype, W, N, K, X, T)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= 5e-3 * bnd + 1e-7), float((err / (bnd + 1e-30)).max())


def _run_variant(rg, variant, wtype, W, N, K, X, T, Y0=None, beta=0.0):
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Y = torch.from_numpy(Y0).to(dev) if Y0 is not None else torch.full((T, N), float("nan"), device=dev)
    rg.check(rg.rg_mul_mat_variant(variant, wtype, torch.from_numpy(W).to(dev), N, K, torch.from_numpy(X).to(dev),
                                   T, Y, beta, s), "rg_mul_mat_variant")
    rg.check(rg.rg_check(s))
    return Y.cpu().numpy()


def _k_aligned(wtype, K):
    a = {inputs.Q6_K: 2048, inputs.Q3_K: 2048, inputs.Q2_K: 1024, inputs.MXFP4: 512}.get(wtype, 1)
    return -(-K // a) * a


@pytest.mark.parametrize("wtype", inputs.ALL_TYPES)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 6])
def test_mul_mat_small_t_parity(rg, wtype, T):
    """The small-T forward (W streamed once per four rows of X, exact F32
    decode and F32 products), named at one to six rows of X: every weight
    type, N ragged against the 8-, 16- and 32-row blocks (8, 200 and 1000
    rows), beta 0 (a NaN-filled Y must not show through) and beta -0.5; the
    error stays near F32 rounding, far inside the forward's bound.  One
    launch and no workspace."""
    half = wtype in (inputs.F16, inputs.BF16, inputs.F32)
    for i, N in enumerate((8, 200, 1000)):
        K = _k_aligned(wtype, 264 if half else 512)  # a half type's last tile ragged
        W = inputs.gen_weight(wtype, N, K, seed=96 + i, stream=1)
        X = inputs.normal_f32(96 + i, 2, T * K, 1e-2).reshape(T, K)
        Wd = oracle.dequant(wtype, W, N, K)
        Y0, beta = (inputs.normal_f32(96 + i, 3, T * N, 1e-3).reshape(T, N), -0.5) if i == 1 else (None, 0.0)
        torch.cuda.synchronize()
        before = rg.rg_launch_count()
        got = _run_variant(rg, rg.RG_VARIANT_SMALLT, wtype, W, N, K, X, T, Y0, beta)
        assert rg.rg_launch_count() - before == 1  # one kernel, nothing converted
        ref = oracle.mul_mat(wtype, W, N, K, X, T, Y0, beta, Wd=Wd)
        bnd = oracle.mul_mat_bound(X, Wd)
        extra = np.abs(beta * Y0.astype(np.float64)) * 2.0 ** -23 if beta else 0.0
        err = np.abs(got.astype(np.float64) - ref)
        assert np.all(err <= 1e-4 * bnd + 1e-9 + extra), (N, float((err / (bnd + 1e-30)).max()))


def test_mul_mat_routes(rg):
    """rg_mul_mat takes the small-T route for one or two rows of X (one
    launch, no workspace) and the tensor-core kernel from three; either
    route can be named at any T (the small-T one in chunks of four rows),
    and both agree with the oracle; rows TMA cannot address take the
    tensor-core route at any T."""
    N, K, wtype = 1000, 1024, inputs.Q4_K
    W = inputs.gen_weight(wtype, N, K, seed=97, stream=1)
    Wd = oracle.dequant(wtype, W, N, K)
    for T, variant, tol in [(2, rg.RG_VARIANT_TC, 5e-3), (9, rg.RG_VARIANT_SMALLT, 1e-4),
                            (3, rg.RG_VARIANT_AUTO, 5e-3), (1, rg.RG_VARIANT_AUTO, 1e-4),
                            (2, rg.RG_VARIANT_AUTO, 1e-4)]:
        X = inputs.normal_f32(97, 2 + T, T * K, 1e-2).reshape(T, K)
        torch.cuda.synchronize()
        before = rg.rg_launch_count()
        got = _run_variant(rg, variant, wtype, W, N, K, X, T)
        if variant == rg.RG_VARIANT_AUTO:
            assert (rg.rg_launch_count() - before == 1) == (T <= 2), T
        ref = oracle.mul_mat(wtype, W, N, K, X, T, Wd=Wd)
        assert np.all(np.abs(got - ref) <= tol * oracle.mul_mat_bound(X, Wd) + 1e-7), (T, variant)
    assert rg.rg_mul_mat_workspace_bytes(wtype, N, K, 2) == 0
    assert rg.rg_mul_mat_workspace_bytes(wtype, N, K, 3) > 0
    # Q6_K rows at K = 512 are not 16-byte aligned: no small-T route
    wtype, K = inputs.Q6_K, 512
    W = inputs.gen_weight(wtype, N, K, seed=98, stream=1)
    X = inputs.normal_f32(98, 2, K, 1e-2).reshape(1, K)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Y = torch.zeros((1, N), device=dev)
    assert rg.rg_mul_mat_variant(rg.RG_VARIANT_SMALLT, wtype, torch.from_numpy(W).to(dev), N, K,
                                 torch.from_numpy(X).to(dev), 1, Y, 0.0, s) == rg.RG_ERR_SHAPE
    Wd = oracle.dequant(wtype, W, N, K)
    got = _run(rg, wtype, W, N, K, X, 1)
    assert np.all(np.abs(got - oracle.mul_mat(wtype, W, N, K, X, 1, Wd=Wd))
                  <= 5e-3 * oracle.mul_mat_bound(X, Wd) + 1e-7)


FULL_SMALLT = [("q4_k", 14336, 4096, 1), ("q8_0", 4096, 14336, 1), ("q4_k", 4096, 14336, 4), ("f16", 4096, 4096, 2),
               ("q6_k", 4096, 4096, 3)]


@pytest.mark.parametrize("name,N,K,T", FULL_SMALLT)
def test_mul_mat_small_t_full_size_sampled(rg, name, N, K, T):
    """The small-T forward at layer sizes: Y finite everywhere, and the
    outputs of 514 sampled rows of W (the first and last among them), every
    row of X, against the oracle one output at a time."""
    wtype = {v: k for k, v in inputs.TYPE_NAMES.items()}[name]
    W = inputs.gen_weight(wtype, N, K, seed=99, stream=1)
    X = inputs.normal_f32(99, 2, T * K, 1e-2).reshape(T, K)
    got = _run_variant(rg, rg.RG_VARIANT_SMALLT, wtype, W, N, K, X, T)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(100)
    ns = np.concatenate([rng.integers(0, N, 512), [0, N - 1]])
    Wd = oracle.dequant(wtype, W, N, K)
    ts = np.repeat(np.arange(T), len(ns))
    nn = np.tile(ns, T)
    ref, bnd = oracle.mul_mat_at(Wd, X, ts, nn)
    err = np.abs(got[ts, nn].astype(np.float64) - ref)
    assert np.all(err <= 1e-4 * bnd + 1e-9), float((err / (bnd + 1e-30)).max())


def test_mul_mat_beta_and_one_hot(rg):
    # one-hot X selects columns of deq(W): Q8_0's decoded operand is the exact
    # product d * q rounded once to fp16, i.e. fp16(deq W)
    N, K, T, wtype = 256, 512, 40, inputs.Q8_0
    W = inputs.gen_weight(wtype, N, K, seed=92, stream=1)
    Wd = oracle.dequant(wtype, W, N, K)
    k0 = (41 * np.arange(T) + 5) % K
    X = np.zeros((T, K), np.float32)
    X[np.arange(T), k0] = 1.0
    got = _run(rg, wtype, W, N, K, X, T)
    want = Wd[:, k0].T.astype(np.float16).astype(np.float32)
    assert np.array_equal(got, want)
    # beta accumulates (Q4_K)
    wtype = inputs.Q4_K
    W = inputs.gen_weight(wtype, N, K, seed=92, stream=1)
    Wd = oracle.dequant(wtype, W, N, K)
    X = inputs.normal_f32(92, 2, T * K, 1e-2).reshape(T, K)
    Y0 = inputs.normal_f32(92, 3, T * N, 1e-3).reshape(T, N)
    got = _run(rg, wtype, W, N, K, X, T, Y0, 1.0)
    ref = oracle.mul_mat(wtype, W, N, K, X, T, Y0, 1.0, Wd=Wd)
    bnd = oracle.mul_mat_bound(X, Wd) + np.abs(Y0) * 2.0 ** -24 / 5e-3
    assert np.all(np.abs(got - ref) <= 5e-3 * bnd + 1e-7)


def test_mul_mat_large_splits_and_waves(rg):
    """A long contraction (K = 14336) with few outputs splits over CTAs; a
    wide one runs many pair tiles."""
    for (N, K, T) in [(256, 14336, 64), (4096, 512, 1100)]:
        wtype = inputs.Q8_0
        W = inputs.gen_weight(wtype, N, K, seed=93, stream=1)
        X = inputs.normal_f32(93, 2, T * K, 1e-2).reshape(T, K)
        Wd = oracle.dequant(wtype, W, N, K)
        got = _run(rg, wtype, W, N, K, X, T)
        ref = oracle.mul_mat(wtype, W, N, K, X, T, Wd=Wd)
        assert np.all(np.abs(got - ref) <= 5e-3 * oracle.mul_mat_bound(X, Wd) + 1e-7)


@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0, inputs.F16, inputs.Q6_K, inputs.NVFP4])
def test_mul_mat_holds_no_copy_of_the_weight(rg, wtype):
    """The fused forward's workspace is X's 16-bit copy (and a split's partial
    sums): far below the 2 N K bytes a dense 16-bit deq(W) would take, on the
    layer-sized shape it is timed on."""
    N, K, T = 14336, 4096, 8192
    ws = rg.rg_mul_mat_workspace_bytes(wtype, N, K, T)
    x16 = T * K * 2
    assert x16 <= ws < x16 + 2 * N * K // 4, (ws, x16)
    # rows TMA cannot address (Q6_K at K % 2048 != 0) take the transient copy
    if wtype == inputs.Q6_K:
        assert rg.rg_mul_mat_workspace_bytes(wtype, 4096, 2304, 512) >= 2 * 4096 * 2304


def test_mul_mat_shape_rules(rg):
    dev = torch.device("cuda:0")
    W = torch.zeros(100 * inputs.row_bytes(inputs.Q8_0, 256), dtype=torch.uint8, device=dev)
    X = torch.zeros((4, 256), device=dev)
    Y = torch.zeros((4, 100), device=dev)
    assert rg.rg_mul_mat(inputs.Q8_0, W, 100, 256, X, 4, Y, 0.0) == rg.RG_ERR_SHAPE   # N % 8
    assert rg.rg_mul_mat(inputs.Q8_0, W, 96, 200, X, 4, Y, 0.0) == rg.RG_ERR_SHAPE    # K % 256


FULL_FWD = [(w, i) for w in ("layer7b_t8192", "types_4096x4096_t8192") for i in range(len(inputs.WORKLOADS[w]))]


@pytest.mark.parametrize("workload,idx", FULL_FWD)
def test_mul_mat_full_size_sampled(rg, workload, idx):
    """The forward at full size, as bench.py --op mul_mat times it (same X
    generator, rg_mul_mat's own plan): the layer sweep's shapes and every
    weight type at 4096 x 4096, T = 8192; 4096 random (t, n) outputs plus the
    whole first and last rows against the oracle, one by one."""
    p = inputs.WORKLOADS[workload][idx]
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    W = p.weight()
    X = inputs.normal_f32(p.seed, 2 + p.stream_base, p.T * p.K, 1e-2).reshape(p.T, p.K)
    Y = torch.full((p.T, p.N), float("nan"), device=dev)
    rg.check(rg.rg_mul_mat(p.wtype, torch.from_numpy(W).to(dev), p.N, p.K, torch.from_numpy(X).to(dev),
                           p.T, Y, 0.0, s), "rg_mul_mat")
    rg.check(rg.rg_check(s))
    got = Y.cpu().numpy()
    assert np.isfinite(got).all()
    Wd = oracle.dequant(p.wtype, W, p.N, p.K)
    rng = np.random.default_rng(idx + 31)
    ts = np.concatenate([rng.integers(0, p.T, 4096), np.zeros(p.N, np.int64), np.full(p.N, p.T - 1, np.int64)])
    ns = np.concatenate([rng.integers(0, p.N, 4096), np.arange(p.N), np.arange(p.N)])
    ref, bnd = oracle.mul_mat_at(Wd, X, ts, ns)
    err = np.abs(got[ts, ns].astype(np.float64) - ref)
    lim = 5e-3 * bnd + 1e-7
    assert np.all(err <= lim), (p.name, int((err > lim).sum()), float((err / (bnd + 1e-30)).max()))


@pytest.mark.parametrize("wtype", [inputs.Q4_0, inputs.Q8_0, inputs.F16])
def test_mul_mat_split_in_two(rg, wtype):
    """A forward whose plan splits the contraction in two (4096 x 4096 at
    T = 512): with beta 0 both halves are added into the Y that X's
    conversion zeroed (a NaN-filled Y must not show through), with beta 1
    into partial sums and a reduction; sampled outputs against the oracle."""
    N, K, T = 4096, 4096, 512
    W = inputs.gen_weight(wtype, N, K, seed=94, stream=1)
    X = inputs.normal_f32(94, 2, T * K, 1e-2).reshape(T, K)
    Wd = oracle.dequant(wtype, W, N, K)
    rng = np.random.default_rng(95)
    ts = np.concatenate([rng.integers(0, T, 4096), np.full(N, T - 1, np.int64)])
    ns = np.concatenate([rng.integers(0, N, 4096), np.arange(N)])
    got = _run(rg, wtype, W, N, K, X, T)
    assert np.isfinite(got).all()
    ref, bnd = oracle.mul_mat_at(Wd, X, ts, ns)
    assert np.all(np.abs(got[ts, ns].astype(np.float64) - ref) <= 5e-3 * bnd + 1e-7)
    Y0 = inputs.normal_f32(94, 3, T * N, 1e-3).reshape(T, N)
    got = _run(rg, wtype, W, N, K, X, T, Y0, 1.0)
    ref, bnd = oracle.mul_mat_at(Wd, X, ts, ns, Y0, 1.0)
    lim = 5e-3 * bnd + 1e-7 + np.abs(Y0[ts, ns]) * 2.0 ** -24
    assert np.all(np.abs(got[ts, ns].astype(np.float64) - ref) <= lim)
