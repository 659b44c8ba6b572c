"""GPU parity: every kernel through the C ABI against the CPU oracle.

Bars (from the acceptance of the method):
  * rg_dequant: bit-exact F32 words (signed zeros included);
  * tensor-core and small-T variants: |dX - ref| <= 5e-3 * B + 1e-7;
  * full-F32 SIMT variant:             |dX - ref| <= 1e-5 * B + 1e-7;
where ref is the oracle's F64 result and B[t, k] = sum_n |dY[t, n]| |deq(W)[n, k]|.
"""
import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TYPES = inputs.ALL_TYPES
TOL = {1: 5e-3, 2: 5e-3, 3: 1e-5, 4: 5e-3, 5: 5e-3}  # tc, smallt, simt32, tc1, tc2
ALL_VARIANTS = [1, 2, 3, 4, 5]


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _dev():
    return torch.device("cuda:0")


ROW_ALIGN_K = {inputs.Q6_K: 2048, inputs.Q3_K: 2048, inputs.Q2_K: 1024, inputs.MXFP4: 512}


def kfit(wtype, K, variant):
    """Q6_K and Q3_K rows are 16-byte aligned only for K % 2048 == 0, Q2_K
    rows for K % 1024 == 0 and MXFP4 rows for K % 512 == 0, which every
    variant but the SIMT one needs: round K up for those."""
    a = ROW_ALIGN_K.get(wtype)
    if a and variant != 3:
        return -(-K // a) * a
    return K


def run_out_prod(rg, variant, wtype, W, N, K, dY, T, dX0=None, beta=0.0, fill=float("nan")):
    dev = _dev()
    Wd = torch.from_numpy(np.ascontiguousarray(W)).to(dev)
    dYd = torch.from_numpy(np.ascontiguousarray(dY, dtype=np.float32)).to(dev)
    if dX0 is not None:
        dX = torch.from_numpy(np.ascontiguousarray(dX0, dtype=np.float32)).to(dev)
    else:
        dX = torch.full((T, K), fill, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream()
    st = rg.rg_out_prod_variant(variant, wtype, Wd, N, K, dYd, T, dX, beta, s)
    rg.check(st, "rg_out_prod_variant")
    rg.check(rg.rg_check(s), "rg_check")
    return dX.cpu().numpy()


def assert_within(got, ref, bnd, tol, what=""):
    err = np.abs(got.astype(np.float64) - ref)
    lim = tol * bnd + 1e-7
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside the bound; "
                             f"first {idx.tolist()}, err {err[bad][:5]}, lim {lim[bad][:5]}")


# ----------------------------------------------------------------------------
# rg_dequant: bit-exact

@pytest.mark.parametrize("wtype", TYPES)
@pytest.mark.parametrize("N,K", [(3, 256), (77, 768), (130, 2048)])
def test_dequant_bit_exact(rg, wtype, N, K):
    W = inputs.gen_weight(wtype, N, K, seed=1, stream=1)
    ref = oracle.dequant(wtype, W, N, K)
    out = torch.full((N, K), float("nan"), device=_dev())
    rg.check(rg.rg_dequant(wtype, torch.from_numpy(W).to(_dev()), N, K, out))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_negative_zero_and_extremes(rg):
    """Hand blocks with d < 0 and zero codes decode to -0.0; fp16 extremes."""
    q40 = bytes.fromhex("00c0f0e1d2c3b4a5968778695a4b3c2d1e0f") * 8     # 256 values
    q80 = bytes.fromhex("0038807ff2f3f4f5f6f7f8f9fafbfcfdfeff000102030405060708090a0b0c0d0e0f")
    q80 = (bytes([0x00, 0xBC]) + bytes([0]) * 32) * 4 + q80 * 4             # d = -1, q = 0
    f16 = np.array([0x0001, 0x8000, 0x7BFF, 0xFBFF, 0x0400, 0x3C00, 0x8001, 0x03FF], np.uint16)
    cases = [(inputs.Q4_0, np.frombuffer(q40, np.uint8)), (inputs.Q8_0, np.frombuffer(q80, np.uint8)),
             (inputs.F16, np.tile(f16, 32).view(np.uint8)), (inputs.BF16, np.tile(f16, 32).view(np.uint8))]
    for wtype, W in cases:
        ref = oracle.dequant(wtype, W, 1, 256)
        out = torch.zeros((1, 256), device=_dev())
        rg.check(rg.rg_dequant(wtype, torch.from_numpy(W.copy()).to(_dev()), 1, 256, out))
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32)), wtype


# ----------------------------------------------------------------------------
# OUT_PROD: every variant, several tiles and ragged tails

SHAPES = [  # (N, K, T): N ragged against the 64-row stage, T against 128/256-row tiles
    (200, 512, 300),
    (64, 256, 1),
    (1000, 768, 520),
    (77, 1024, 33),
]


@pytest.mark.parametrize("variant", ALL_VARIANTS)
@pytest.mark.parametrize("wtype", TYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_out_prod_parity(rg, variant, wtype, shape):
    N, K, T = shape
    K = kfit(wtype, K, variant)
    W = inputs.gen_weight(wtype, N, K, seed=3, stream=1)
    dY = inputs.normal_f32(3, 2, T * N, 1e-3).reshape(T, N)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd)
    got = run_out_prod(rg, variant, wtype, W, N, K, dY, T)
    assert_within(got, ref, bnd, TOL[variant], f"variant {variant} type {wtype} {shape}")


@pytest.mark.parametrize("variant", ALL_VARIANTS)
@pytest.mark.parametrize("beta", [1.0, 0.5, -2.0])
def test_beta_accumulates(rg, variant, beta):
    N, K, T = 192, 512, 130
    wtype = inputs.Q4_K
    W = inputs.gen_weight(wtype, N, K, seed=4, stream=1)
    dY = inputs.normal_f32(4, 2, T * N, 1e-3).reshape(T, N)
    dX0 = inputs.normal_f32(4, 3, T * K, 1e-3).reshape(T, K)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, dX0, beta, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd)
    got = run_out_prod(rg, variant, wtype, W, N, K, dY, T, dX0, beta)
    # beta*dX0 is one F32 rounding: allow 2^-24 |beta dX0| on top of the bound
    assert_within(got, ref, bnd + np.abs(beta * dX0) * (2.0 ** -24) / TOL[variant], TOL[variant])


@pytest.mark.parametrize("variant", ALL_VARIANTS)
def test_beta_zero_ignores_nan(rg, variant):
    N, K, T = 96, 256, 40
    W = inputs.gen_weight(inputs.Q8_0, N, K, seed=5, stream=1)
    dY = inputs.normal_f32(5, 2, T * N, 1.0).reshape(T, N)
    got = run_out_prod(rg, variant, inputs.Q8_0, W, N, K, dY, T, fill=float("nan"))
    assert np.isfinite(got).all()


def _q4_k_scale_part(W, N, K):
    """d * sc * q of every Q4_K value (the decode with dmin zeroed)."""
    Wz = W.copy().reshape(-1, 144)
    Wz[:, 2:4] = 0
    return oracle.dequant(inputs.Q4_K, Wz.reshape(-1), N, K)


@pytest.mark.parametrize("variant", [2, 3])
@pytest.mark.parametrize("wtype", TYPES)
def test_one_hot_f32_variants_equal_rows(rg, variant, wtype):
    """F32 variants: one-hot dY reproduces rows of deq(W) exactly.  Q4_K on
    the small-T variant multiplies in the MMA with fp16(y * d * sc): one
    rounding of the scale part, 2^-11 relative, and the F32 subtraction.
    Q8_0's MMA operands are exact there (fp16(2^s * d) = 2^s * d, q an fp16
    integer), so its rows come out exactly too."""
    N, K, T = 80, kfit(wtype, 512, variant), 6
    W = inputs.gen_weight(wtype, N, K, seed=6, stream=1)
    Wd = oracle.dequant(wtype, W, N, K)
    n0 = [(13 * t + 5) % N for t in range(T)]
    dY = np.zeros((T, N), np.float32)
    dY[np.arange(T), n0] = 1.0
    got = run_out_prod(rg, variant, wtype, W, N, K, dY, T)
    if variant == 2 and wtype == inputs.Q4_K:
        dsq = _q4_k_scale_part(W, N, K).astype(np.float64)
        for t in range(T):
            err = np.abs(got[t].astype(np.float64) - Wd[n0[t]])
            lim = 2.0 ** -11 * dsq[n0[t]] + 2.0 ** -23 * (np.abs(Wd[n0[t]]) + dsq[n0[t]])
            assert np.all(err <= lim), (t, float((err - lim).max()))
        return
    for t in range(T):
        assert np.array_equal(np.abs(got[t]), np.abs(Wd[n0[t]])), (t,)


@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 11])
def test_smallt_mma_rows(rg, T, wtype):
    """The small-T MMA consumer of Q4_K and Q8_0 (warp-level MMA, one to
    eight dY rows a pass): ragged N against the 64-row stages and the row
    splits, three k tiles, one dY row all zero (exact zeros out), one tiny
    (1e-30) and one large (1e3) row, each kept in fp16's normal range by the
    row's power-of-two scale."""
    N, K = 1000, 768
    W = inputs.gen_weight(wtype, N, K, seed=31, stream=1)
    dY = inputs.normal_f32(31, 2, T * N, 1e-3).reshape(T, N)
    if T >= 3:
        dY[1] = 0.0
        dY[2] *= np.float32(1e-27)
    if T >= 4:
        dY[3] *= np.float32(1e6)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd)
    got = run_out_prod(rg, 2, wtype, W, N, K, dY, T)
    assert_within(got, ref, bnd, 5e-3, f"T {T}")
    if T >= 3:
        assert np.all(got[1] == 0.0)
        # the tiny and large rows on their own scale (no absolute slack)
        for t in range(2, min(T, 4)):
            err = np.abs(got[t].astype(np.float64) - ref[t])
            assert np.all(err <= 5e-3 * bnd[t]), (t, float((err / bnd[t]).max()))


@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0])
@pytest.mark.parametrize("T", [1, 4])
def test_smallt_mma_rows_spanning_octaves(rg, T, wtype):
    """dY whose elements spread over nine decades inside every row slice
    (|y| = |N(0, 1)| * 10^u, u uniform in [-9, 0]): the entries of the
    small-T MMA consumer's fp16 table far below the slice's maximum are
    subnormal and keep fewer bits, yet the result stays within 5e-3 of the
    bound with no absolute slack, the bound's sum being carried by the
    slice's large rows."""
    N, K = 1000, 768
    W = inputs.gen_weight(wtype, N, K, seed=33, stream=1)
    g = inputs.normal_f32(33, 2, T * N, 1.0)
    u = inputs.uniform01(inputs.stream_key(33, 4), 0, T * N)
    dY = (g * 10.0 ** (-9.0 * u)).astype(np.float32).reshape(T, N)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd)
    assert rg.rg_select_variant(wtype, N, K, T) == rg.RG_VARIANT_SMALLT
    got = run_out_prod(rg, 2, wtype, W, N, K, dY, T)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= 5e-3 * bnd), float((err / bnd).max())


@pytest.mark.parametrize("variant", [4, 5])
@pytest.mark.parametrize("wtype", TYPES)
def test_all_ones_closed_form_tc(rg, variant, wtype):
    """All-ones weight times one-hot dY gives exactly 1 on the tensor cores too."""
    from test_oracle import _all_ones_weight
    N, K, T = 128, kfit(wtype, 512, variant), 260
    W = _all_ones_weight(wtype, N, K).copy()
    dY = np.zeros((T, N), np.float32)
    dY[np.arange(T), (7 * np.arange(T) + 3) % N] = 1.0
    got = run_out_prod(rg, variant, wtype, W, N, K, dY, T)
    assert np.all(got == 1.0)


@pytest.mark.parametrize("wtype", TYPES)
def test_pair_tiles_many_waves(rg, wtype):
    """Enough 256 x 256 tiles that the pair kernel's persistent CTAs loop over
    several tiles each (both accumulators, ragged N and T)."""
    N, K, T = 520, 4096, 1300
    W = inputs.gen_weight(wtype, N, K, seed=12, stream=1)
    dY = inputs.normal_f32(12, 2, T * N, 1e-3).reshape(T, N)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd)
    for variant in (1, 5):
        got = run_out_prod(rg, variant, wtype, W, N, K, dY, T)
        assert_within(got, ref, bnd, 5e-3, f"variant {variant} type {wtype}")


@pytest.mark.parametrize("variant", [0] + ALL_VARIANTS)
def test_empty_contraction_scales(rg, variant):
    T, K = 5, 256
    dX0 = inputs.normal_f32(7, 3, T * K, 1.0).reshape(T, K)
    got = run_out_prod(rg, variant, inputs.Q4_0, np.zeros(0, np.uint8), 0, K,
                       np.zeros((T, 0), np.float32), T, dX0, 0.5)
    assert np.array_equal(got, (np.float32(0.5) * dX0).astype(np.float32))
    got0 = run_out_prod(rg, variant, inputs.Q4_0, np.zeros(0, np.uint8), 0, K,
                        np.zeros((T, 0), np.float32), T, fill=float("nan"))
    assert np.all(got0 == 0.0)


def test_workspace_entry_point_matches(rg):
    N, K, T = 300, 512, 270
    wtype = inputs.Q4_0
    W = inputs.gen_weight(wtype, N, K, seed=8, stream=1)
    dY = inputs.normal_f32(8, 2, T * N, 1e-3).reshape(T, N)
    a = run_out_prod(rg, 1, wtype, W, N, K, dY, T)
    need = rg.rg_workspace_bytes(1, wtype, N, K, T)
    ws = torch.empty(need, dtype=torch.uint8, device=_dev())
    dev = _dev()
    dX = torch.empty((T, K), device=dev)
    s = torch.cuda.current_stream()
    args = (1, wtype, torch.from_numpy(W).to(dev), N, K, torch.from_numpy(dY).to(dev), T, dX, 0.0)
    assert rg.rg_out_prod_ws(*args, ws, need - 1, s) == rg.RG_ERR_ARG
    rg.check(rg.rg_out_prod_ws(*args, ws, need, s))
    rg.check(rg.rg_check(s))
    assert np.array_equal(dX.cpu().numpy(), a)   # same kernels, same order: identical


def test_timeout_probe_reports_and_context_survives(rg):
    s = torch.cuda.current_stream()
    rg.check(rg.rg_check(s))
    rg.check(rg.rg_debug_wait_probe(200, s))
    assert rg.rg_check(s) == rg.RG_ERR_TIMEOUT
    assert rg.rg_check(s) == rg.RG_OK     # read-and-clear
    N, K, T = 64, 256, 40                 # the context still computes
    W = inputs.gen_weight(inputs.Q8_0, N, K, seed=9, stream=1)
    dY = inputs.normal_f32(9, 2, T * N, 1.0).reshape(T, N)
    got = run_out_prod(rg, 1, inputs.Q8_0, W, N, K, dY, T)
    Wd = oracle.dequant(inputs.Q8_0, W, N, K)
    assert_within(got, oracle.out_prod(inputs.Q8_0, W, N, K, dY, T, Wd=Wd),
                  oracle.abs_bound(dY, Wd), 5e-3)


_STALL_CHILD = r"""
import sys
import numpy as np
import torch
sys.path[:0] = sys.argv[1:3]
import oracle
from quantized_weight_out_gb300 import binding as rg, inputs
rg.load()
dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
def call(variant, wtype, N, K, T):
    W = inputs.gen_weight(wtype, N, K, seed=8, stream=1)
    dY = inputs.normal_f32(8, 2, T * N, 1e-3).reshape(T, N)
    dX = torch.empty((T, K), device=dev)
    rg.check(rg.rg_out_prod_variant(variant, wtype, torch.from_numpy(W).to(dev), N, K,
                                    torch.from_numpy(dY).to(dev), T, dX, 0.0, s))
    return W, dY, dX
# the three small-T consumers: Q4_K (MMA, row splits), Q8_0 (a row per lane,
# one slice), F16 (eight values a lane)
for wtype, N, K, T in ((inputs.Q4_K, 1000, 512, 1), (inputs.Q8_0, 200, 256, 2),
                       (inputs.F16, 300, 256, 5)):
    call(2, wtype, N, K, T)
    st = rg.rg_check(s)
    assert st == rg.RG_ERR_TIMEOUT, (wtype, st)
W, dY, dX = call(3, inputs.Q8_0, 64, 256, 6)  # the SIMT variant waits on nothing
assert rg.rg_check(s) == rg.RG_OK
Wd = oracle.dequant(inputs.Q8_0, W, 64, 256)
err = np.abs(dX.cpu().numpy() - oracle.out_prod(inputs.Q8_0, W, 64, 256, dY, 6, Wd=Wd))
assert np.all(err <= 1e-5 * oracle.abs_bound(dY, Wd) + 1e-7)
print("stall ok")
"""


def test_small_t_stalled_stage_times_out_and_context_survives(rg):
    """A child process whose small-T producers skip their first stage
    (RG_DEBUG_INJECT_STALL, with a 300 ms wait limit): every consumer's wait
    runs out, all warps leave together, rg_check reports RG_ERR_TIMEOUT for
    each consumer kind, and the context still computes exactly afterwards.
    No fault: the stage is a flag that nothing sets."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RG_DEBUG_INJECT_STALL="1", RG_WAIT_TIMEOUT_MS="300")
    r = subprocess.run([sys.executable, "-c", _STALL_CHILD, root, os.path.join(root, "tests")],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "stall ok" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])


@pytest.mark.parametrize("variant", [1, 4, 5])
@pytest.mark.parametrize("wtype", TYPES)
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_split_contraction(rg, variant, wtype, beta):
    """Few output tiles and a long contraction: the tensor-core kernel splits
    the rows of W over CTAs and a second kernel adds the partial tiles."""
    N, K, T = 2050, kfit(wtype, 512, variant), 100  # ragged N: the last split runs past W's end
    W = inputs.gen_weight(wtype, N, K, seed=31, stream=1)
    dY = inputs.normal_f32(31, 2, T * N, 1e-3).reshape(T, N)
    dX0 = inputs.normal_f32(31, 3, T * K, 1e-3).reshape(T, K) if beta else None
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, dX0, beta, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd)
    got = run_out_prod(rg, variant, wtype, W, N, K, dY, T, dX0, beta)
    extra = np.abs(beta * dX0) * 2.0 ** -24 / 5e-3 if beta else 0.0
    assert_within(got, ref, bnd + extra, 5e-3, f"split variant {variant} type {wtype}")


@pytest.mark.parametrize("wtype", [inputs.Q6_K, inputs.Q3_K, inputs.Q2_K, inputs.MXFP4])
def test_unaligned_super_block_rows(rg, wtype):
    """K % 2048 (Q2_K: 1024, MXFP4: 512) != 0: the tensor-core and small-T variants
    refuse the shape (nothing launched), and the dispatcher runs the SIMT
    variant instead."""
    N, K, T = 70, 768, 40                 # Q6_K rows of 630 bytes: only 2-byte aligned
    W = inputs.gen_weight(wtype, N, K, seed=41, stream=1)
    dY = inputs.normal_f32(41, 2, T * N, 1e-3).reshape(T, N)
    dev, s = _dev(), torch.cuda.current_stream()
    Wt, dYt = torch.from_numpy(W).to(dev), torch.from_numpy(dY).to(dev)
    dX = torch.full((T, K), 3.0, device=dev)
    for v in (1, 2, 4, 5):
        assert rg.rg_out_prod_variant(v, wtype, Wt, N, K, dYt, T, dX, 0.0, s) == rg.RG_ERR_SHAPE
    torch.cuda.synchronize()
    assert bool(torch.all(dX == 3.0))
    assert rg.rg_select_variant(wtype, N, K, T) == rg.RG_VARIANT_SIMT32
    got = run_out_prod(rg, 0, wtype, W, N, K, dY, T)
    Wd = oracle.dequant(wtype, W, N, K)
    assert_within(got, oracle.out_prod(wtype, W, N, K, dY, T, Wd=Wd),
                  oracle.abs_bound(dY, Wd), 1e-5, "simt")


# ----------------------------------------------------------------------------
# rg_plan agrees with what a call launches

@pytest.mark.parametrize("variant", [0] + ALL_VARIANTS)
@pytest.mark.parametrize("wtype,N,K,T", [(inputs.Q4_K, 2050, 512, 100), (inputs.Q8_0, 1024, 4096, 600),
                                         (inputs.Q4_0, 300, 256, 3), (inputs.F16, 64, 1024, 40)])
def test_plan_matches_the_call(rg, variant, wtype, N, K, T):
    info = rg.rg_plan_info()
    rg.check(rg.rg_plan(variant, wtype, N, K, T, info), "rg_plan")
    expect = variant if variant else rg.rg_select_variant(wtype, N, K, T)
    assert info.variant == expect
    assert info.decode_ops == -(-T // info.tile_t) * N * K
    assert info.workspace_bytes == rg.rg_workspace_bytes(expect, wtype, N, K, T)
    assert (info.cta_group in (1, 2)) == (expect in (1, 4, 5))
    assert info.n_splits >= 1 and info.grid >= 1
    W = inputs.gen_weight(wtype, N, K, seed=5, stream=1)
    dY = inputs.normal_f32(5, 2, T * N, 1e-3).reshape(T, N)
    torch.cuda.synchronize()
    before = rg.rg_launch_count()
    got = run_out_prod(rg, variant, wtype, W, N, K, dY, T)
    assert rg.rg_launch_count() - before == info.launches
    ref = oracle.out_prod(wtype, W, N, K, dY, T)
    assert_within(got, ref, oracle.abs_bound(dY, oracle.dequant(wtype, W, N, K)), TOL[expect], "plan")


def test_plan_of_empty_shapes(rg):
    info = rg.rg_plan_info()
    rg.check(rg.rg_plan(0, inputs.Q8_0, 64, 256, 0, info))
    assert info.launches == 0 and info.decode_ops == 0
    rg.check(rg.rg_plan(0, inputs.Q8_0, 0, 256, 8, info))
    assert info.launches == 1 and info.decode_ops == 0


# ----------------------------------------------------------------------------
# the fp16 operand range

@pytest.mark.parametrize("strided", [False, True])
def test_dy_beyond_fp16_range_is_reported_not_silent(rg, strided):
    """One |dY| = 1e5 element, beyond fp16's largest value: the tensor-core
    call on an fp16 kind (Q4_K W) reports RG_ERR_RANGE through rg_check (the
    read clears it), so an inf in dX never goes unreported; the bf16 kind
    (BF16 W) takes the same dY within its bound, and so does the SIMT
    variant for the Q4_K weight.  Strided: dY given transposed (the tiled
    conversion)."""
    N, K, T = 300, 512, 64
    dY = inputs.normal_f32(61, 2, T * N, 1e-3).reshape(T, N)
    dY[5, 17] = -1.0e5
    dev, s = _dev(), torch.cuda.current_stream()
    for wtype, variant, expect in ((inputs.Q4_K, 1, rg.RG_ERR_RANGE), (inputs.BF16, 1, rg.RG_OK),
                                   (inputs.Q4_K, 3, rg.RG_OK)):
        W = inputs.gen_weight(wtype, N, K, seed=61, stream=1)
        Wt = torch.from_numpy(W).to(dev)
        dX = torch.full((T, K), float("nan"), device=dev)
        if strided:
            dYt = torch.from_numpy(np.ascontiguousarray(dY.T)).to(dev)   # [N, T]: dY[t, n] at n*T + t
            st = rg.rg_out_prod_ex(variant, wtype, Wt, N, K, 0, dYt, T, 1, T, 0, dX, K, 0, 1, 0.0, s)
        else:
            st = rg.rg_out_prod_variant(variant, wtype, Wt, N, K, torch.from_numpy(dY).to(dev), T,
                                        dX, 0.0, s)
        assert st == rg.RG_OK
        assert rg.rg_check(s) == expect, (wtype, variant)
        assert rg.rg_check(s) == rg.RG_OK          # read and cleared
        if expect == rg.RG_OK:
            Wd = oracle.dequant(wtype, W, N, K)
            assert_within(dX.cpu().numpy(), oracle.out_prod(wtype, W, N, K, dY, T, Wd=Wd),
                          oracle.abs_bound(dY, Wd), TOL[variant], f"range {wtype} {variant}")
