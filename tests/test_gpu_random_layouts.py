"""Seeded random memory layouts through rg_out_prod_batched and random
adapters through rg_out_prod_lora, against the oracle.

Batched cases draw two batch dimensions with fewer weights than gradient
batches (each weight count dividing the gradient's), dY stacked, with padded
rows or transposed per batch, and dX stacked, with padded rows or as
interleaved column blocks of one wide array; every batch is compared with
the oracle's product for the weight ggml's broadcast rule gives it, and the
memory between the batches' dX rows must be left untouched.  LoRA cases
draw the rank (0 to 69; every eighth case 0), the scale, beta and the
variant.  A call the library rejects for its documented shape or alignment
rules is skipped."""
import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
needs_gpu = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

N_BATCHED, N_LORA = 60, 40
ALIGN = {inputs.Q6_K: 2048, inputs.Q3_K: 2048, inputs.Q2_K: 1024, inputs.MXFP4: 512}
HALF = (inputs.F16, inputs.BF16, inputs.F32)
TOL = {1: 5e-3, 2: 5e-3, 3: 1e-5, 4: 5e-3, 5: 5e-3}
LORA_TOL = {1: 1e-2, 2: 1e-5, 3: 1e-5, 4: 1e-2, 5: 1e-2}
SENTINEL = 7.0


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _common(rng):
    wt = int(rng.choice(inputs.ALL_TYPES))
    variant = int(rng.choice([0, 0, 1, 2, 3, 4, 5]))
    N = int(rng.integers(1, 600))
    K = int(rng.integers(1, 5)) * (8 if wt in HALF else 256)
    if wt in HALF and rng.random() < 0.5:
        K = int(rng.integers(1, 5)) * 256
    if wt in ALIGN and variant != 3:
        K = -(-K // ALIGN[wt]) * ALIGN[wt]
    T = int(rng.integers(1, 9)) if rng.random() < 0.35 else int(rng.integers(9, 300))
    beta = float(rng.choice([0.0, 0.0, 1.0, -0.5]))
    return wt, variant, N, K, T, beta


def draw_batched(i: int) -> dict:
    rng = np.random.default_rng([104729, i])
    wt, variant, N, K, T, beta = _common(rng)
    n2, n3 = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    w_n2 = int(rng.choice([d for d in range(1, n2 + 1) if n2 % d == 0]))
    w_n3 = int(rng.choice([d for d in range(1, n3 + 1) if n3 % d == 0]))
    return dict(wt=wt, variant=variant, N=N, K=K, T=T, beta=beta, n2=n2, n3=n3, w_n2=w_n2, w_n3=w_n3,
                lay_y=str(rng.choice(["stack", "pad", "trans"])), pad_y=int(rng.integers(1, 8)),
                lay_x=str(rng.choice(["stack", "pad", "wide"])), pad_x=4 * int(rng.integers(1, 4)),
                seed=9000 + 97 * i)


def draw_lora(i: int) -> dict:
    rng = np.random.default_rng([130363, i])
    wt, variant, N, K, T, beta = _common(rng)
    R = 0 if i % 8 == 0 else int(rng.integers(1, 70))
    return dict(wt=wt, variant=variant, N=N, K=K, T=T, beta=beta, R=R,
                scale=float(rng.choice([0.5, 2.0, -1.0])), seed=12000 + i)


def test_layout_draws_cover_every_form():
    """(host only) the draws reach every dY and dX layout, weight broadcast
    along both batch dimensions, every variant and rank 0."""
    b = [draw_batched(i) for i in range(N_BATCHED)]
    assert {(c["lay_y"], c["lay_x"]) for c in b} == {(y, x) for y in ("stack", "pad", "trans")
                                                     for x in ("stack", "pad", "wide")}
    assert any(c["w_n2"] < c["n2"] for c in b) and any(c["w_n3"] < c["n3"] for c in b)
    lo = [draw_lora(i) for i in range(N_LORA)]
    assert {c["variant"] for c in lo} == {0, 1, 2, 3, 4, 5} and any(c["R"] == 0 for c in lo)


@needs_gpu[0]
@needs_gpu[1]
@pytest.mark.parametrize("i", range(N_BATCHED))
def test_random_batched_layout(rg, i):
    c = draw_batched(i)
    wt, N, K, T, beta, seed = c["wt"], c["N"], c["K"], c["T"], c["beta"], c["seed"]
    n2, n3, w_n2, w_n3 = c["n2"], c["n3"], c["w_n2"], c["w_n3"]
    nb, rb = n2 * n3, inputs.row_bytes(wt, K)
    Ws = [[inputs.gen_weight(wt, N, K, seed=seed + 10 * j3 + j2, stream=1) for j2 in range(w_n2)]
          for j3 in range(w_n3)]
    dYs = [[inputs.normal_f32(seed + 1 + 10 * i3 + i2, 2, T * N, 1e-3).reshape(T, N) for i2 in range(n2)]
           for i3 in range(n3)]
    dX0s = [[inputs.normal_f32(seed + 2 + 10 * i3 + i2, 3, T * K, 1e-3).reshape(T, K) for i2 in range(n2)]
            for i3 in range(n3)]
    # dY: batch b = i3 * n2 + i2 at b * per
    if c["lay_y"] == "trans":
        dy_t, dy_n, per = 1, T, N * T
        ybuf = np.concatenate([np.ascontiguousarray(dYs[i3][i2].T).reshape(-1)
                               for i3 in range(n3) for i2 in range(n2)])
    else:
        dy_t = N + (c["pad_y"] if c["lay_y"] == "pad" else 0)
        dy_n, per = 1, T * dy_t
        ybuf = np.zeros(nb * per, np.float32)
        for i3 in range(n3):
            for i2 in range(n2):
                b = i3 * n2 + i2
                ybuf[b * per:(b + 1) * per].reshape(T, dy_t)[:, :N] = dYs[i3][i2]
    # dX: rows of batch (i2, i3) at i2 * xs2 + i3 * xs3 + t * dx_t
    if c["lay_x"] == "wide":
        dx_t, xs2, xs3, total = nb * K, K, n2 * K, T * nb * K
    else:
        dx_t = K + (c["pad_x"] if c["lay_x"] == "pad" else 0)
        xs2, xs3, total = T * dx_t, n2 * T * dx_t, nb * T * dx_t
    xbuf = np.full(total, SENTINEL, np.float32)
    rows = {}
    for i3 in range(n3):
        for i2 in range(n2):
            idx = (i2 * xs2 + i3 * xs3 + np.arange(T)[:, None] * dx_t + np.arange(K)[None, :])
            rows[(i2, i3)] = idx
            xbuf[idx] = dX0s[i3][i2] if beta else np.nan
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Wall = torch.from_numpy(np.concatenate([w for row in Ws for w in row])).to(dev)
    Xd = torch.from_numpy(xbuf).to(dev)
    st = rg.rg_out_prod_batched(c["variant"], wt, Wall, N, K, w_n2, w_n3, N * rb, w_n2 * N * rb,
                                torch.from_numpy(ybuf).to(dev), T, dy_t, dy_n, per, n2 * per,
                                Xd, dx_t, xs2, xs3, n2, n3, beta, s)
    if st in (rg.RG_ERR_SHAPE, rg.RG_ERR_ALIGN):
        pytest.skip(f"rejected by the documented rules ({rg.strerror(st)}): {c}")
    rg.check(st, f"rg_out_prod_batched {c}")
    rg.check(rg.rg_check(s), f"rg_check {c}")
    got = Xd.cpu().numpy()
    untouched = np.ones(total, bool)
    tol = TOL[c["variant"] or rg.rg_select_variant(wt, N, K, T)]
    for (i2, i3), idx in rows.items():
        untouched[idx] = False
        j2, j3 = oracle.batch_weight(i2, i3, n2, n3, w_n2, w_n3)
        Wd = oracle.dequant(wt, Ws[j3][j2], N, K)
        ref = oracle.out_prod(wt, Ws[j3][j2], N, K, dYs[i3][i2], T, dX0s[i3][i2], beta, Wd=Wd)
        bnd = oracle.abs_bound(dYs[i3][i2], Wd)
        lim = tol * bnd + 1e-7 + (np.abs(beta * dX0s[i3][i2].astype(np.float64)) * 2.0 ** -23 if beta else 0.0)
        err = np.abs(got[idx].astype(np.float64) - ref)
        assert np.all(err <= lim), (c, (i2, i3), float(np.nanmax(err / (bnd + 1e-30))))
    assert np.all(got[untouched] == SENTINEL), c


@needs_gpu[0]
@needs_gpu[1]
@pytest.mark.parametrize("i", range(N_LORA))
def test_random_lora(rg, i):
    c = draw_lora(i)
    wt, N, K, T, beta, R, scale, seed = (c[k] for k in ("wt", "N", "K", "T", "beta", "R", "scale", "seed"))
    variant = c["variant"] or rg.rg_select_variant(wt, N, K, T)  # the automatic choice's tolerance
    W = inputs.gen_weight(wt, N, K, seed=seed, stream=1)
    dY = inputs.normal_f32(seed, 2, T * N, 1.0).reshape(T, N)
    A = inputs.normal_f32(seed, 3, R * K, 0.05).reshape(R, K)
    B = inputs.normal_f32(seed, 4, N * R, 0.05).reshape(N, R)
    dX0 = inputs.normal_f32(seed, 5, T * K, 1.0).reshape(T, K)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    dX = t(dX0) if beta else torch.full((T, K), float("nan"), device=dev)
    Ad = t(A) if R > 0 else torch.zeros(4, device=dev)
    Bd = t(B) if R > 0 else torch.zeros(4, device=dev)
    st = rg.rg_out_prod_lora(c["variant"], wt, t(W), N, K, t(dY), T, dX, beta, Ad, Bd, R, scale, s)
    if st in (rg.RG_ERR_SHAPE, rg.RG_ERR_ALIGN):
        pytest.skip(f"rejected by the documented rules ({rg.strerror(st)}): {c}")
    rg.check(st, f"rg_out_prod_lora {c}")
    rg.check(rg.rg_check(s), f"rg_check {c}")
    Wd = oracle.dequant(wt, W, N, K)
    ref = oracle.out_prod_lora(wt, W, N, K, dY, T, A, B, R, scale, dX0, beta, Wd=Wd)
    b_base = oracle.abs_bound(dY, Wd)
    b_lora = oracle.lora_bound(dY, A, B, scale) if R > 0 else 0.0
    lim = (TOL[variant] * b_base + LORA_TOL[variant] * b_lora + 1e-7
           + (np.abs(beta * dX0.astype(np.float64)) * 2.0 ** -23 if beta else 0.0))
    err = np.abs(dX.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= lim), (c, float(np.nanmax(err / (b_base + b_lora + 1e-30))))
