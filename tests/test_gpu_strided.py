"""rg_out_prod_ex: strided, transposed and batched dY / dX against the oracle."""
import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {0: 5e-3, 1: 5e-3, 2: 5e-3, 3: 1e-5, 4: 5e-3, 5: 5e-3}


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def _check(got, ref, bnd, tol, what):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= tol * bnd + 1e-7), (what, float(err.max()))


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0, inputs.F16])
def test_transposed_dy_and_padded_dx(rg, variant, wtype):
    """dY given as grad^T ([N, T] contiguous: dy_t = 1, dy_n = T) and dX rows
    padded to K + 12, beta = 1: values match, the padding is untouched."""
    N, K, T = 300, 512, 90
    W = inputs.gen_weight(wtype, N, K, seed=51, stream=1)
    dY = inputs.normal_f32(51, 2, T * N, 1e-3).reshape(T, N)
    dX0 = inputs.normal_f32(51, 3, T * K, 1e-3).reshape(T, K)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    dYT = torch.from_numpy(np.ascontiguousarray(dY.T)).to(dev)           # [N, T]
    ldx = K + 12
    buf = torch.full((T, ldx), 7.0, device=dev)
    buf[:, :K] = torch.from_numpy(dX0).to(dev)
    Wt = torch.from_numpy(W).to(dev)
    st = rg.rg_out_prod_ex(variant, wtype, Wt, N, K, 0, dYT, T, 1, T, 0, buf, ldx, 0, 1, 1.0, s)
    rg.check(st, "rg_out_prod_ex")
    rg.check(rg.rg_check(s))
    out = buf.cpu().numpy()
    assert np.all(out[:, K:] == 7.0)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, dX0, 1.0, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd) + np.abs(dX0) * 2.0 ** -24 / TOL[variant]
    _check(out[:, :K], ref, bnd, TOL[variant], f"variant {variant}")


@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0, inputs.F16])
def test_small_t_one_slice_writes_dx(rg, wtype):
    """At most 256 rows of W: one small-T kernel per call takes all the rows
    of its tile and writes dX itself (beta applied, padded rows, padding
    untouched), with no partial sums and no second kernel."""
    N, K, T, beta = 200, 512, 6, -0.5
    info = rg.rg_plan_info()
    rg.check(rg.rg_plan(2, wtype, N, K, T, info), "rg_plan")
    assert info.n_splits == 1 and info.launches == 1 and info.workspace_bytes == 0, info.as_dict()
    W = inputs.gen_weight(wtype, N, K, seed=53, stream=1)
    dY = inputs.normal_f32(53, 2, T * N, 1e-3).reshape(T, N)
    dX0 = inputs.normal_f32(53, 3, T * K, 1e-3).reshape(T, K)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    ldx = K + 4
    buf = torch.full((T, ldx), 7.0, device=dev)
    buf[:, :K] = torch.from_numpy(dX0).to(dev)
    torch.cuda.synchronize()
    before = rg.rg_launch_count()
    rg.check(rg.rg_out_prod_ex(2, wtype, torch.from_numpy(W).to(dev), N, K, 0,
                               torch.from_numpy(dY).to(dev), T, N, 1, 0, buf, ldx, 0, 1, beta, s))
    rg.check(rg.rg_check(s))
    assert rg.rg_launch_count() - before == 1
    out = buf.cpu().numpy()
    assert np.all(out[:, K:] == 7.0)
    Wd = oracle.dequant(wtype, W, N, K)
    ref = oracle.out_prod(wtype, W, N, K, dY, T, dX0, beta, Wd=Wd)
    bnd = oracle.abs_bound(dY, Wd) + np.abs(beta * dX0) * 2.0 ** -24 / 5e-3
    _check(out[:, :K], ref, bnd, 5e-3, "one slice")


@pytest.mark.parametrize("variant", [0, 2, 3])
def test_padded_dy_rows(rg, variant):
    """dY rows N + 5 floats apart (only 4-byte aligned)."""
    N, K, T, wtype = 200, 256, 33, inputs.Q4_0
    W = inputs.gen_weight(wtype, N, K, seed=52, stream=1)
    dY = inputs.normal_f32(52, 2, T * N, 1e-3).reshape(T, N)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    pad = np.zeros((T, N + 5), np.float32)
    pad[:, :N] = dY
    dYp = torch.from_numpy(pad).to(dev)
    dX = torch.full((T, K), float("nan"), device=dev)
    rg.check(rg.rg_out_prod_ex(variant, wtype, torch.from_numpy(W).to(dev), N, K, 0, dYp, T, N + 5, 1,
                               0, dX, K, 0, 1, 0.0, s))
    rg.check(rg.rg_check(s))
    Wd = oracle.dequant(wtype, W, N, K)
    _check(dX.cpu().numpy(), oracle.out_prod(wtype, W, N, K, dY, T, Wd=Wd), oracle.abs_bound(dY, Wd),
           TOL[variant], "padded dY")


@pytest.mark.parametrize("shared_w", [True, False])
def test_batches(rg, shared_w):
    """Three batches: a shared W (stacked into one call) or one W each (run in
    turn), each batch's dY and dX at its own offset."""
    B, N, K, T, wtype = 3, 256, 512, 70, inputs.Q5_K
    rb = inputs.row_bytes(wtype, K)
    Ws = [inputs.gen_weight(wtype, N, K, seed=60 + (0 if shared_w else b), stream=1) for b in range(B)]
    dYs = [inputs.normal_f32(61 + b, 2, T * N, 1e-3).reshape(T, N) for b in range(B)]
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Wall = torch.from_numpy(np.concatenate(Ws if not shared_w else Ws[:1])).to(dev)
    dYall = torch.from_numpy(np.concatenate(dYs)).to(dev)                # [B*T, N]
    dX = torch.empty((B * T, K), device=dev)
    rg.check(rg.rg_out_prod_ex(0, wtype, Wall, N, K, 0 if shared_w else N * rb, dYall, T, N, 1, T * N,
                               dX, K, T * K, B, 0.0, s))
    rg.check(rg.rg_check(s))
    got = dX.cpu().numpy().reshape(B, T, K)
    for b in range(B):
        Wd = oracle.dequant(wtype, Ws[b], N, K)
        _check(got[b], oracle.out_prod(wtype, Ws[b], N, K, dYs[b], T, Wd=Wd),
               oracle.abs_bound(dYs[b], Wd), 5e-3, f"batch {b}")


def test_strided_batches_run_in_turn(rg):
    """Batches whose dX are interleaved column blocks of one wide array (not
    stackable): dX_b = out[:, b*K:(b+1)*K], dY transposed per batch."""
    B, N, K, T, wtype = 2, 128, 256, 40, inputs.Q8_0
    W = inputs.gen_weight(wtype, N, K, seed=70, stream=1)
    dYs = [inputs.normal_f32(71 + b, 2, T * N, 1e-3).reshape(T, N) for b in range(B)]
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    dYT = torch.from_numpy(np.concatenate([np.ascontiguousarray(d.T) for d in dYs])).to(dev)  # [B*N, T]
    out = torch.empty((T, B * K), device=dev)
    rg.check(rg.rg_out_prod_ex(0, wtype, torch.from_numpy(W).to(dev), N, K, 0, dYT, T, 1, T, N * T,
                               out, B * K, K, B, 0.0, s))
    rg.check(rg.rg_check(s))
    got = out.cpu().numpy()
    Wd = oracle.dequant(wtype, W, N, K)
    for b in range(B):
        _check(got[:, b * K:(b + 1) * K], oracle.out_prod(wtype, W, N, K, dYs[b], T, Wd=Wd),
               oracle.abs_bound(dYs[b], Wd), 5e-3, f"batch {b}")


def _batched_case(wtype, N, K, T, n2, n3, w_n2, w_n3, seed):
    Ws = [[inputs.gen_weight(wtype, N, K, seed=seed + 10 * j3 + j2, stream=1) for j2 in range(w_n2)]
          for j3 in range(w_n3)]
    dYs = [[inputs.normal_f32(seed + 100 + 10 * i3 + i2, 2, T * N, 1e-3).reshape(T, N)
            for i2 in range(n2)] for i3 in range(n3)]
    return Ws, dYs


@pytest.mark.parametrize("n2,w_n2,n3,w_n3", [(8, 4, 1, 1), (8, 2, 1, 1), (4, 2, 3, 1), (2, 1, 4, 2)])
def test_batched_broadcast_stacks_each_weights_run(rg, n2, w_n2, n3, w_n3):
    """Fewer weights than gradient batches (ratio 2 and 4 along dim 2, and two
    batch dims): batch (i2, i3) reads weight (i2 / (n2 / w_n2), i3 / (n3 /
    w_n3)).  dY and dX batches are stacked in memory, so the batches one weight
    serves run as one call (counted by the library's launches), and every
    batch matches the oracle's batched product."""
    wtype, N, K, T = inputs.Q4_K, 320, 512, 48
    rb = inputs.row_bytes(wtype, K)
    Ws, dYs = _batched_case(wtype, N, K, T, n2, n3, w_n2, w_n3, 80)
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Wall = torch.from_numpy(np.concatenate([w for row in Ws for w in row])).to(dev)   # [j3][j2]
    dYall = torch.from_numpy(np.concatenate([d for row in dYs for d in row])).to(dev)  # [i3][i2][T, N]
    dX = torch.full((n3 * n2 * T, K), float("nan"), device=dev)
    r2, r3 = n2 // w_n2, n3 // w_n3
    # calls: runs of consecutive batches (i2 fastest) reading one weight
    runs = 0
    prev = None
    for i3 in range(n3):
        for i2 in range(n2):
            w = oracle.batch_weight(i2, i3, n2, n3, w_n2, w_n3)
            runs += w != prev
            prev = w
    info = rg.rg_plan_info()
    torch.cuda.synchronize()
    before = rg.rg_launch_count()
    rg.check(rg.rg_out_prod_batched(0, wtype, Wall, N, K, w_n2, w_n3, N * rb, w_n2 * N * rb,
                                    dYall, T, N, 1, T * N, n2 * T * N, dX, K, T * K, n2 * T * K,
                                    n2, n3, 0.0, s), "rg_out_prod_batched")
    rg.check(rg.rg_check(s))
    launches = rg.rg_launch_count() - before
    expect = 0
    # each run is one call over T * (its batches) rows
    lens, prev, cur = [], None, 0
    for i3 in range(n3):
        for i2 in range(n2):
            w = oracle.batch_weight(i2, i3, n2, n3, w_n2, w_n3)
            if w != prev and cur:
                lens.append(cur)
                cur = 0
            prev = w
            cur += 1
    lens.append(cur)
    assert len(lens) == runs
    for c in lens:
        rg.check(rg.rg_plan(0, wtype, N, K, T * c, info))
        expect += info.launches
    assert launches == expect
    got = dX.cpu().numpy().reshape(n3, n2, T, K)
    ref = oracle.out_prod_batched(wtype, Ws, N, K, dYs, T)
    for i3 in range(n3):
        for i2 in range(n2):
            j2, j3 = oracle.batch_weight(i2, i3, n2, n3, w_n2, w_n3)
            Wd = oracle.dequant(wtype, Ws[j3][j2], N, K)
            _check(got[i3, i2], ref[i3][i2], oracle.abs_bound(dYs[i3][i2], Wd), 5e-3, f"({i2}, {i3})")


def test_batched_transposed_gradients_run_in_turn(rg):
    """Two batch dims with dY given transposed per batch (not stackable) and
    beta = 1 on an interleaved dX: each batch is its own call, and each
    matches the oracle."""
    wtype, N, K, T = inputs.Q8_0, 128, 256, 40
    n2, n3, w_n2, w_n3 = 4, 2, 2, 2
    rb = inputs.row_bytes(wtype, K)
    Ws, dYs = _batched_case(wtype, N, K, T, n2, n3, w_n2, w_n3, 90)
    dX0s = [[inputs.normal_f32(95 + 10 * i3 + i2, 3, T * K, 1e-3).reshape(T, K) for i2 in range(n2)]
            for i3 in range(n3)]
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    Wall = torch.from_numpy(np.concatenate([w for row in Ws for w in row])).to(dev)
    dYT = torch.from_numpy(np.concatenate([np.ascontiguousarray(d.T) for row in dYs for d in row])).to(dev)
    # dX: [T, n3, n2, K] (batches interleaved inside each row)
    out = np.stack([np.stack(row, axis=1) for row in dX0s], axis=1)    # [T, n3, n2, K]
    dX = torch.from_numpy(np.ascontiguousarray(out)).to(dev)
    rg.check(rg.rg_out_prod_batched(0, wtype, Wall, N, K, w_n2, w_n3, N * rb, w_n2 * N * rb,
                                    dYT, T, 1, T, N * T, n2 * N * T, dX, n3 * n2 * K, K, n2 * K,
                                    n2, n3, 1.0, s), "rg_out_prod_batched")
    rg.check(rg.rg_check(s))
    got = dX.cpu().numpy()
    ref = oracle.out_prod_batched(wtype, Ws, N, K, dYs, T, dX0s, 1.0)
    for i3 in range(n3):
        for i2 in range(n2):
            j2, j3 = oracle.batch_weight(i2, i3, n2, n3, w_n2, w_n3)
            Wd = oracle.dequant(wtype, Ws[j3][j2], N, K)
            bnd = oracle.abs_bound(dYs[i3][i2], Wd) + np.abs(dX0s[i3][i2]) * 2.0 ** -24 / 5e-3
            _check(got[:, i3, i2, :], ref[i3][i2], bnd, 5e-3, f"({i2}, {i3})")
