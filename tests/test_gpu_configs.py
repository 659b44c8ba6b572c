"""GPU parity at the full sizes of every workload, in the launch configuration
the bench times (rg_out_prod, dispatcher's choice): the oracle computes
sampled outputs one by one (4096 random (t, k) pairs plus the whole first and
last rows) and rg_dequant is compared bit for bit on the full weight."""
import numpy as np
import pytest

import oracle
from quantized_weight_out_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

CASES = [(w, i) for w in sorted(inputs.WORKLOADS) if w != "layer7b_gate_t8192"
         for i in range(len(inputs.WORKLOADS[w]))]


@pytest.fixture(scope="module")
def rg():
    from quantized_weight_out_gb300 import binding, build
    build.build()
    binding.load()
    return binding


@pytest.mark.parametrize("workload,idx", CASES)
def test_full_size_sampled(rg, workload, idx):
    p = inputs.WORKLOADS[workload][idx]
    dev = torch.device("cuda:0")
    W = p.weight()
    dY = p.dy()
    dX0 = p.dx0()
    Wt = torch.from_numpy(W).to(dev)
    dYt = torch.from_numpy(dY).to(dev)
    dX = torch.from_numpy(dX0).to(dev) if dX0 is not None else \
        torch.full((p.T, p.K), float("nan"), device=dev)
    s = torch.cuda.current_stream()
    rg.check(rg.rg_out_prod(p.wtype, Wt, p.N, p.K, dYt, p.T, dX, p.beta, s))
    # the decode, bit for bit, on the whole weight
    Wd_gpu = torch.empty((p.N, p.K), device=dev)
    rg.check(rg.rg_dequant_async(p.wtype, Wt, p.N, p.K, Wd_gpu, s))
    rg.check(rg.rg_check(s))
    Wd = oracle.dequant(p.wtype, W, p.N, p.K)
    assert np.array_equal(Wd_gpu.cpu().numpy().view(np.uint32), Wd.view(np.uint32))
    del Wd_gpu
    got = dX.cpu().numpy()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(idx + 17)
    ts = np.concatenate([rng.integers(0, p.T, 4096), np.zeros(p.K, np.int64),
                         np.full(p.K, p.T - 1, np.int64)])
    ks = np.concatenate([rng.integers(0, p.K, 4096), np.arange(p.K), np.arange(p.K)])
    ref, bnd = oracle.out_prod_at(Wd, dY, ts, ks, dX0, p.beta)
    g = got[ts, ks].astype(np.float64)
    lim = 5e-3 * bnd + 1e-7
    if p.beta != 0.0:
        lim = lim + np.abs(p.beta * dX0[ts, ks]) * 2.0 ** -24
    err = np.abs(g - ref)
    assert np.all(err <= lim), (workload, int((err > lim).sum()), float(err.max()))
