"""Stream-K plans of the tensor-core kernel against the oracle.

When the output tiles fill at least one wave of persistent units but not
the last, the kernel gives every unit its whole tiles and then an even share
of the last tiles' contraction chunks.  Of a tile shared by several units,
the piece with the first chunk writes dX (beta applied) and the others write
partial slabs, which a second kernel adds to dX in chunk order.  These
shapes take that plan (rg_plan reports it), with a ragged T, K and N, beta,
one-CTA tiles, both 16-bit kinds and the window decoders; sampled outputs
are checked against the oracle's bound and whole results for being the same
on every call."""
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


def _plan(rg, variant, wtype, N, K, T):
    info = rg.rg_plan_info()
    rg.check(rg.rg_plan(variant, wtype, N, K, T, info), "rg_plan")
    return info


def _call(rg, variant, wtype, W, N, K, dY, T, dX0, beta):
    dev, s = torch.device("cuda:0"), torch.cuda.current_stream()
    dX = (torch.from_numpy(dX0).to(dev) if dX0 is not None
          else torch.full((T, K), float("nan"), device=dev))
    rg.check(rg.rg_out_prod_variant(variant, wtype, torch.from_numpy(W).to(dev), N, K,
                                    torch.from_numpy(dY).to(dev), T, dX, beta, s))
    rg.check(rg.rg_check(s))
    return dX.cpu().numpy()


def _sampled(rg, case, seed):
    """The call twice (bit-identical), and 4096 random outputs plus the whole
    first and last rows and a row of the last t tile against the oracle."""
    wtype, N, K, T, variant, beta = case
    info = _plan(rg, variant, wtype, N, K, T)
    assert info.stream_k == 1 and info.n_splits == 1, info.as_dict()
    W = inputs.gen_weight(wtype, N, K, seed=seed, stream=1)
    dY = inputs.normal_f32(seed, 2, T * N, 1e-3).reshape(T, N)
    dX0 = inputs.normal_f32(seed, 3, T * K, 1e-3).reshape(T, K) if beta else None
    torch.cuda.synchronize()
    before = rg.rg_launch_count()
    got = _call(rg, variant, wtype, W, N, K, dY, T, dX0, beta)
    # the dY conversion, the main kernel and the pass over the shared tiles
    # (and F32 W's conversion)
    assert rg.rg_launch_count() - before == info.launches
    again = _call(rg, variant, wtype, W, N, K, dY, T, dX0, beta)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32)), "not deterministic"
    Wd = oracle.dequant(wtype, W, N, K)
    rng = np.random.default_rng(seed)
    last = (T - 1) // 256 * 256
    ts = np.concatenate([rng.integers(0, T, 4096), np.zeros(K, np.int64), np.full(K, T - 1, np.int64),
                         np.full(K, last, np.int64)])
    ks = np.concatenate([rng.integers(0, K, 4096), np.arange(K), np.arange(K), np.arange(K)])
    ref, bnd = oracle.out_prod_at(Wd, dY, ts, ks, dX0, beta)
    if beta:
        bnd = bnd + np.abs(beta * dX0[ts, ks]) * 2.0 ** -24 / 5e-3
    err = np.abs(got[ts, ks].astype(np.float64) - ref)
    assert np.all(err <= 5e-3 * bnd + 1e-7), (case, float(err.max()))


CASES = [  # (wtype, N, K, T, variant, beta): one whole wave, then shared tiles
    (inputs.Q4_K, 2048, 2304, 2560, 0, 0.0),   # 90 pair tiles on 76 pairs
    (inputs.Q8_0, 2048, 2304, 2500, 5, 1.0),   # ragged T, beta
    (inputs.F16, 2052, 2296, 2560, 5, 0.0),    # ragged N (a partial last chunk) and K
    (inputs.BF16, 2048, 2304, 2560, 5, 1.0),   # bf16 operands, beta
    (inputs.Q4_0, 4864, 2048, 1280, 4, 0.0),   # one-CTA tiles: 160 tiles on 152 CTAs
    (inputs.Q6_K, 2048, 4096, 1536, 5, 0.0),   # window decoders
    (inputs.Q2_K, 2560, 3072, 1700, 5, 0.5),
]


@pytest.mark.parametrize("case", CASES)
def test_stream_k_parity(rg, case):
    _sampled(rg, case, 71)


def test_stream_k_after_whole_waves(rg):
    """80 pair tiles on 76 pairs: one whole wave, then 4 tiles' chunks over
    every pair (each shared tile split over about 20 units)."""
    _sampled(rg, (inputs.Q4_K, 8192, 2048, 2560, 0, 0.0), 72)


def test_fewer_tiles_than_units_keep_splits(rg):
    """With fewer tiles than units the plan splits the contraction instead
    (a split's reduction is cheaper than sharing every tile)."""
    info = _plan(rg, 0, inputs.Q4_0, 4096, 4096, 512)
    assert info.stream_k == 0 and info.n_splits > 1, info.as_dict()
