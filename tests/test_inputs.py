"""The seeded input generators: deterministic, the stated distributions, and
valid encodings (these affect inputs only, never parity)."""
import numpy as np

from quantized_weight_out_gb300 import inputs


def test_splitmix64_reference_values():
    # SplitMix64 from state 0: the first outputs of the published generator
    # (Steele, Lea, Flood 2014; also java.util.SplittableRandom's mix).
    out = inputs._mix(np.arange(1, 4, dtype=np.uint64) * inputs._GAMMA)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_chunk_independent():
    a = inputs.normal_f32(0, 2, 10000, 1.0)
    b = inputs.normal_f32(0, 2, 10000, 1.0)
    assert np.array_equal(a, b)
    c = inputs.normal_f32(0, 3, 10000, 1.0)
    assert not np.array_equal(a, c)
    saved = inputs._CHUNK
    inputs._CHUNK = 777
    try:
        d = inputs.normal_f32(0, 2, 10000, 1.0)
    finally:
        inputs._CHUNK = saved
    assert np.array_equal(a, d)


def test_normal_moments():
    x = inputs.normal_f32(0, 2, 400000, 1e-3).astype(np.float64)
    assert abs(x.mean()) < 1e-5
    assert abs(x.std() / 1e-3 - 1) < 0.01


def test_uniform_int_range():
    v = inputs.uniform_int(0, 1, 100000, 64, field=3)
    assert v.min() == 0 and v.max() == 63
    assert abs(np.bincount(v, minlength=64).std() / (100000 / 64)) < 0.1


def test_q8_0_generator_fields():
    N, K = 8, 64
    W = inputs.gen_weight(inputs.Q8_0, N, K, 0, 1).reshape(N, K // 32, 34)
    q = W[..., 2:].view(np.int8)
    assert q.min() >= -127 and q.max() <= 127
    assert np.all(np.abs(q).max(axis=-1) == 127)    # amax maps to +-127


def test_q4_0_generator_fields():
    N, K = 8, 64
    W = inputs.gen_weight(inputs.Q4_0, N, K, 0, 1).reshape(N, K // 32, 18)
    d = W[..., 0:2].copy().view(np.float16)[..., 0]
    assert np.all(d != 0)
    lo, hi = W[..., 2:] & 15, W[..., 2:] >> 4
    nib = np.concatenate([lo, hi], -1)
    # the element of largest magnitude maps to q = 0 (value -8 * d = mx)
    assert np.all(nib.min(axis=-1) == 0)


def test_half_encoders_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -65504.0], dtype=np.float32)
    assert list(inputs.f32_to_f16_bits(x)) == [0x3C00, 0x3C00, 0x3C02, 0xFBFF]
    y = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -123.5], dtype=np.float32)
    assert list(inputs.f32_to_bf16_bits(y)) == [0x3F80, 0x3F80, 0x3F82, 0xC2F7]


def test_workloads_and_row_bytes():
    w = inputs.WORKLOADS
    assert [p.N for p in w["layer7b_t8192"]] == [4096, 1024, 1024, 4096, 14336, 14336, 4096]
    assert w["layer7b_t8192"][-1].wtype == inputs.Q8_0
    assert w["f16_5120x17408_t4096_beta1"][0].beta == 1.0
    assert sum(p.flops for p in w["layer7b_t8192"]) == 3_573_412_790_272
    assert w["q4_k_14336x4096_t2048"][0].w_bytes == 33_030_144


def test_row_prefixes_are_smaller_calls():
    """The first rows of every generated input equal a smaller call's."""
    for wt in inputs.ALL_TYPES:
        p = inputs.Problem("x", wt, 40, 512, 12, 1e-3, 1.0, stream_base=32)
        rb = inputs.row_bytes(wt, 512)
        assert np.array_equal(p.weight()[: 7 * rb], p.weight(7))
        assert np.array_equal(p.dy()[:5], p.dy(5))
        assert np.array_equal(p.dx0()[:3], p.dx0(3))
