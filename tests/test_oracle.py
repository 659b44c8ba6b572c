"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against one of: hand-decoded blocks (fixtures
under tests/golden, derived from the GGUF block definitions), an independent
library routine (Python's struct half-float codec, numpy's float16, torch's
bfloat16), closed forms, a brute-force pure-Python evaluation with exactly
rounded sums, or an algebraic invariant.  The mutation tests at the end plant
plausible mistakes in copies of the oracle's steps and check that a pin
catches each of them.
"""
import math
import os
import struct

import numpy as np
import pytest

import oracle
from oracle import quant_out_prod as qop
from quantized_weight_out_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------
# fixture readers

def _read(golden_dir, name):
    rows = []
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _bits_equal(a, b):
    a = np.asarray(a, dtype=np.float32).view(np.uint32)
    b = np.asarray(b, dtype=np.float32).view(np.uint32)
    return np.array_equal(a, b)


# ----------------------------------------------------------------------------
# hand-decoded blocks

def test_q8_0_hand_block(golden_dir):
    rows = dict((r[0], r[1:]) for r in _read(golden_dir, "q8_0_block.txt"))
    W = np.frombuffer(bytes.fromhex(rows["hex"][0]), dtype=np.uint8)
    want = np.array([float(v) for v in rows["values"]], dtype=np.float32)
    got = oracle.decode_q8_0(W, 1, 32)[0]
    assert _bits_equal(got, want)


def test_q4_0_hand_block_nibble_order_and_negative_zero(golden_dir):
    rows = dict((r[0], r[1:]) for r in _read(golden_dir, "q4_0_block.txt"))
    W = np.frombuffer(bytes.fromhex(rows["hex"][0]), dtype=np.uint8)
    want = np.array([float(v) for v in rows["values"]], dtype=np.float32)
    got = oracle.decode_q4_0(W, 1, 32)[0]
    # bitwise: includes the sign of the two zeros (d < 0 times 0 is -0.0)
    assert _bits_equal(got, want)
    assert np.signbit(got[8]) and np.signbit(got[23])


def _q4_k_fixture(golden_dir):
    rows = _read(golden_dir, "q4_k_superblock.txt")
    kv = {}
    ats, rng = [], None
    for r in rows:
        if r[0] == "at":
            ats.append((int(r[1]), float(r[2])))
        elif r[0] == "range":
            rng = (int(r[1]), int(r[2]), float(r[3]))
        else:
            kv[r[0]] = r[1:]
    blk = bytearray(144)
    blk[0:2] = int(kv["d"][0], 16).to_bytes(2, "little")
    blk[2:4] = int(kv["dmin"][0], 16).to_bytes(2, "little")
    blk[4:16] = bytes.fromhex(kv["scales"][0])
    for c in range(4):
        for l in range(32):
            blk[16 + 32 * c + l] = (l % 16) | (((l + c) % 16) << 4)
    return np.frombuffer(bytes(blk), dtype=np.uint8), kv, ats, rng


def test_q4_k_hand_superblock(golden_dir):
    W, kv, ats, rng = _q4_k_fixture(golden_dir)
    sc, mn = oracle.q4_k_scale_min(W[4:16])
    assert list(sc) == [int(v) for v in kv["sc"]]
    assert list(mn) == [int(v) for v in kv["m"]]
    y = oracle.decode_q4_k(W, 1, 256)[0]
    for i, v in ats:
        assert y[i] == np.float32(v), (i, y[i], v)
    lo, hi, v = rng
    assert np.all(y[lo:hi] == np.float32(v))
    assert math.fsum(float(x) for x in y) == float(kv["sum"][0])


@pytest.mark.parametrize("name,decode,zeros", [
    ("q4_1_block.txt", oracle.decode_q4_1, [2, 29]),
    ("q5_0_block.txt", oracle.decode_q5_0, [0, 31]),
    ("q5_1_block.txt", oracle.decode_q5_1, [19]),
])
def test_32_value_hand_blocks(golden_dir, name, decode, zeros):
    rows = dict((r[0], r[1:]) for r in _read(golden_dir, name))
    W = np.frombuffer(bytes.fromhex(rows["hex"][0]), dtype=np.uint8)
    want = np.array([float(v) for v in rows["values"]], dtype=np.float32)
    got = decode(W, 1, 32)[0]
    assert _bits_equal(got, want)      # bitwise, signed zeros included
    for i in zeros:
        assert got[i] == 0.0 and np.signbit(got[i]) == np.signbit(want[i])


def _q5_k_fixture(golden_dir):
    rows = _read(golden_dir, "q5_k_superblock.txt")
    kv, ats, rng = {}, [], None
    for r in rows:
        if r[0] == "at":
            ats.append((int(r[1]), float(r[2])))
        elif r[0] == "range":
            rng = (int(r[1]), int(r[2]), float(r[3]))
        else:
            kv[r[0]] = r[1:]
    blk = bytearray(176)
    blk[0:2] = int(kv["d"][0], 16).to_bytes(2, "little")
    blk[2:4] = int(kv["dmin"][0], 16).to_bytes(2, "little")
    blk[4:16] = bytes.fromhex(kv["scales"][0])
    for l in range(32):
        blk[16 + l] = 0x55 if l % 2 == 0 else 0xAA
    for c in range(4):
        for l in range(32):
            blk[48 + 32 * c + l] = (l % 16) | (((l + c) % 16) << 4)
    return np.frombuffer(bytes(blk), dtype=np.uint8), kv, ats, rng


def test_q5_k_hand_superblock(golden_dir):
    W, kv, ats, rng = _q5_k_fixture(golden_dir)
    y = oracle.decode_q5_k(W, 1, 256)[0]
    for i, v in ats:
        assert y[i] == np.float32(v), (i, y[i], v)
    lo, hi, v = rng
    assert np.all(y[lo:hi] == np.float32(v))
    assert math.fsum(float(x) for x in y) == float(kv["sum"][0])


def _q6_k_fixture(golden_dir):
    rows = _read(golden_dir, "q6_k_superblock.txt")
    kv, ats, subs = {}, [], []
    for r in rows:
        if r[0] == "at":
            ats.append((int(r[1]), float(r[2])))
        elif r[0] == "subsum":
            subs.append((int(r[1]), int(r[2]), float(r[3])))
        else:
            kv[r[0]] = r[1:]
    blk = bytearray(210)
    for x in range(128):
        blk[x] = (x % 16) | (((x + 3) % 16) << 4)
    for x in range(64):
        blk[128 + x] = sum(((x + i) % 4) << (2 * i) for i in range(4))
    blk[192:208] = bytes.fromhex(kv["scales"][0])
    blk[208:210] = int(kv["d"][0], 16).to_bytes(2, "little")
    return np.frombuffer(bytes(blk), dtype=np.uint8), kv, ats, subs


def test_q6_k_hand_superblock(golden_dir):
    W, kv, ats, subs = _q6_k_fixture(golden_dir)
    y = oracle.decode_q6_k(W, 1, 256)[0]
    for i, v in ats:
        assert y[i] == np.float32(v), (i, y[i], v)
    for lo, hi, v in subs:
        assert math.fsum(float(x) for x in y[lo:hi]) == v


def _k_fixture(golden_dir, name, build):
    rows = _read(golden_dir, name)
    kv, ats, subs = {}, [], []
    for r in rows:
        if r[0] == "at":
            ats.append((int(r[1]), float(r[2])))
        elif r[0] == "subsum":
            subs.append((int(r[1]), int(r[2]), float(r[3])))
        else:
            kv[r[0]] = r[1:]
    return np.frombuffer(bytes(build(kv)), dtype=np.uint8), ats, subs


def _q2_k_bytes(kv):
    blk = bytearray(84)
    for b in range(16):
        blk[b] = ((b % 15) + 1) | ((b % 4) << 4)
    for x in range(64):
        blk[16 + x] = sum(((x + j) % 4) << (2 * j) for j in range(4))
    blk[80:82] = int(kv["d"][0], 16).to_bytes(2, "little")
    blk[82:84] = int(kv["dmin"][0], 16).to_bytes(2, "little")
    return blk


def _q3_k_bytes(kv):
    blk = bytearray(110)
    for x in range(32):
        blk[x] = 0x0F if x < 16 else 0x33
    for x in range(64):
        blk[32 + x] = sum(((x + j) % 4) << (2 * j) for j in range(4))
    blk[96:108] = bytes.fromhex(kv["scales"][0])
    blk[108:110] = int(kv["d"][0], 16).to_bytes(2, "little")
    return blk


@pytest.mark.parametrize("name,build,decode", [
    ("q2_k_superblock.txt", _q2_k_bytes, qop.decode_q2_k),
    ("q3_k_superblock.txt", _q3_k_bytes, qop.decode_q3_k)])
def test_q2_q3_k_hand_superblocks(golden_dir, name, build, decode):
    W, ats, subs = _k_fixture(golden_dir, name, build)
    y = decode(W, 1, 256)[0]
    for i, v in ats:
        assert y[i] == np.float32(v), (i, y[i], v)
    for lo, hi, v in subs:
        assert math.fsum(float(x) for x in y[lo:hi]) == v


def _mxfp4_fixture(golden_dir):
    rows = _read(golden_dir, "mxfp4_blocks.txt")
    out = []
    for i in range(0, len(rows), 2):
        assert rows[i][0] == "hex" and rows[i + 1][0] == "values"
        W = np.frombuffer(bytes.fromhex(rows[i][1]), dtype=np.uint8)
        out.append((W, np.array([float(v) for v in rows[i + 1][1:]], dtype=np.float32)))
    return out


def _same_values(got, want):
    """Bitwise equal, except that any NaN matches a NaN."""
    nan = np.isnan(want)
    return np.array_equal(np.isnan(got), nan) and _bits_equal(got[~nan], want[~nan])


def test_mxfp4_hand_blocks(golden_dir):
    """Scales 1, 4, 2^-7, 2^-127 (a float32 subnormal) and NaN; every E2M1
    code in both nibble halves, signed zeros included."""
    blocks = _mxfp4_fixture(golden_dir)
    assert len(blocks) == 5
    for W, want in blocks:
        assert _same_values(oracle.decode_mxfp4(W, 1, 32)[0], want)
    W = np.concatenate([w for w, _ in blocks])          # five blocks in one row
    assert _same_values(oracle.decode_mxfp4(W, 1, 160)[0], np.concatenate([v for _, v in blocks]))


def _nvfp4_fixture(golden_dir):
    rows = _read(golden_dir, "nvfp4_blocks.txt")
    out = []
    for i in range(0, len(rows), 2):
        assert rows[i][0] == "hex" and rows[i + 1][0] == "values"
        W = np.frombuffer(bytes.fromhex(rows[i][1]), dtype=np.uint8)
        out.append((W, np.array([float(v) for v in rows[i + 1][1:]], dtype=np.float32)))
    return out


def test_nvfp4_hand_blocks(golden_dir):
    """Scales 1, 2, 0.5, +0, the smallest and largest subnormal, the smallest
    normal, 240, 448, -1, -0.0 and NaN; every E2M1 code in both nibble
    halves of a micro-block, signed zeros included."""
    blocks = _nvfp4_fixture(golden_dir)
    assert len(blocks) == 3
    for W, want in blocks:
        assert _same_values(oracle.decode_nvfp4(W, 1, 64)[0], want)
    W = np.concatenate([w for w, _ in blocks] + [blocks[0][0]])   # four blocks: a 256-value row
    want = np.concatenate([v for _, v in blocks] + [blocks[0][1]])
    assert _same_values(oracle.decode_nvfp4(W, 1, 256)[0], want)
    assert _same_values(oracle.dequant(oracle.NVFP4, np.concatenate([W, W]), 2, 256),
                        np.stack([want, want]))


def test_e4m3_codes_against_torch_float8():
    """All 256 E4M3 bytes against torch's float8_e4m3fn (the same OCP
    format: no infinities, NaN at 0x7f and 0xff)."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch has no float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert _same_values(oracle.e4m3_to_f32(codes), want)


def test_e4m3_codes_against_ldexp():
    """E4M3 from math.ldexp: normals (1 + m/8) * 2^(e-7), subnormals
    m * 2^-9, the sign, 0x7f / 0xff NaN."""
    got = oracle.e4m3_to_f32(np.arange(256))
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(got[c])
            continue
        mag = math.ldexp(m, -9) if e == 0 else math.ldexp(8 + m, e - 10)
        want = struct.unpack("<f", struct.pack("<f", -mag if s else mag))[0]
        assert got[c] == want and math.copysign(1.0, float(got[c])) == (-1.0 if s else 1.0), c
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_nvfp4_pack_roundtrip_through_oracle():
    """The generator's packer places every scale and code where the
    oracle reads it: y[16s + j] = E2M1(q[16s + j]) * E4M3(d[s])."""
    rng = np.random.default_rng(8)
    nb = 5
    d = rng.integers(0, 0x7F, (nb, 4))
    q = rng.integers(0, 16, (nb, 64))
    W = inputs.pack_nvfp4(d, q).reshape(-1)
    y = oracle.decode_nvfp4(W, 1, 64 * nb).reshape(nb, 64)
    sub = np.arange(64) // 16
    want = (oracle.e2m1_to_f32(q).astype(np.float64) *
            oracle.e4m3_to_f32(d)[:, sub].astype(np.float64)).astype(np.float32)
    assert _same_values(y, want)


def test_e2m1_codes_against_the_element_table():
    """The OCP FP4 (E2M1) element table: codes 0..7 are 0, 0.5, 1, 1.5, 2,
    3, 4, 6 and codes 8..15 their negatives (code 8 is -0.0)."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    want = np.array(table + [-v for v in table], dtype=np.float32)
    assert _bits_equal(oracle.e2m1_to_f32(np.arange(16)), want)


def test_e8m0_scales_against_ldexp():
    """E8M0: 2^(e - 127), e = 0 the float32 subnormal 2^-127, e = 255 NaN;
    checked against math.ldexp packed by struct."""
    got = oracle.e8m0_to_f32(np.arange(256))
    for e in range(255):
        want = struct.unpack("<f", struct.pack("<f", math.ldexp(1.0, e - 127)))[0]
        assert got[e] == want and got[e] > 0, e
    assert np.isnan(got[255])


def test_q3_k_scales_unpack_every_field():
    """Each 6-bit scale set alone to 63 (others 0) lights exactly its own
    output: the low nibble and the two high bits come from the bytes the
    definition names."""
    for i in range(16):
        S = np.zeros(12, np.uint8)
        if i < 8:
            S[i] |= 15
        else:
            S[i - 8] |= 15 << 4
        S[8 + i % 4] |= 3 << (2 * (i // 4))
        sc = oracle.q3_k_scales(S) + 32
        assert sc[i] == 63 and np.count_nonzero(sc) == 1, (i, sc)


def test_half_codes_hand_decoded(golden_dir):
    for kind, code, val in _read(golden_dir, "half_codes.txt"):
        bits = np.array([int(code, 16)], dtype=np.uint16)
        fn = oracle.f16_bits_to_f32 if kind == "f16" else oracle.bf16_bits_to_f32
        got = fn(bits)[0]
        assert _bits_equal(got, np.float32(float(val))), (kind, code, got, val)


def test_f32_codes_hand_decoded(golden_dir):
    for kind, code, val in _read(golden_dir, "f32_codes.txt"):
        W = np.frombuffer(int(code, 16).to_bytes(4, "little"), dtype=np.uint8)
        got = oracle.decode_f32(W, 1, 1)[0, 0]
        assert _bits_equal(got, np.float32(float(val))), (code, got, val)
        # Python's own binary32 codec, independent of numpy
        assert float(got) == struct.unpack("<f", int(code, 16).to_bytes(4, "little"))[0]


def test_f16_all_codes_against_numpy_and_struct():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_f32(codes)
    ref = codes.view(np.float16).astype(np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    # Python's own binary16 codec, independent of numpy
    for c in (0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x8001, 0xFBFF, 0xC000, 0x1234):
        py = struct.unpack("<e", struct.pack("<H", c))[0]
        assert float(oracle.f16_bits_to_f32(np.array([c], dtype=np.uint16))[0]) == py


def test_bf16_all_codes_against_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_bits_to_f32(codes)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# ----------------------------------------------------------------------------
# closed forms of the contraction

def _all_ones_weight(wtype, N, K, variant=0):
    """Every decoded value is 1.0 (variant 1 of Q4_K goes through the min term)."""
    if wtype == inputs.Q8_0:
        blk = bytes([0x00, 0x3C]) + bytes([1]) * 32
        return np.frombuffer(blk * (N * K // 32), dtype=np.uint8)
    if wtype == inputs.Q4_0:
        blk = bytes([0x00, 0x3C]) + bytes([0x99]) * 16        # nibble 9 -> 9-8 = 1
        return np.frombuffer(blk * (N * K // 32), dtype=np.uint8)
    if wtype == inputs.Q4_K:
        if variant == 0:   # d = 1, sc = 1, q = 1, dmin = 0
            S = bytes([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1])
            blk = bytes([0x00, 0x3C, 0x00, 0x00]) + S + bytes([0x11]) * 128
        else:              # d = 1, sc = 1, q = 2, dmin = 1, m = 1: 2 - 1 = 1
            S = bytes([1, 1, 1, 1, 1, 1, 1, 1, 0x11, 0x11, 0x11, 0x11])
            blk = bytes([0x00, 0x3C, 0x00, 0x3C]) + S + bytes([0x22]) * 128
        return np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    if wtype == inputs.Q4_1:     # d = 1, m = 0, nibble 1
        blk = bytes([0x00, 0x3C, 0x00, 0x00]) + bytes([0x11]) * 16
        return np.frombuffer(blk * (N * K // 32), dtype=np.uint8)
    if wtype == inputs.Q5_0:     # d = 1, q = 17 (nibble 1, fifth bit set): 17 - 16 = 1
        blk = bytes([0x00, 0x3C]) + bytes([0xFF]) * 4 + bytes([0x11]) * 16
        return np.frombuffer(blk * (N * K // 32), dtype=np.uint8)
    if wtype == inputs.Q5_1:
        if variant == 0:         # d = 1, m = 0, q = 1
            blk = bytes([0x00, 0x3C, 0x00, 0x00]) + bytes(4) + bytes([0x11]) * 16
        else:                    # d = 0.5, m = -7, q = 16 (fifth bit only): 8 - 7 = 1
            blk = bytes([0x00, 0x38, 0x00, 0xC7]) + bytes([0xFF]) * 4 + bytes(16)
        return np.frombuffer(blk * (N * K // 32), dtype=np.uint8)
    if wtype == inputs.Q5_K:
        if variant == 0:         # d = 1, sc = 1, q = 1 (nibble only), dmin = 0
            S = bytes([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1])
            blk = bytes([0x00, 0x3C, 0x00, 0x00]) + S + bytes(32) + bytes([0x11]) * 128
        else:                    # d = 1, sc = 1, q = 17 (fifth bit), dmin = 1, m = 16: 17 - 16
            # m = 16 = 0b010000: sub-blocks 0..3 keep it in S[4..7] & 63; 4..7 take
            # their low nibble (0) from S[8..11] >> 4 and their top bits (01) from S[4..7] >> 6
            S = bytes([1, 1, 1, 1, 0x50, 0x50, 0x50, 0x50, 0x01, 0x01, 0x01, 0x01])
            blk = bytes([0x00, 0x3C, 0x00, 0x3C]) + S + bytes([0xFF]) * 32 + bytes([0x11]) * 128
        return np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    if wtype == inputs.Q6_K:
        # q = 33 = 0b10_0001: nibbles 1 (ql bytes 0x11), high pairs 2 (qh bytes
        # 0xaa); d * sc * (33 - 32) = 1 with (d, sc) = (1, 1) or (0.5, 2)
        d, sc = (bytes([0x00, 0x3C]), 1) if variant == 0 else (bytes([0x00, 0x38]), 2)
        blk = bytes([0x11]) * 128 + bytes([0xAA]) * 64 + bytes([sc]) * 16 + d
        return np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    if wtype == inputs.Q2_K:
        if variant == 0:         # d = 1, sc = 1, m = 0, q = 1 (every 2-bit field 01)
            blk = bytes([0x01]) * 16 + bytes([0x55]) * 64 + bytes([0x00, 0x3C, 0x00, 0x00])
        else:                    # d = 1, sc = 1, q = 3, dmin = 1, m = 2: 3 - 2 = 1
            blk = bytes([0x21]) * 16 + bytes([0xFF]) * 64 + bytes([0x00, 0x3C, 0x00, 0x3C])
        return np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    if wtype == inputs.Q3_K:
        if variant == 0:         # d = 1, scale 33 - 32 = 1 (low 1, high 2), q = 1 (bit set)
            S = bytes([0x11]) * 8 + bytes([0xAA]) * 4
            blk = bytes([0xFF]) * 32 + bytes([0x55]) * 64 + S + bytes([0x00, 0x3C])
        else:                    # d = 1, scale 31 - 32 = -1 (low 15, high 1), q = 3 - 4 = -1
            S = bytes([0xFF]) * 8 + bytes([0x55]) * 4
            blk = bytes(32) + bytes([0xFF]) * 64 + S + bytes([0x00, 0x3C])
        return np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    if wtype == inputs.MXFP4:    # scale 2^0, E2M1 code 2 (1.0) in both nibbles
        blk = bytes([0x7F]) + bytes([0x22]) * 16
        return np.frombuffer(blk * (N * K // 32), dtype=np.uint8)
    if wtype == inputs.NVFP4:    # E4M3 scales 1.0 (0x38), E2M1 code 2 (1.0) in both nibbles
        blk = bytes([0x38]) * 4 + bytes([0x22]) * 32
        return np.frombuffer(blk * (N * K // 64), dtype=np.uint8)
    if wtype == inputs.F16:
        return np.frombuffer(bytes([0x00, 0x3C]) * (N * K), dtype=np.uint8)
    if wtype == inputs.F32:
        return np.frombuffer(bytes([0x00, 0x00, 0x80, 0x3F]) * (N * K), dtype=np.uint8)
    if wtype == inputs.BF16:
        return np.frombuffer(bytes([0x80, 0x3F]) * (N * K), dtype=np.uint8)
    raise ValueError(wtype)


CASES = [(inputs.Q8_0, 0), (inputs.Q4_0, 0), (inputs.Q4_K, 0), (inputs.Q4_K, 1),
         (inputs.F16, 0), (inputs.BF16, 0), (inputs.Q4_1, 0), (inputs.Q5_0, 0),
         (inputs.Q5_1, 0), (inputs.Q5_1, 1), (inputs.Q5_K, 0), (inputs.Q5_K, 1),
         (inputs.Q6_K, 0), (inputs.Q6_K, 1), (inputs.F32, 0), (inputs.Q2_K, 0),
         (inputs.Q2_K, 1), (inputs.Q3_K, 0), (inputs.Q3_K, 1), (inputs.MXFP4, 0),
         (inputs.NVFP4, 0)]


@pytest.mark.parametrize("wtype,variant", CASES)
def test_all_ones_times_one_hot(wtype, variant):
    N, K, T = 64, 256, 5
    W = _all_ones_weight(wtype, N, K, variant)
    assert np.all(oracle.dequant(wtype, W, N, K) == 1.0)
    dY = np.zeros((T, N), dtype=np.float32)
    for t in range(T):
        dY[t, (7 * t + 3) % N] = 1.0
    assert np.all(oracle.out_prod(wtype, W, N, K, dY, T) == 1.0)


@pytest.mark.parametrize("wtype", inputs.ALL_TYPES)
def test_one_hot_selects_rows(wtype):
    """One-hot dY[t] = e_{n0(t)} gives dX[t, :] = deq(W)[n0(t), :] exactly:
    the contraction runs over the rows of W, not its columns."""
    N, K, T = 48, 512, 6
    W = inputs.gen_weight(wtype, N, K, seed=5, stream=1)
    Wd = oracle.dequant(wtype, W, N, K)
    n0 = [(11 * t + 2) % N for t in range(T)]
    dY = np.zeros((T, N), dtype=np.float32)
    for t in range(T):
        dY[t, n0[t]] = 1.0
    ref = oracle.out_prod(wtype, W, N, K, dY, T)
    for t in range(T):
        assert np.array_equal(ref[t], Wd[n0[t]].astype(np.float64))


@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q5_K])
def test_k_quant_min_path_closed_form(wtype):
    """q = 0 everywhere: dX[t, k] = -sum_n dY[t, n] * dmin_n * m_{n, k // 32}."""
    N, K, T = 20, 512, 3
    pack = inputs.pack_q4_k if wtype == inputs.Q4_K else inputs.pack_q5_k
    nb = N * K // 256
    rng = np.random.default_rng(3)
    d = inputs.f32_to_f16_bits(np.abs(rng.normal(0, 1e-2, nb)).astype(np.float32))
    dmin_f = np.abs(rng.normal(0, 1e-2, nb)).astype(np.float32)
    dmin = inputs.f32_to_f16_bits(dmin_f)
    sc = rng.integers(0, 64, (nb, 8))
    m = rng.integers(0, 64, (nb, 8))
    W = pack(d, dmin, sc, m, np.zeros((nb, 256), dtype=np.int64)).reshape(-1)
    dY = rng.normal(0, 1, (T, N)).astype(np.float32)
    dmin_exact = dmin.view(np.float16).astype(np.float64).reshape(N, K // 256)
    m_r = m.reshape(N, K // 256, 8)
    want = np.zeros((T, K))
    for t in range(T):
        for k in range(K):
            b, j = divmod(k // 32, 8)
            want[t, k] = -math.fsum(float(dY[t, n]) * float(dmin_exact[n, b]) * int(m_r[n, b, j])
                                    for n in range(N))
    got = oracle.out_prod(wtype, W, N, K, dY, T)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------
# brute force: an independent pure-Python decode and exactly rounded sums

def _py_f16(b0, b1):
    return struct.unpack("<e", bytes([b0, b1]))[0]


def _py_decode(wtype, raw, N, K):
    """Per-byte decode written from the block definitions, no numpy."""
    rb = inputs.row_bytes(wtype, K)
    out = [[0.0] * K for _ in range(N)]
    for n in range(N):
        row = raw[n * rb:(n + 1) * rb]
        if wtype == inputs.F32:
            for k in range(K):
                out[n][k] = struct.unpack("<f", bytes(row[4 * k: 4 * k + 4]))[0]
        elif wtype in (inputs.F16, inputs.BF16):
            for k in range(K):
                lo, hi = row[2 * k], row[2 * k + 1]
                if wtype == inputs.F16:
                    out[n][k] = _py_f16(lo, hi)
                else:
                    out[n][k] = struct.unpack("<f", bytes([0, 0, lo, hi]))[0]
        elif wtype == inputs.Q8_0:
            for b in range(K // 32):
                blk = row[34 * b: 34 * b + 34]
                d = _py_f16(blk[0], blk[1])
                for i in range(32):
                    q = blk[2 + i] - 256 if blk[2 + i] > 127 else blk[2 + i]
                    out[n][32 * b + i] = d * q
        elif wtype == inputs.Q4_0:
            for b in range(K // 32):
                blk = row[18 * b: 18 * b + 18]
                d = _py_f16(blk[0], blk[1])
                for j in range(16):
                    out[n][32 * b + j] = d * ((blk[2 + j] & 15) - 8)
                    out[n][32 * b + 16 + j] = d * ((blk[2 + j] >> 4) - 8)
        elif wtype == inputs.Q4_K:
            for b in range(K // 256):
                blk = row[144 * b: 144 * b + 144]
                d = _py_f16(blk[0], blk[1])
                dmin = _py_f16(blk[2], blk[3])
                S = blk[4:16]
                for j in range(8):
                    if j < 4:
                        sc, m = S[j] & 63, S[j + 4] & 63
                    else:
                        sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4)
                        m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4)
                    c, half = divmod(j, 2)
                    for l in range(32):
                        byte = blk[16 + 32 * c + l]
                        q = (byte >> 4) if half else (byte & 15)
                        # F32 evaluation: both products exact, one rounding
                        v = np.float32(np.float32(d * sc) * q) - np.float32(dmin * m)
                        out[n][256 * b + 64 * c + 32 * half + l] = float(v)
        elif wtype in (inputs.Q4_1, inputs.Q5_0, inputs.Q5_1):
            bb = {inputs.Q4_1: 20, inputs.Q5_0: 22, inputs.Q5_1: 24}[wtype]
            for b in range(K // 32):
                blk = row[bb * b: bb * b + bb]
                d = _py_f16(blk[0], blk[1])
                m = _py_f16(blk[2], blk[3]) if wtype != inputs.Q5_0 else 0.0
                qh_at = {inputs.Q4_1: None, inputs.Q5_0: 2, inputs.Q5_1: 4}[wtype]
                qs_at = {inputs.Q4_1: 4, inputs.Q5_0: 6, inputs.Q5_1: 8}[wtype]
                qh = int.from_bytes(bytes(blk[qh_at:qh_at + 4]), "little") if qh_at else 0
                for i in range(32):
                    byte = blk[qs_at + (i % 16)]
                    q = (byte & 15) if i < 16 else (byte >> 4)
                    q += 16 * ((qh >> i) & 1)
                    if wtype == inputs.Q5_0:
                        out[n][32 * b + i] = d * (q - 16)
                    else:   # F32 evaluation: exact product, one rounding in the sum
                        out[n][32 * b + i] = float(np.float32(np.float32(d * q) + np.float32(m)))
        elif wtype == inputs.Q5_K:
            for b in range(K // 256):
                blk = row[176 * b: 176 * b + 176]
                d = _py_f16(blk[0], blk[1])
                dmin = _py_f16(blk[2], blk[3])
                S = blk[4:16]
                for j in range(8):
                    if j < 4:
                        sc, m = S[j] & 63, S[j + 4] & 63
                    else:
                        sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4)
                        m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4)
                    c, half = divmod(j, 2)
                    for l in range(32):
                        byte = blk[48 + 32 * c + l]
                        q = ((byte >> 4) if half else (byte & 15)) + 16 * ((blk[16 + l] >> j) & 1)
                        v = np.float32(np.float32(d * sc) * q) - np.float32(dmin * m)
                        out[n][256 * b + 64 * c + 32 * half + l] = float(v)
        elif wtype == inputs.Q6_K:
            for b in range(K // 256):
                blk = row[210 * b: 210 * b + 210]
                d = _py_f16(blk[208], blk[209])
                for v in range(256):
                    h, rest = divmod(v, 128)
                    i, l = divmod(rest, 32)
                    byte = blk[64 * h + 32 * (i % 2) + l]
                    q = ((byte >> 4) if i >= 2 else (byte & 15)) | (((blk[128 + 32 * h + l] >> (2 * i)) & 3) << 4)
                    sc = blk[192 + v // 16] - 256 if blk[192 + v // 16] > 127 else blk[192 + v // 16]
                    out[n][256 * b + v] = d * sc * (q - 32)
        elif wtype == inputs.Q2_K:
            for b in range(K // 256):
                blk = row[84 * b: 84 * b + 84]
                d, dmin = _py_f16(blk[80], blk[81]), _py_f16(blk[82], blk[83])
                for v in range(256):
                    h, rest = divmod(v, 128)
                    j, rest = divmod(rest, 32)
                    s, l = divmod(rest, 16)
                    q = (blk[16 + 32 * h + 16 * s + l] >> (2 * j)) & 3
                    sb = blk[8 * h + 2 * j + s]
                    # F32 evaluation: exact product, one rounding in the difference
                    val = np.float32(np.float32(d * (sb & 15)) * q) - np.float32(dmin * (sb >> 4))
                    out[n][256 * b + v] = float(val)
        elif wtype == inputs.MXFP4:
            e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
            for b in range(K // 32):
                blk = row[17 * b: 17 * b + 17]
                scale = 2.0 ** (blk[0] - 127) if blk[0] != 255 else float("nan")
                for j in range(32):
                    code = (blk[1 + j % 16] >> (4 * (j // 16))) & 15
                    mag = e2m1[code & 7] * scale
                    out[n][32 * b + j] = -mag if code & 8 else mag
        elif wtype == inputs.NVFP4:
            e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
            for b in range(K // 64):
                blk = row[36 * b: 36 * b + 36]
                for v in range(64):
                    s, j = divmod(v, 16)
                    code = (blk[4 + 8 * s + j % 8] >> (4 * (j // 8))) & 15
                    e8 = blk[s]
                    ex, mt = (e8 >> 3) & 15, e8 & 7
                    if ex == 15 and mt == 7:
                        scale = float("nan")
                    else:
                        scale = mt / 8 * 2.0 ** -6 if ex == 0 else (1 + mt / 8) * 2.0 ** (ex - 7)
                        scale = -scale if e8 & 0x80 else scale
                    mag = e2m1[code & 7] * scale
                    out[n][64 * b + v] = -mag if code & 8 else mag
        elif wtype == inputs.Q3_K:
            for b in range(K // 256):
                blk = row[110 * b: 110 * b + 110]
                d = _py_f16(blk[108], blk[109])
                S = blk[96:108]
                for v in range(256):
                    h, rest = divmod(v, 128)
                    j, rest = divmod(rest, 32)
                    s, l = divmod(rest, 16)
                    i = 8 * h + 2 * j + s
                    lo4 = (S[i] & 15) if i < 8 else (S[i - 8] >> 4)
                    hi2 = (S[8 + i % 4] >> (2 * (i // 4))) & 3
                    q = (blk[32 + 32 * h + 16 * s + l] >> (2 * j)) & 3
                    if not (blk[16 * s + l] >> (4 * h + j)) & 1:
                        q -= 4
                    out[n][256 * b + v] = d * ((lo4 | (hi2 << 4)) - 32) * q
    return out


BRUTE = [(inputs.Q8_0, 40, 64, 3), (inputs.Q4_0, 33, 96, 2), (inputs.Q4_K, 12, 512, 2),
         (inputs.F16, 24, 40, 3), (inputs.BF16, 24, 40, 3), (inputs.Q8_0, 7, 32, 1),
         (inputs.Q4_1, 21, 64, 2), (inputs.Q5_0, 19, 96, 2), (inputs.Q5_1, 17, 64, 2),
         (inputs.Q5_K, 10, 512, 2), (inputs.Q6_K, 9, 512, 2), (inputs.F32, 20, 48, 3),
         (inputs.Q2_K, 11, 512, 2), (inputs.Q3_K, 10, 512, 2), (inputs.MXFP4, 13, 96, 2),
         (inputs.NVFP4, 11, 256, 2)]


@pytest.mark.parametrize("wtype,N,K,T", BRUTE)
def test_brute_force(wtype, N, K, T):
    W = inputs.gen_weight(wtype, N, K, seed=11, stream=1)
    dY = inputs.normal_f32(11, 2, T * N, 1.0).reshape(T, N)
    raw = bytes(W)
    Wpy = _py_decode(wtype, raw, N, K)
    Wd = oracle.dequant(wtype, W, N, K)
    assert _bits_equal(Wd, np.array(Wpy, dtype=np.float32))
    ref = oracle.out_prod(wtype, W, N, K, dY, T)
    bnd = oracle.abs_bound(dY, Wd)
    for t in range(T):
        for k in range(K):
            exact = math.fsum(float(dY[t, n]) * Wpy[n][k] for n in range(N))
            babs = math.fsum(abs(float(dY[t, n]) * Wpy[n][k]) for n in range(N))
            assert abs(ref[t, k] - exact) <= 1e-12 * babs + 1e-300
            assert abs(bnd[t, k] - babs) <= 1e-12 * babs + 1e-300


# ----------------------------------------------------------------------------
# invariants

def test_linearity_and_beta():
    N, K, T = 96, 256, 4
    W = inputs.gen_weight(inputs.Q4_K, N, K, seed=2, stream=1)
    Wd = oracle.dequant(inputs.Q4_K, W, N, K)
    d1 = inputs.normal_f32(2, 2, T * N, 1.0).reshape(T, N)
    d2 = inputs.normal_f32(2, 3, T * N, 1.0).reshape(T, N)
    a, b = np.float32(0.5), np.float32(-2.0)   # powers of two keep a*d1 + b*d2 exact-ish
    lhs = oracle.out_prod(inputs.Q4_K, W, N, K, (a * d1 + b * d2).astype(np.float32), T)
    rhs = float(a) * oracle.out_prod(inputs.Q4_K, W, N, K, d1, T) + \
        float(b) * oracle.out_prod(inputs.Q4_K, W, N, K, d2, T)
    B = oracle.abs_bound(np.abs(a * d1) + np.abs(b * d2), Wd)
    assert np.all(np.abs(lhs - rhs) <= 1e-6 * B + 1e-12)
    dX0 = inputs.normal_f32(2, 4, T * K, 1.0).reshape(T, K)
    beta = 0.75
    with_beta = oracle.out_prod(inputs.Q4_K, W, N, K, d1, T, dX0, beta)
    base = oracle.out_prod(inputs.Q4_K, W, N, K, d1, T)
    assert np.allclose(with_beta, base + beta * dX0.astype(np.float64), rtol=1e-15, atol=0)
    # beta = 0 never reads dX0, even when it is NaN
    nan0 = np.full((T, K), np.nan, dtype=np.float32)
    assert np.array_equal(oracle.out_prod(inputs.Q4_K, W, N, K, d1, T, nan0, 0.0), base)


def test_mul_mat_at_matches_full():
    """The sampled forward against the full one (itself pinned by one-hot
    rows, the adjoint identity and brute force) and the pinned bound; the
    operands swapped (deq(W) rows against X's columns) must not pass."""
    N, K, T = 40, 512, 9
    W = inputs.gen_weight(inputs.Q4_K, N, K, seed=10, stream=1)
    X = inputs.normal_f32(10, 2, T * K, 1.0).reshape(T, K)
    Y0 = inputs.normal_f32(10, 3, T * N, 1.0).reshape(T, N)
    Wd = oracle.dequant(inputs.Q4_K, W, N, K)
    full = oracle.mul_mat(inputs.Q4_K, W, N, K, X, T, Y0, 0.5, Wd=Wd)
    bnd = oracle.mul_mat_bound(X, Wd)
    ts = np.array([0, 8, 3, 3, 5])
    ns = np.array([0, 39, 17, 18, 1])
    ref, b = oracle.mul_mat_at(Wd, X, ts, ns, Y0, 0.5)
    assert np.allclose(ref, full[ts, ns], rtol=1e-13, atol=1e-15)
    assert np.allclose(b, bnd[ts, ns], rtol=1e-13)
    bad, _ = oracle.mul_mat_at(Wd, X, ns % T, ts % N, Y0, 0.5)
    assert not np.allclose(bad, full[ts, ns], rtol=1e-6)


def test_out_prod_at_matches_full():
    N, K, T = 64, 256, 7
    W = inputs.gen_weight(inputs.Q8_0, N, K, seed=9, stream=1)
    dY = inputs.normal_f32(9, 2, T * N, 1.0).reshape(T, N)
    dX0 = inputs.normal_f32(9, 3, T * K, 1.0).reshape(T, K)
    Wd = oracle.dequant(inputs.Q8_0, W, N, K)
    full = oracle.out_prod(inputs.Q8_0, W, N, K, dY, T, dX0, 1.0)
    bnd = oracle.abs_bound(dY, Wd)
    ts = np.array([0, 3, 6, 6, 1])
    ks = np.array([0, 255, 17, 128, 64])
    ref, b = oracle.out_prod_at(Wd, dY, ts, ks, dX0, 1.0)
    assert np.allclose(ref, full[ts, ks], rtol=1e-13, atol=1e-15)
    assert np.allclose(b, bnd[ts, ks], rtol=1e-13)


def test_sizes():
    # the dense F32 copy of a 5120 x 17408 weight: the "356 MB" of the PR's
    # memory note (llama.cpp fork PR "cuda: out_prod accepts a quantized src0", "What")
    assert 5120 * 17408 * 4 == 356_515_840
    # stored row bytes from the block sizes: 34 B / 32, 18 B / 32, 144 B / 256, 2 B / value
    assert oracle.row_bytes(oracle.Q8_0, 256) == 272
    assert oracle.row_bytes(oracle.Q4_0, 4096) == 2304
    assert oracle.row_bytes(oracle.Q4_K, 4096) == 2304
    assert oracle.row_bytes(oracle.F16, 17408) == 34816
    assert oracle.row_bytes(oracle.Q8_0, 14336) == 15232
    assert 256 * 272 == 69_632 and 4096 * 2304 == 9_437_184
    assert 14336 * 2304 == 33_030_144 and 5120 * 34816 == 178_257_920
    assert oracle.row_bytes(oracle.Q4_K, 300) == 0 and oracle.row_bytes(oracle.Q8_0, 48) == 0
    # 20 B / 32, 22 B / 32, 24 B / 32, 176 B / 256
    assert oracle.row_bytes(oracle.Q4_1, 4096) == 2560 and oracle.row_bytes(oracle.Q5_0, 4096) == 2816
    assert oracle.row_bytes(oracle.Q5_1, 4096) == 3072 and oracle.row_bytes(oracle.Q5_K, 4096) == 2816
    assert oracle.row_bytes(oracle.Q6_K, 4096) == 3360     # 210 B / 256


def test_q4_k_pack_roundtrip_through_oracle():
    rng = np.random.default_rng(0)
    nb = 50
    sc = rng.integers(0, 64, (nb, 8))
    m = rng.integers(0, 64, (nb, 8))
    blk = inputs.pack_q4_k(np.zeros(nb, np.uint16), np.zeros(nb, np.uint16), sc, m,
                           rng.integers(0, 16, (nb, 256)))
    sc2, m2 = oracle.q4_k_scale_min(blk[:, 4:16])
    assert np.array_equal(sc, sc2) and np.array_equal(m, m2)


# ----------------------------------------------------------------------------
# planted mistakes: each mutant of an oracle step must fail one of the pins

def _mut_q4_0_swapped_nibbles(W, N, K):
    blk = qop._rows(W, N, K, qop.Q4_0).reshape(N, K // 32, 18)
    d = qop.f16_bits_to_f32(qop._le16(blk[..., 0], blk[..., 1]))
    qs = blk[..., 2:18]
    nib = np.concatenate([qs >> 4, qs & 0x0F], axis=-1).astype(np.float32)
    return (d[..., None] * (nib - 8)).reshape(N, K)


def _mut_q4_0_select_zero(W, N, K):
    y = qop.decode_q4_0(W, N, K)
    return np.where(y == 0, np.float32(0.0), y)   # drops the sign of zero


def _mut_q4_k_wrong_high_bits(W, N, K):
    real = qop.q4_k_scale_min

    def bad(S):
        sc, mn = real(S)
        S = np.asarray(S, dtype=np.int64)
        for j in range(4, 8):
            sc[..., j] = (S[..., j + 4] & 15) | ((S[..., j] >> 6) << 4)   # j instead of j-4
        return sc, mn
    qop.q4_k_scale_min = bad
    try:
        return qop.decode_q4_k(W, N, K)
    finally:
        qop.q4_k_scale_min = real


def _mut_q5_0_high_bits_from_low_half(W, N, K):
    """Values j + 16 take bit j of qh instead of bit j + 16."""
    blk = qop._rows(W, N, K, qop.Q5_0).reshape(N, K // 32, 22)
    d = qop.f16_bits_to_f32(qop._le16(blk[..., 0], blk[..., 1]))
    bits = qop._fifth_bits_32(blk[..., 2:6])
    bits = np.concatenate([bits[..., :16], bits[..., :16]], axis=-1)
    q = qop._nibbles_32(blk[..., 6:22]) + 16 * bits
    return (d[..., None] * (q - 16).astype(np.float32)).reshape(N, K)


def _mut_q5_1_min_subtracted(W, N, K):
    blk = qop._rows(W, N, K, qop.Q5_1).reshape(N, K // 32, 24)
    d = qop.f16_bits_to_f32(qop._le16(blk[..., 0], blk[..., 1]))
    m = qop.f16_bits_to_f32(qop._le16(blk[..., 2], blk[..., 3]))
    q = qop._nibbles_32(blk[..., 8:24]) + 16 * qop._fifth_bits_32(blk[..., 4:8])
    return (d[..., None] * q.astype(np.float32) - m[..., None]).reshape(N, K)


def _mut_q5_k_swapped_qh_bits(W, N, K):
    """The low-nibble half takes bit 2c+1 and the high half bit 2c."""
    blk = np.array(qop._rows(W, N, K, qop.Q5_K).reshape(N, K // 256, 176))
    qh = blk[..., 16:48].astype(np.int64)
    swapped = ((qh & 0x55) << 1) | ((qh & 0xAA) >> 1)
    blk[..., 16:48] = swapped.astype(np.uint8)
    return qop.decode_q5_k(blk.reshape(-1), N, K)


def _mut_q6_k_pairs_by_parity(W, N, K):
    """High bits from bits 2*(i % 2) instead of 2i (a plausible index slip)."""
    blk = np.array(qop._rows(W, N, K, qop.Q6_K).reshape(N, K // 256, 210))
    qh = blk[..., 128:192].astype(np.int64)
    pair = lambda x, i: (x >> (2 * i)) & 3  # noqa: E731
    fixed = pair(qh, 0) | (pair(qh, 1) << 2) | (pair(qh, 0) << 4) | (pair(qh, 1) << 6)
    blk[..., 128:192] = fixed.astype(np.uint8)
    return qop.decode_q6_k(blk.reshape(-1), N, K)


def _mut_q2_k_scale_min_swapped(W, N, K):
    """The high nibble taken as the scale and the low as the min."""
    blk = np.array(qop._rows(W, N, K, qop.Q2_K).reshape(N, K // 256, 84))
    sb = blk[..., 0:16]
    blk[..., 0:16] = ((sb >> 4) | (sb << 4)).astype(np.uint8)
    return qop.decode_q2_k(blk.reshape(-1), N, K)


def _mut_q3_k_hmask_bit_j(W, N, K):
    """The third bit read from bit j of hmask for both halves (not 4h + j)."""
    blk = np.array(qop._rows(W, N, K, qop.Q3_K).reshape(N, K // 256, 110))
    hm = blk[..., 0:32].astype(np.int64)
    blk[..., 0:32] = ((hm & 0x0F) | ((hm & 0x0F) << 4)).astype(np.uint8)
    return qop.decode_q3_k(blk.reshape(-1), N, K)


def _mut_q3_k_unbiased_scale(W, N, K):
    """The 6-bit scale used without subtracting 32."""
    return qop.decode_q3_k(W, N, K) * 0 + _q3_k_plus32(W, N, K)


def _q3_k_plus32(W, N, K):
    real = qop.q3_k_scales
    qop.q3_k_scales = lambda S: real(S) + 32
    try:
        return qop.decode_q3_k(W, N, K)
    finally:
        qop.q3_k_scales = real


def test_q2_q3_k_mutants_are_caught(golden_dir):
    for name, build, mutants in [
            ("q2_k_superblock.txt", _q2_k_bytes, [_mut_q2_k_scale_min_swapped]),
            ("q3_k_superblock.txt", _q3_k_bytes, [_mut_q3_k_hmask_bit_j, _mut_q3_k_unbiased_scale])]:
        W, ats, subs = _k_fixture(golden_dir, name, build)
        for mut in mutants:
            y = mut(W, 1, 256)[0]
            assert any(y[i] != np.float32(v) for i, v in ats), (name, mut.__name__)


def test_q6_k_mutant_is_caught(golden_dir):
    W, kv, ats, subs = _q6_k_fixture(golden_dir)
    y = _mut_q6_k_pairs_by_parity(W, 1, 256)[0]
    assert any(y[i] != np.float32(v) for i, v in ats)


def _mut_mxfp4_bias_128(W, N, K):
    """The scale as 2^(e - 128)."""
    blk = qop._rows(W, N, K, qop.MXFP4).reshape(N, K // 32, 17)
    sc = np.ldexp(1.0, blk[..., 0].astype(np.int64) - 128)
    nib = np.concatenate([blk[..., 1:17] & 0x0F, blk[..., 1:17] >> 4], axis=-1)
    return (sc[..., None] * qop.e2m1_to_f32(nib)).astype(np.float32).reshape(N, K)


def _mut_mxfp4_no_subnormal_elements(W, N, K):
    """E2M1 exponent 0 read as a normal number (code 1 -> 0.75)."""
    real = qop.e2m1_to_f32

    def bad(code):
        c = np.asarray(code).astype(np.int64)
        e, m = (c >> 1) & 3, (c & 1).astype(np.float64)
        mag = np.where((c & 7) == 0, 0.0, np.ldexp(1.0 + m / 2.0, e - 1))
        return np.where((c >> 3) & 1 == 1, -mag, mag).astype(np.float32)
    qop.e2m1_to_f32 = bad
    try:
        return qop.decode_mxfp4(W, N, K)
    finally:
        qop.e2m1_to_f32 = real


def _mut_mxfp4_swapped_nibbles(W, N, K):
    blk = qop._rows(W, N, K, qop.MXFP4).reshape(N, K // 32, 17)
    sc = qop.e8m0_to_f32(blk[..., 0]).astype(np.float64)
    nib = np.concatenate([blk[..., 1:17] >> 4, blk[..., 1:17] & 0x0F], axis=-1)
    return (sc[..., None] * qop.e2m1_to_f32(nib)).astype(np.float32).reshape(N, K)


def test_mxfp4_mutants_are_caught(golden_dir):
    W, want = _mxfp4_fixture(golden_dir)[0]
    for mut in (_mut_mxfp4_bias_128, _mut_mxfp4_no_subnormal_elements, _mut_mxfp4_swapped_nibbles):
        assert not _same_values(mut(W, 1, 32)[0], want), mut.__name__


def _mut_nvfp4_q4_0_nibble_order(W, N, K):
    """Nibbles ordered over the whole 64-value block (low = j, high = j + 32)."""
    blk = qop._rows(W, N, K, qop.NVFP4).reshape(N, K // 64, 36)
    sc = qop.e4m3_to_f32(blk[..., 0:4]).astype(np.float64)
    qs = blk[..., 4:36]
    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)              # [.., 64]
    y = sc[..., np.arange(64) // 16] * qop.e2m1_to_f32(nib).astype(np.float64)
    return y.astype(np.float32).reshape(N, K)


def _mut_nvfp4_scale_bias_8(W, N, K):
    """E4M3 scales decoded with exponent bias 8."""
    blk = qop._rows(W, N, K, qop.NVFP4).reshape(N, K // 64, 36)
    sc = qop.e4m3_to_f32(blk[..., 0:4]).astype(np.float64) / 2.0
    qs = blk[..., 4:36].reshape(N, K // 64, 4, 8)
    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)
    return (sc[..., None] * qop.e2m1_to_f32(nib)).astype(np.float32).reshape(N, K)


def _mut_nvfp4_normal_subnormals(W, N, K):
    """E4M3 exponent 0 read as a normal binade, (1 + m/8) * 2^-7."""
    real = qop.e4m3_to_f32

    def bad(code):
        c = np.asarray(code).astype(np.int64)
        e, m = (c >> 3) & 15, (c & 7).astype(np.float64)
        mag = np.ldexp(1.0 + m / 8.0, e - 7)
        mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
        return np.where((c >> 7) & 1 == 1, -mag, mag).astype(np.float32)
    qop.e4m3_to_f32 = bad
    try:
        return qop.decode_nvfp4(W, N, K)
    finally:
        qop.e4m3_to_f32 = real


def _mut_nvfp4_scale_per_32(W, N, K):
    """One scale per 32 values (d[0], d[1] over the block's halves)."""
    blk = qop._rows(W, N, K, qop.NVFP4).reshape(N, K // 64, 36)
    sc = qop.e4m3_to_f32(blk[..., 0:4]).astype(np.float64)
    qs = blk[..., 4:36].reshape(N, K // 64, 4, 8)
    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=-1).reshape(N, K // 64, 64)
    y = sc[..., np.arange(64) // 32] * qop.e2m1_to_f32(nib).astype(np.float64)
    return y.astype(np.float32).reshape(N, K)


def test_nvfp4_mutants_are_caught(golden_dir):
    blocks = _nvfp4_fixture(golden_dir)
    for mut in (_mut_nvfp4_q4_0_nibble_order, _mut_nvfp4_scale_bias_8,
                _mut_nvfp4_normal_subnormals, _mut_nvfp4_scale_per_32):
        assert any(not _same_values(mut(W, 1, 64)[0], want) for W, want in blocks), mut.__name__


def test_new_type_mutants_are_caught(golden_dir):
    rows = dict((r[0], r[1:]) for r in _read(golden_dir, "q5_0_block.txt"))
    W = np.frombuffer(bytes.fromhex(rows["hex"][0]), dtype=np.uint8)
    want = np.array([float(v) for v in rows["values"]], dtype=np.float32)
    assert not _bits_equal(_mut_q5_0_high_bits_from_low_half(W, 1, 32)[0], want)
    rows = dict((r[0], r[1:]) for r in _read(golden_dir, "q5_1_block.txt"))
    W = np.frombuffer(bytes.fromhex(rows["hex"][0]), dtype=np.uint8)
    want = np.array([float(v) for v in rows["values"]], dtype=np.float32)
    assert not _bits_equal(_mut_q5_1_min_subtracted(W, 1, 32)[0], want)
    Wk, kv, ats, rng = _q5_k_fixture(golden_dir)
    yk = _mut_q5_k_swapped_qh_bits(Wk, 1, 256)[0]
    assert any(yk[i] != np.float32(v) for i, v in ats)


def test_mutants_are_caught(golden_dir):
    rows = dict((r[0], r[1:]) for r in _read(golden_dir, "q4_0_block.txt"))
    W = np.frombuffer(bytes.fromhex(rows["hex"][0]), dtype=np.uint8)
    want = np.array([float(v) for v in rows["values"]], dtype=np.float32)
    assert not _bits_equal(_mut_q4_0_swapped_nibbles(W, 1, 32)[0], want)
    assert not _bits_equal(_mut_q4_0_select_zero(W, 1, 32)[0], want)
    Wk, kv, ats, rng = _q4_k_fixture(golden_dir)
    yk = _mut_q4_k_wrong_high_bits(Wk, 1, 256)[0]
    assert any(yk[i] != np.float32(v) for i, v in ats)


def test_transposed_contraction_is_caught():
    """Contracting over K (dY @ deq(W).T) instead of N breaks the one-hot pin."""
    N, K, T = 32, 32, 3
    W = inputs.gen_weight(inputs.Q8_0, N, K, seed=5, stream=1)
    Wd = oracle.dequant(inputs.Q8_0, W, N, K)
    dY = np.zeros((T, N), dtype=np.float32)
    dY[0, 4] = dY[1, 9] = dY[2, 30] = 1.0
    wrong = dY.astype(np.float64) @ Wd.T.astype(np.float64)
    assert not all(np.array_equal(wrong[t], Wd[n].astype(np.float64))
                   for t, n in enumerate([4, 9, 30]))


def test_dropped_beta_is_caught():
    N, K, T = 32, 256, 2
    W = inputs.gen_weight(inputs.Q4_K, N, K, seed=5, stream=1)
    dY = inputs.normal_f32(5, 2, T * N, 1.0).reshape(T, N)
    dX0 = inputs.normal_f32(5, 3, T * K, 1.0).reshape(T, K)
    good = oracle.out_prod(inputs.Q4_K, W, N, K, dY, T, dX0, 1.0)
    dropped = oracle.out_prod(inputs.Q4_K, W, N, K, dY, T)
    assert not np.allclose(good, dropped)


# ----------------------------------------------------------------------------
# the forward mul_mat(W, x) through the same decode

@pytest.mark.parametrize("wtype", [inputs.Q4_K, inputs.Q8_0, inputs.F16])
def test_mul_mat_one_hot_selects_columns(wtype):
    """X[t] = e_{k0(t)} gives Y[t, :] = deq(W)[:, k0(t)] exactly: the forward
    contracts over the K values of each row, not over the rows."""
    N, K, T = 40, 512, 5
    W = inputs.gen_weight(wtype, N, K, seed=81, stream=1)
    Wd = oracle.dequant(wtype, W, N, K)
    k0 = [(37 * t + 3) % K for t in range(T)]
    X = np.zeros((T, K), np.float32)
    X[np.arange(T), k0] = 1.0
    Y = oracle.mul_mat(wtype, W, N, K, X, T)
    for t in range(T):
        assert np.array_equal(Y[t], Wd[:, k0[t]].astype(np.float64))


def test_mul_mat_is_the_adjoint_of_out_prod():
    """<dY, W x> = <W^T dY, x> for the same W: the forward and the backward
    contract the same decoded matrix along opposite axes."""
    N, K, T = 48, 768, 6
    W = inputs.gen_weight(inputs.Q5_K, N, K, seed=82, stream=1)
    X = inputs.normal_f32(82, 2, T * K, 1.0).reshape(T, K)
    dY = inputs.normal_f32(82, 3, T * N, 1.0).reshape(T, N)
    Y = oracle.mul_mat(inputs.Q5_K, W, N, K, X, T)
    dX = oracle.out_prod(inputs.Q5_K, W, N, K, dY, T)
    lhs = float(np.sum(dY.astype(np.float64) * Y))
    rhs = float(np.sum(dX * X.astype(np.float64)))
    assert abs(lhs - rhs) <= 1e-9 * (abs(lhs) + 1.0)


def test_mul_mat_brute_force_and_beta():
    N, K, T = 9, 64, 3
    W = inputs.gen_weight(inputs.Q4_0, N, K, seed=83, stream=1)
    X = inputs.normal_f32(83, 2, T * K, 1.0).reshape(T, K)
    Y0 = inputs.normal_f32(83, 3, T * N, 1.0).reshape(T, N)
    Wpy = _py_decode(inputs.Q4_0, bytes(W), N, K)
    got = oracle.mul_mat(inputs.Q4_0, W, N, K, X, T, Y0, 0.5)
    for t in range(T):
        for n in range(N):
            exact = math.fsum(float(X[t, k]) * Wpy[n][k] for k in range(K)) + 0.5 * float(Y0[t, n])
            assert abs(got[t, n] - exact) <= 1e-12 * (abs(exact) + 1.0)


# ----------------------------------------------------------------------------
# the input gradient through the base weight plus a low-rank adapter

def _lora_fixture(golden_dir):
    rows = dict((r[0], r[1:]) for r in _read(golden_dir, "lora_tiny.txt"))
    N, K, T, R = (int(rows[x][0]) for x in ("N", "K", "T", "R"))
    W = np.array([int(c, 16) for c in rows["W"]], np.uint16).view(np.uint8)
    f = lambda key: np.array([float(v) for v in rows[key]], np.float32)  # noqa: E731
    return (N, K, T, R, float(rows["scale"][0]), float(rows["beta"][0]), W,
            f("dY").reshape(T, N), f("B").reshape(N, R), f("A").reshape(R, K),
            f("dX0").reshape(T, K), f("dX").reshape(T, K))


def test_lora_hand_example(golden_dir):
    N, K, T, R, s, beta, W, dY, B, A, dX0, want = _lora_fixture(golden_dir)
    got = oracle.out_prod_lora(inputs.F16, W, N, K, dY, T, A, B, R, s, dX0, beta)
    assert np.array_equal(got, want.astype(np.float64))


def test_lora_without_adapter_is_out_prod():
    """scale 0, or rank 0, leaves the base gradient bit for bit."""
    N, K, T, R = 24, 256, 3, 4
    W = inputs.gen_weight(inputs.Q4_K, N, K, seed=91, stream=1)
    dY = inputs.normal_f32(91, 2, T * N, 1.0).reshape(T, N)
    A = inputs.normal_f32(91, 3, R * K, 1.0).reshape(R, K)
    B = inputs.normal_f32(91, 4, N * R, 1.0).reshape(N, R)
    base = oracle.out_prod(inputs.Q4_K, W, N, K, dY, T)
    assert np.array_equal(oracle.out_prod_lora(inputs.Q4_K, W, N, K, dY, T, A, B, R, 0.0), base)
    assert np.array_equal(oracle.out_prod_lora(inputs.Q4_K, W, N, K, dY, T, A[:0], B[:, :0], 0, 2.0),
                          base)


def test_lora_one_hot_row_closed_form():
    """dY[t] = e_n: dX[t] = deq(W)[n] + scale * sum_j B[n, j] A[j] (the
    adapter's row n of B A), with one nonzero per sum up to the r ranks."""
    N, K, T, R = 20, 64, 4, 3
    W = inputs.gen_weight(inputs.Q8_0, N, K, seed=92, stream=1)
    Wd = oracle.dequant(inputs.Q8_0, W, N, K)
    A = inputs.normal_f32(92, 3, R * K, 1.0).reshape(R, K)
    B = inputs.normal_f32(92, 4, N * R, 1.0).reshape(N, R)
    rows = [3, 0, 19, 11]
    dY = np.zeros((T, N), np.float32)
    dY[np.arange(T), rows] = 1.0
    got = oracle.out_prod_lora(inputs.Q8_0, W, N, K, dY, T, A, B, R, 0.75)
    for t, n in enumerate(rows):
        want = [float(Wd[n, k]) + 0.75 * math.fsum(float(B[n, j]) * float(A[j, k]) for j in range(R))
                for k in range(K)]
        assert np.allclose(got[t], want, rtol=1e-15, atol=1e-15)


def test_lora_brute_force():
    """Pure-Python sums with exact rounding over both contractions."""
    N, K, T, R = 7, 32, 3, 5
    W = inputs.gen_weight(inputs.Q4_0, N, K, seed=93, stream=1)
    Wpy = _py_decode(inputs.Q4_0, bytes(W), N, K)
    dY = inputs.normal_f32(93, 2, T * N, 1.0).reshape(T, N)
    A = inputs.normal_f32(93, 3, R * K, 1.0).reshape(R, K)
    B = inputs.normal_f32(93, 4, N * R, 1.0).reshape(N, R)
    dX0 = inputs.normal_f32(93, 5, T * K, 1.0).reshape(T, K)
    got = oracle.out_prod_lora(inputs.Q4_0, W, N, K, dY, T, A, B, R, -1.5, dX0, 0.25)
    for t in range(T):
        U = [math.fsum(float(dY[t, n]) * float(B[n, j]) for n in range(N)) for j in range(R)]
        for k in range(K):
            exact = (math.fsum(float(dY[t, n]) * Wpy[n][k] for n in range(N))
                     - 1.5 * math.fsum(U[j] * float(A[j, k]) for j in range(R))
                     + 0.25 * float(dX0[t, k]))
            assert abs(got[t, k] - exact) <= 1e-12 * (abs(exact) + 1.0)


def test_lora_is_the_adjoint_of_the_adapted_forward():
    """<dY, y(x)> = <dX(dY), x> for y = x deq(W)^T + scale (x A^T) B^T: the
    backward contracts the adapter's matrices along the opposite axes."""
    N, K, T, R = 40, 512, 6, 8
    W = inputs.gen_weight(inputs.Q5_K, N, K, seed=94, stream=1)
    X = inputs.normal_f32(94, 2, T * K, 1.0).reshape(T, K).astype(np.float64)
    dY = inputs.normal_f32(94, 3, T * N, 1.0).reshape(T, N)
    A = inputs.normal_f32(94, 4, R * K, 1.0).reshape(R, K)
    B = inputs.normal_f32(94, 5, N * R, 1.0).reshape(N, R)
    Y = oracle.mul_mat(inputs.Q5_K, W, N, K, X.astype(np.float32), T)
    for t in range(T):   # the adapter's forward, written out on its own
        for n in range(N):
            Y[t, n] += 0.5 * sum(float(B[n, j]) * float(np.dot(X[t], A[j].astype(np.float64)))
                                 for j in range(R))
    dX = oracle.out_prod_lora(inputs.Q5_K, W, N, K, dY, T, A, B, R, 0.5)
    lhs = float(np.sum(dY.astype(np.float64) * Y))
    rhs = float(np.sum(dX * X))
    assert abs(lhs - rhs) <= 1e-9 * (abs(lhs) + 1.0)


def test_lora_bound_covers_terms():
    N, K, T, R = 16, 64, 2, 3
    dY = inputs.normal_f32(95, 2, T * N, 1.0).reshape(T, N)
    A = inputs.normal_f32(95, 3, R * K, 1.0).reshape(R, K)
    B = inputs.normal_f32(95, 4, N * R, 1.0).reshape(N, R)
    bnd = oracle.lora_bound(dY, A, B, -2.0)
    for t in range(T):
        for k in range(K):
            terms = [abs(2.0 * float(dY[t, n]) * float(B[n, j]) * float(A[j, k]))
                     for n in range(N) for j in range(R)]
            assert abs(bnd[t, k] - math.fsum(terms)) <= 1e-12 * bnd[t, k]


def _mul_mat_bound_matches_terms(bound_fn) -> bool:
    """Whether bound_fn(X, Wd)[t, n] equals the exact sum of the absolute
    terms |X[t, k] * deq(W)[n, k]| over the K values of row n (the forward's
    contraction), written out one term at a time; signed inputs, so a dropped
    absolute value shows, and N != K, so a transposed operand shows."""
    N, K, T = 7, 256, 3
    W = inputs.gen_weight(inputs.Q8_0, N, K, seed=97, stream=1)
    Wd = oracle.dequant(inputs.Q8_0, W, N, K)
    X = inputs.normal_f32(97, 2, T * K, 1.0).reshape(T, K)
    try:
        bnd = np.asarray(bound_fn(X, Wd), dtype=np.float64)
    except ValueError:  # mismatched shapes
        return False
    if bnd.shape != (T, N):
        return False
    for t in range(T):
        for n in range(N):
            exact = math.fsum(abs(float(X[t, k]) * float(Wd[n, k])) for k in range(K))
            if not abs(bnd[t, n] - exact) <= 1e-12 * exact:
                return False
    return True


def test_mul_mat_bound_covers_terms():
    assert _mul_mat_bound_matches_terms(oracle.mul_mat_bound)


@pytest.mark.parametrize("mutant", ["no_abs_x", "no_abs_w", "signed", "w_not_transposed_sq"])
def test_mul_mat_bound_mutants_are_caught(mutant):
    """Plausible mistakes in a copy of the forward bound fail the term check."""
    def fn(X, Wd):
        X64, W64 = np.asarray(X, dtype=np.float64), np.asarray(Wd, dtype=np.float64)
        if mutant == "no_abs_x":
            return X64 @ np.abs(W64).T
        if mutant == "no_abs_w":
            return np.abs(X64) @ W64.T
        if mutant == "signed":
            return np.abs(X64 @ W64.T)
        return np.abs(X64) @ np.abs(W64)   # the backward's orientation: shapes do not fit
    assert not _mul_mat_bound_matches_terms(fn)


@pytest.mark.parametrize("mutant", ["b_transposed_role", "dropped_scale", "a_rows_reversed",
                                    "u_from_base"])
def test_lora_mutants_are_caught(golden_dir, mutant):
    """Plausible mistakes in a copy of the adapter term fail the hand example."""
    N, K, T, R, s, beta, W, dY, B, A, dX0, want = _lora_fixture(golden_dir)
    base = oracle.out_prod(inputs.F16, W, N, K, dY, T, dX0, beta)
    dY64, A64, B64 = dY.astype(np.float64), A.astype(np.float64), B.astype(np.float64)
    if mutant == "b_transposed_role":
        term = s * ((dY64 @ B64.T) @ A64)          # square fixture: shapes still fit
    elif mutant == "dropped_scale":
        term = (dY64 @ B64) @ A64
    elif mutant == "a_rows_reversed":
        term = s * ((dY64 @ B64) @ A64[::-1])
    else:
        Wd = oracle.dequant(inputs.F16, W, N, K).astype(np.float64)
        term = s * (((dY64 @ Wd) @ B64) @ A64)
    assert not np.array_equal(base + term, want.astype(np.float64))


def test_lora_at_matches_full():
    N, K, T, R = 30, 64, 5, 6
    W = inputs.gen_weight(inputs.F16, N, K, seed=96, stream=1)
    dY = inputs.normal_f32(96, 2, T * N, 1.0).reshape(T, N)
    A = inputs.normal_f32(96, 3, R * K, 1.0).reshape(R, K)
    B = inputs.normal_f32(96, 4, N * R, 1.0).reshape(N, R)
    full = (oracle.out_prod_lora(inputs.F16, W, N, K, dY, T, A, B, R, 1.25)
            - oracle.out_prod(inputs.F16, W, N, K, dY, T))
    bnd = oracle.lora_bound(dY, A, B, 1.25)
    ts, ks = [0, 4, 2, 3], [63, 0, 17, 40]
    v, b = oracle.lora_at(dY, A, B, 1.25, ts, ks)
    assert np.allclose(v, full[ts, ks], rtol=1e-12, atol=1e-12)
    assert np.allclose(b, bnd[ts, ks], rtol=1e-12)


def test_q2_q3_k_pack_roundtrip_through_oracle():
    """The generators' packers place every field where the oracle reads it."""
    rng = np.random.default_rng(7)
    B = 3
    d = rng.integers(0x3000, 0x3c00, B).astype(np.uint16)
    dmin = rng.integers(0x2c00, 0x3800, B).astype(np.uint16)
    sc = rng.integers(0, 16, (B, 16))
    m = rng.integers(0, 16, (B, 16))
    q = rng.integers(0, 4, (B, 256))
    W = inputs.pack_q2_k(d, dmin, sc, m, q).reshape(-1)
    y = oracle.decode_q2_k(W, B, 256)
    df, mf = qop.f16_bits_to_f32(d), qop.f16_bits_to_f32(dmin)
    sub = np.array([8 * (v // 128) + 2 * ((v % 128) // 32) + (v % 32) // 16 for v in range(256)])
    want = (df[:, None] * sc[:, sub].astype(np.float32)) * q.astype(np.float32) \
        - mf[:, None] * m[:, sub].astype(np.float32)
    assert _bits_equal(y, want.astype(np.float32))
    sc6 = rng.integers(0, 64, (B, 16))
    q3 = rng.integers(-4, 4, (B, 256))
    W = inputs.pack_q3_k(d, sc6, q3).reshape(-1)
    y = oracle.decode_q3_k(W, B, 256)
    want = (df[:, None] * (sc6[:, sub] - 32).astype(np.float32)) * q3.astype(np.float32)
    assert _bits_equal(y, want.astype(np.float32))


# ----------------------------------------------------------------------------
# batched OUT_PROD: which weight a batch reads

def test_batch_weight_hand_table():
    """Eight gradient batches over two weights: the first four read weight 0,
    the next four weight 1 (a run of consecutive batches per weight, as a
    grouped k/v projection shares one weight among neighbouring heads); the
    second dimension the same way, independently."""
    assert [oracle.batch_weight(i, 0, 8, 1, 2, 1)[0] for i in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.batch_weight(i, 0, 6, 1, 3, 1)[0] for i in range(6)] == [0, 0, 1, 1, 2, 2]
    assert [oracle.batch_weight(0, i, 1, 4, 1, 4)[1] for i in range(4)] == [0, 1, 2, 3]
    assert [oracle.batch_weight(2, i, 4, 6, 2, 2) for i in range(6)] == \
        [(1, 0), (1, 0), (1, 0), (1, 1), (1, 1), (1, 1)]
    with pytest.raises(ValueError):
        oracle.batch_weight(0, 0, 6, 1, 4, 1)


def test_batched_out_prod_picks_weights_by_value():
    """Closed form: weight (j2, j3) is the constant c = 1 + j2 + 4 j3 (F16),
    dY is one-hot, so every output of batch (i2, i3) equals the constant of
    the weight that batch reads."""
    N, K, T = 16, 32, 3
    n2, n3, w_n2, w_n3 = 4, 2, 2, 1
    consts = [[1.0 + j2 + 4 * j3 for j2 in range(w_n2)] for j3 in range(w_n3)]
    Ws = [[np.frombuffer(inputs.f32_to_f16_bits(np.full(N * K, c, np.float32)).tobytes(),
                         dtype=np.uint8) for c in row] for row in consts]
    dY = np.zeros((T, N), np.float32)
    dY[np.arange(T), [3, 7, 11]] = 1.0
    out = oracle.out_prod_batched(inputs.F16, Ws, N, K, [[dY] * n2 for _ in range(n3)], T)
    want = {(0, 0): 1.0, (1, 0): 1.0, (2, 0): 2.0, (3, 0): 2.0,
            (0, 1): 1.0, (1, 1): 1.0, (2, 1): 2.0, (3, 1): 2.0}
    for (i2, i3), c in want.items():
        assert np.all(out[i3][i2] == c), (i2, i3)


def test_batch_weight_mutant_is_caught():
    """Interleaving the weights (i % w_n, the other plausible reading) fails
    the hand table."""
    def interleaved(i2, i3, n2, n3, w_n2, w_n3):
        return i2 % w_n2, i3 % w_n3
    assert [interleaved(i, 0, 8, 1, 2, 1)[0] for i in range(8)] != [0, 0, 0, 0, 1, 1, 1, 1]
