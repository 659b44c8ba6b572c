"""Plain, slow, CPU oracle of the activation-gradient OUT_PROD through a
resident quantized / half-precision weight.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's CPU
baseline call this.  It shares no code with the CUDA library.

What it computes
----------------
The llama.cpp fork's PR "cuda: out_prod accepts a quantized src0" (commit
message and section "What") states that the backward of ``mul_mat(W, x)``
with respect to ``x`` is ``out_prod(W, grad^T)``, and that the CPU backend's
``out_prod_q_f32`` (every quantized ``src0``) is the oracle its CUDA route is
compared against.  The pages print no index formula; the plainest reading,
with ``W`` holding N rows (output features) of K values (input features) and
the incoming gradient ``dY`` of shape [T, N], is

    dX[t, k] = beta * dX0[t, k] + sum_n dY[t, n] * deq(W)[n, k]

i.e. ``dX = dY @ deq(W)``.  ``beta`` follows BLAS: 0 means dX0 is not read.

Steps (in this order, nothing fused or reordered):
1. decode every stored row of W to F32 per its format definition; fp16 fields
   are widened exactly (subnormals included), then the format's formula is
   evaluated in F32;
2. contract in F64: every F32 x F32 product is exact in F64;
3. the acceptance bound  B[t, k] = sum_n |dY[t, n]| * |deq(W)[n, k]|  (F64).

Block formats (little-endian), ggml's GGUF block types:
* Q8_0  34 B / 32: fp16 d, int8 qs[32];          y_i = d * qs_i
* Q4_0  18 B / 32: fp16 d, qs[16] (lo nibble = value j, hi = value j+16);
                                                  y = d * (nib - 8)
* Q4_K 144 B / 256: fp16 d, fp16 dmin, 12 B of 6-bit (sc, m) x 8, qs[128];
                                                  y = (d*sc)*q - dmin*m
* Q4_1  20 B / 32: fp16 d, fp16 m, qs[16] (nibbles as Q4_0); y = d * nib + m
* Q5_0  22 B / 32: fp16 d, qh (32-bit LE: bit i = fifth bit of value i),
                   qs[16] (nibbles as Q4_0);      y = d * (q - 16)
* Q5_1  24 B / 32: fp16 d, fp16 m, qh, qs[16];     y = d * q + m
* Q5_K 176 B / 256: fp16 d, fp16 dmin, 12 B (sc, m) as Q4_K, qh[32], qs[128]:
                   the nibbles of Q4_K plus bit 2c (low) / 2c+1 (high) of
                   qh[l] as the fifth bit;        y = (d*sc)*q - dmin*m
* Q6_K 210 B / 256: ql[128], qh[64], int8 scales[16], fp16 d.  Value
                   128h + 32i + l (h = 0..1, i = 0..3, l = 0..31) takes the
                   low (i < 2) or high (i >= 2) nibble of ql[64h + 32(i%2) + l]
                   and bits 2i..2i+1 of qh[32h + l] as bits 4..5;
                                                  y = (d*sc[v/16]) * (q - 32)
* Q2_K  84 B / 256: scales[16] (lo nibble sc, hi nibble m), qs[64], fp16 d,
                   fp16 dmin.  Value 128h + 32j + 16s + l takes bits 2j..2j+1
                   of qs[32h + 16s + l], byte 8h + 2j + s of scales;
                                                  y = (d*sc)*q - dmin*m
* Q3_K 110 B / 256: hmask[32], qs[64], 12 B of sixteen 6-bit scales, fp16 d.
                   Value 128h + 32j + 16s + l: q = bits 2j..2j+1 of
                   qs[32h + 16s + l], minus 4 unless bit 4h + j of
                   hmask[16s + l] is set;         y = (d*(sc - 32)) * q
* MXFP4 17 B / 32: E8M0 scale byte e, qs[16] (nibbles as Q4_0), each an
                   E2M1 code (sign bit 3, two exponent bits, one mantissa
                   bit; the OCP microscaling formats);
                                                  y = E2M1(nib) * 2^(e - 127)
* NVFP4 36 B / 64: d[4] (one FP8 E4M3 scale per 16-value micro-block),
                   qs[32]; micro-block s holds values 16s .. 16s+15: value
                   16s + j (j < 8) is the low nibble of qs[8s + j], value
                   16s + j + 8 its high nibble; each nibble an E2M1 element
                   as in MXFP4;                   y = E2M1(nib) * E4M3(d[s])
* F16 / BF16: 2 B per value.
* F32: 4 B per value, the value itself.

The adapter variant (out_prod_lora) adds scale * (dY @ B) @ A for a
low-rank adapter A [r, K], B [N, r] beside the resident W; see its docstring.

Parity pins for each function live in tests/test_oracle.py.
"""
from __future__ import annotations

import numpy as np

F16, BF16, Q8_0, Q4_0, Q4_K = 1, 2, 3, 4, 5
Q4_1, Q5_0, Q5_1, Q5_K, Q6_K = 6, 7, 8, 9, 10
F32, Q2_K, Q3_K, MXFP4, NVFP4 = 11, 12, 13, 14, 15

_BLOCK = {F16: (1, 2), BF16: (1, 2), Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144),
          Q4_1: (32, 20), Q5_0: (32, 22), Q5_1: (32, 24), Q5_K: (256, 176),
          Q6_K: (256, 210), F32: (1, 4), Q2_K: (256, 84), Q3_K: (256, 110),
          MXFP4: (32, 17), NVFP4: (64, 36)}


def row_bytes(wtype: int, K: int) -> int:
    """Stored bytes of one row of K values, or 0 if K does not fit the type."""
    if wtype not in _BLOCK or K <= 0:
        return 0
    bs, bb = _BLOCK[wtype]
    if K % bs:
        return 0
    return (K // bs) * bb


# ----------------------------------------------------------------------------
# scalar field decoders

def f16_bits_to_f32(bits) -> np.ndarray:
    """IEEE 754 binary16 -> float32, from the definition:
    exponent 0 -> (-1)^s * 2^-14 * m/1024 (subnormal),
    exponent 31 -> inf (m == 0) or NaN,
    else        -> (-1)^s * 2^(e-15) * (1 + m/1024).
    Every binary16 value is exactly representable in float32."""
    h = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = (h >> 15) & 1
    e = (h >> 10) & 0x1F
    m = h & 0x3FF
    sub = np.ldexp(m.astype(np.float64), -24)                 # m * 2^-24
    nrm = np.ldexp((m + 1024).astype(np.float64), e - 25)    # (1024+m) * 2^(e-25)
    mag = np.where(e == 0, sub, nrm)
    mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    return np.where(s == 1, -mag, mag).astype(np.float32)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bfloat16 -> float32: the 16 bits are the top half of the float32 word."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def e8m0_to_f32(e) -> np.ndarray:
    """OCP MX E8M0 shared scale: 2^(e - 127) for e < 255 (e = 0 gives
    2^-127, a float32 subnormal), NaN for e = 255."""
    e = np.asarray(e).astype(np.int64)
    v = np.ldexp(np.ones(e.shape), e - 127)
    return np.where(e == 255, np.nan, v).astype(np.float32)


def e2m1_to_f32(code) -> np.ndarray:
    """OCP FP4 E2M1 element: bit 3 sign, bits 1-2 exponent (bias 1), bit 0
    mantissa; exponent 0 -> (-1)^s * m / 2 (subnormal, signed zero kept),
    else (-1)^s * 2^(e - 1) * (1 + m / 2)."""
    c = np.asarray(code).astype(np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m / 2.0, np.ldexp(1.0 + m / 2.0, e - 1))
    return np.where(s == 1, -mag, mag).astype(np.float32)


def e4m3_to_f32(code) -> np.ndarray:
    """FP8 E4M3 (the OCP 8-bit floating-point format with four exponent and
    three mantissa bits; NVFP4's micro-block scale): bit 7 sign, bits 3-6
    exponent (bias 7), bits 0-2 mantissa; exponent 0 -> (-1)^s * 2^-6 * m/8
    (subnormal, signed zero kept); exponent 15 with mantissa 7 -> NaN (the
    format has no infinities); else (-1)^s * 2^(e - 7) * (1 + m/8), up to 448."""
    c = np.asarray(code).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag).astype(np.float32)


def _le16(lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    return lo.astype(np.uint16) | (hi.astype(np.uint16) << np.uint16(8))


# ----------------------------------------------------------------------------
# format decoders: stored bytes -> F32 [N, K]

def _rows(W, N, K, wtype):
    rb = row_bytes(wtype, K)
    if rb == 0:
        raise ValueError(f"K={K} does not fit type {wtype}")
    W = np.asarray(W, dtype=np.uint8).reshape(-1)
    if W.size != N * rb:
        raise ValueError(f"expected {N * rb} bytes, got {W.size}")
    return W.reshape(N, rb)


def decode_q8_0(W, N: int, K: int) -> np.ndarray:
    """Q8_0: y[i] = F32(d) * qs[i], exact in F32 (11-bit x 8-bit product)."""
    blk = _rows(W, N, K, Q8_0).reshape(N, K // 32, 34)
    d = f16_bits_to_f32(_le16(blk[..., 0], blk[..., 1]))
    qs = blk[..., 2:34].view(np.int8).astype(np.float32)
    return (d[..., None] * qs).reshape(N, K)


def decode_q4_0(W, N: int, K: int) -> np.ndarray:
    """Q4_0: value j (< 16) = low nibble of qs[j], value j+16 = high nibble;
    y = F32(d) * (nib - 8), exact in F32."""
    blk = _rows(W, N, K, Q4_0).reshape(N, K // 32, 18)
    d = f16_bits_to_f32(_le16(blk[..., 0], blk[..., 1]))
    qs = blk[..., 2:18]
    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=-1).astype(np.float32)
    return (d[..., None] * (nib - np.float32(8.0))).reshape(N, K)


def q4_k_scale_min(S: np.ndarray):
    """The eight 6-bit (scale, min) pairs of a Q4_K super-block from its 12
    packed bytes S[..., 0:12].  Sub-blocks 0..3 use the low 6 bits of S[j]
    (scale) and S[j+4] (min); sub-blocks 4..7 take their low 4 bits from the
    two nibbles of S[j+4] (j >= 4) and their high 2 bits from the top 2 bits
    of S[j-4] (scale) and S[j] (min)."""
    S = np.asarray(S, dtype=np.uint8).astype(np.int64)
    sc = np.empty(S.shape[:-1] + (8,), dtype=np.int64)
    mn = np.empty_like(sc)
    for j in range(8):
        if j < 4:
            sc[..., j] = S[..., j] & 63
            mn[..., j] = S[..., j + 4] & 63
        else:
            sc[..., j] = (S[..., j + 4] & 15) | ((S[..., j - 4] >> 6) << 4)
            mn[..., j] = (S[..., j + 4] >> 4) | ((S[..., j] >> 6) << 4)
    return sc, mn


def decode_q4_k(W, N: int, K: int) -> np.ndarray:
    """Q4_K: 256 values in 8 sub-blocks of 32.  For chunk c = 0..3 and
    l = 0..31, value 64c+l is the low nibble of qs[32c+l] (sub-block 2c) and
    value 64c+32+l the high nibble (sub-block 2c+1).
    y = (F32(d) * sc) * q - F32(dmin) * m: both products exact in F32, one
    rounding in the subtraction."""
    blk = _rows(W, N, K, Q4_K).reshape(N, K // 256, 144)
    d = f16_bits_to_f32(_le16(blk[..., 0], blk[..., 1]))
    dmin = f16_bits_to_f32(_le16(blk[..., 2], blk[..., 3]))
    sc, mn = q4_k_scale_min(blk[..., 4:16])
    qs = blk[..., 16:144]
    q = np.empty(blk.shape[:-1] + (256,), dtype=np.float32)
    sub = np.empty(256, dtype=np.int64)
    for c in range(4):
        q[..., 64 * c: 64 * c + 32] = qs[..., 32 * c: 32 * c + 32] & 0x0F
        q[..., 64 * c + 32: 64 * c + 64] = qs[..., 32 * c: 32 * c + 32] >> 4
        sub[64 * c: 64 * c + 32] = 2 * c
        sub[64 * c + 32: 64 * c + 64] = 2 * c + 1
    dsc = d[..., None] * sc.astype(np.float32)       # [N, nb, 8], exact
    dmm = dmin[..., None] * mn.astype(np.float32)    # [N, nb, 8], exact
    y = dsc[..., sub] * q - dmm[..., sub]
    return y.astype(np.float32).reshape(N, K)


def _nibbles_32(qs: np.ndarray) -> np.ndarray:
    """The 32 nibbles of a 32-value block's qs[16]: value j < 16 is the low
    nibble of qs[j], value j + 16 the high nibble (int64)."""
    qs = qs.astype(np.int64)
    return np.concatenate([qs & 0x0F, qs >> 4], axis=-1)


def _fifth_bits_32(qh4: np.ndarray) -> np.ndarray:
    """Bit i (i = 0..31) of the little-endian 32-bit word in qh4[..., 0:4]:
    the fifth bit of value i of a Q5_0 / Q5_1 block (int64)."""
    qh4 = qh4.astype(np.int64)
    word = qh4[..., 0] | (qh4[..., 1] << 8) | (qh4[..., 2] << 16) | (qh4[..., 3] << 24)
    return (word[..., None] >> np.arange(32, dtype=np.int64)) & 1


def decode_q4_1(W, N: int, K: int) -> np.ndarray:
    """Q4_1: y = F32(d) * nib + F32(m); the product is exact (11-bit x 4-bit),
    the sum rounds once."""
    blk = _rows(W, N, K, Q4_1).reshape(N, K // 32, 20)
    d = f16_bits_to_f32(_le16(blk[..., 0], blk[..., 1]))
    m = f16_bits_to_f32(_le16(blk[..., 2], blk[..., 3]))
    nib = _nibbles_32(blk[..., 4:20]).astype(np.float32)
    return (d[..., None] * nib + m[..., None]).reshape(N, K)


def decode_q5_0(W, N: int, K: int) -> np.ndarray:
    """Q5_0: q = nibble + 16 * (bit i of qh) for value i; y = F32(d) * (q - 16),
    exact (11-bit x 5-bit)."""
    blk = _rows(W, N, K, Q5_0).reshape(N, K // 32, 22)
    d = f16_bits_to_f32(_le16(blk[..., 0], blk[..., 1]))
    q = _nibbles_32(blk[..., 6:22]) + 16 * _fifth_bits_32(blk[..., 2:6])
    return (d[..., None] * (q - 16).astype(np.float32)).reshape(N, K)


def decode_q5_1(W, N: int, K: int) -> np.ndarray:
    """Q5_1: q = nibble + 16 * (bit i of qh); y = F32(d) * q + F32(m), the
    product exact, the sum rounded once."""
    blk = _rows(W, N, K, Q5_1).reshape(N, K // 32, 24)
    d = f16_bits_to_f32(_le16(blk[..., 0], blk[..., 1]))
    m = f16_bits_to_f32(_le16(blk[..., 2], blk[..., 3]))
    q = _nibbles_32(blk[..., 8:24]) + 16 * _fifth_bits_32(blk[..., 4:8])
    return (d[..., None] * q.astype(np.float32) + m[..., None]).reshape(N, K)


def decode_q5_k(W, N: int, K: int) -> np.ndarray:
    """Q5_K: the Q4_K layout plus qh[32].  For chunk c = 0..3 and l = 0..31,
    value 64c+l is the low nibble of qs[32c+l] plus 16 * bit 2c of qh[l]
    (sub-block 2c) and value 64c+32+l the high nibble plus 16 * bit 2c+1 of
    qh[l] (sub-block 2c+1).  y = (F32(d) * sc) * q - F32(dmin) * m: both
    products exact (at most 22 bits), one rounding in the subtraction."""
    blk = _rows(W, N, K, Q5_K).reshape(N, K // 256, 176)
    d = f16_bits_to_f32(_le16(blk[..., 0], blk[..., 1]))
    dmin = f16_bits_to_f32(_le16(blk[..., 2], blk[..., 3]))
    sc, mn = q4_k_scale_min(blk[..., 4:16])
    qh = blk[..., 16:48].astype(np.int64)
    qs = blk[..., 48:176].astype(np.int64)
    q = np.empty(blk.shape[:-1] + (256,), dtype=np.float32)
    sub = np.empty(256, dtype=np.int64)
    for c in range(4):
        ql = qs[..., 32 * c: 32 * c + 32]
        q[..., 64 * c: 64 * c + 32] = (ql & 0x0F) + 16 * ((qh >> (2 * c)) & 1)
        q[..., 64 * c + 32: 64 * c + 64] = (ql >> 4) + 16 * ((qh >> (2 * c + 1)) & 1)
        sub[64 * c: 64 * c + 32] = 2 * c
        sub[64 * c + 32: 64 * c + 64] = 2 * c + 1
    dsc = d[..., None] * sc.astype(np.float32)       # exact
    dmm = dmin[..., None] * mn.astype(np.float32)    # exact
    y = dsc[..., sub] * q - dmm[..., sub]
    return y.astype(np.float32).reshape(N, K)


def decode_q6_k(W, N: int, K: int) -> np.ndarray:
    """Q6_K: value v = 128h + 32i + l (h = 0..1, i = 0..3, l = 0..31):
    q = nibble | (bits 2i..2i+1 of qh[32h + l]) << 4, the nibble being the low
    (i = 0, 1) or high (i = 2, 3) half of ql[64h + 32(i % 2) + l];
    y = (F32(d) * sc[v // 16]) * (q - 32).  Both products are exact: 11 + 7 +
    5 significant bits."""
    blk = _rows(W, N, K, Q6_K).reshape(N, K // 256, 210)
    ql = blk[..., 0:128].astype(np.int64)
    qh = blk[..., 128:192].astype(np.int64)
    sc = blk[..., 192:208].view(np.int8).astype(np.float32)
    d = f16_bits_to_f32(_le16(blk[..., 208], blk[..., 209]))
    q = np.empty(blk.shape[:-1] + (256,), dtype=np.float32)
    for h in range(2):
        for i in range(4):
            src = ql[..., 64 * h + 32 * (i % 2): 64 * h + 32 * (i % 2) + 32]
            nib = (src >> 4) if i >= 2 else (src & 0x0F)
            hb = (qh[..., 32 * h: 32 * h + 32] >> (2 * i)) & 3
            q[..., 128 * h + 32 * i: 128 * h + 32 * i + 32] = (nib | (hb << 4)) - 32
    scale = d[..., None] * sc                      # [N, nb, 16], exact
    y = np.repeat(scale, 16, axis=-1) * q          # exact
    return y.astype(np.float32).reshape(N, K)


def decode_q2_k(W, N: int, K: int) -> np.ndarray:
    """Q2_K: value v = 128h + 32j + 16s + l (h, s = 0..1, j = 0..3,
    l = 0..15): q = bits 2j..2j+1 of qs[32h + 16s + l]; its sub-block of 16
    takes scales byte 8h + 2j + s, low nibble sc, high nibble m;
    y = (F32(d) * sc) * q - F32(dmin) * m.  d * sc * q is exact (11 + 4 + 2
    bits), the subtraction rounds once."""
    blk = _rows(W, N, K, Q2_K).reshape(N, K // 256, 84)
    sb = blk[..., 0:16].astype(np.int64)
    qs = blk[..., 16:80].astype(np.int64)
    d = f16_bits_to_f32(_le16(blk[..., 80], blk[..., 81]))
    dmin = f16_bits_to_f32(_le16(blk[..., 82], blk[..., 83]))
    q = np.empty(blk.shape[:-1] + (256,), dtype=np.float32)
    sub = np.empty(256, dtype=np.int64)   # the scales byte of each value
    for h in range(2):
        for j in range(4):
            for s in range(2):
                v0 = 128 * h + 32 * j + 16 * s
                q[..., v0: v0 + 16] = (qs[..., 32 * h + 16 * s: 32 * h + 16 * s + 16] >> (2 * j)) & 3
                sub[v0: v0 + 16] = 8 * h + 2 * j + s
    dsc = d[..., None] * (sb & 0x0F).astype(np.float32)    # exact
    dmm = dmin[..., None] * (sb >> 4).astype(np.float32)   # exact
    y = dsc[..., sub] * q - dmm[..., sub]
    return y.astype(np.float32).reshape(N, K)


def q3_k_scales(S: np.ndarray) -> np.ndarray:
    """The sixteen 6-bit scales of a Q3_K super-block from its 12 bytes S
    (last axis): scale i has low 4 bits from S[i] (i < 8, low nibble) or
    S[i - 8] (high nibble), and high 2 bits from bits 2(i // 4).. of
    S[8 + i % 4]; the value used is the 6-bit number minus 32."""
    S = np.asarray(S).astype(np.int64)
    out = np.empty(S.shape[:-1] + (16,), dtype=np.int64)
    for i in range(16):
        lo = (S[..., i] & 0x0F) if i < 8 else (S[..., i - 8] >> 4)
        hi = (S[..., 8 + i % 4] >> (2 * (i // 4))) & 3
        out[..., i] = (lo | (hi << 4)) - 32
    return out


def decode_q3_k(W, N: int, K: int) -> np.ndarray:
    """Q3_K: value v = 128h + 32j + 16s + l: q = (bits 2j..2j+1 of
    qs[32h + 16s + l]) - (0 if bit 4h + j of hmask[16s + l] is set else 4);
    y = (F32(d) * sc) * q with sc the sub-block's scale (byte index
    8h + 2j + s).  Both products are exact (11 + 6 + 3 bits)."""
    blk = _rows(W, N, K, Q3_K).reshape(N, K // 256, 110)
    hm = blk[..., 0:32].astype(np.int64)
    qs = blk[..., 32:96].astype(np.int64)
    sc = q3_k_scales(blk[..., 96:108]).astype(np.float32)
    d = f16_bits_to_f32(_le16(blk[..., 108], blk[..., 109]))
    q = np.empty(blk.shape[:-1] + (256,), dtype=np.float32)
    sub = np.empty(256, dtype=np.int64)
    for h in range(2):
        for j in range(4):
            for s in range(2):
                v0 = 128 * h + 32 * j + 16 * s
                low = (qs[..., 32 * h + 16 * s: 32 * h + 16 * s + 16] >> (2 * j)) & 3
                high = (hm[..., 16 * s: 16 * s + 16] >> (4 * h + j)) & 1
                q[..., v0: v0 + 16] = low - 4 * (1 - high)
                sub[v0: v0 + 16] = 8 * h + 2 * j + s
    dsc = d[..., None] * sc          # exact
    y = dsc[..., sub] * q            # exact
    return y.astype(np.float32).reshape(N, K)


def decode_mxfp4(W, N: int, K: int) -> np.ndarray:
    """MXFP4: value j (< 16) = low nibble of qs[j], value j+16 = high
    nibble; y = E2M1(nib) * 2^(e - 127).  Exact in F32: a two-bit significand
    times a power of two, the smallest magnitude 2^-128 a float32 subnormal
    (the largest, 6 * 2^127, overflows to inf; e = 255 gives NaN)."""
    blk = _rows(W, N, K, MXFP4).reshape(N, K // 32, 17)
    sc = e8m0_to_f32(blk[..., 0]).astype(np.float64)
    qs = blk[..., 1:17]
    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)
    with np.errstate(over="ignore", invalid="ignore"):
        y = sc[..., None] * e2m1_to_f32(nib).astype(np.float64)
        return y.astype(np.float32).reshape(N, K)


def decode_nvfp4(W, N: int, K: int) -> np.ndarray:
    """NVFP4: 36-byte blocks of 64 values, four micro-blocks of 16 with an
    E4M3 scale each (bytes 0-3), then qs[32]: micro-block s takes qs[8s ..
    8s+7], value 16s + j (j < 8) the low nibble of qs[8s + j] and value
    16s + j + 8 its high nibble; y = E2M1(nib) * E4M3(d[s]).  Exact in F32:
    a two-bit significand times a four-bit one, magnitudes 2^-10 .. 2688
    (a NaN scale gives NaN values)."""
    blk = _rows(W, N, K, NVFP4).reshape(N, K // 64, 36)
    sc = e4m3_to_f32(blk[..., 0:4]).astype(np.float64)            # [N, B, 4]
    qs = blk[..., 4:36].reshape(N, K // 64, 4, 8)                  # [N, B, s, j]
    nib = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)            # [N, B, s, 16]
    with np.errstate(invalid="ignore"):
        y = sc[..., None] * e2m1_to_f32(nib).astype(np.float64)
        return y.astype(np.float32).reshape(N, K)


def decode_f16(W, N: int, K: int) -> np.ndarray:
    b = _rows(W, N, K, F16).reshape(N, K, 2)
    return f16_bits_to_f32(_le16(b[..., 0], b[..., 1]))


def decode_f32(W, N: int, K: int) -> np.ndarray:
    """F32: the stored little-endian binary32 words."""
    return _rows(W, N, K, F32).reshape(-1).view("<f4").astype(np.float32).reshape(N, K)


def decode_bf16(W, N: int, K: int) -> np.ndarray:
    b = _rows(W, N, K, BF16).reshape(N, K, 2)
    return bf16_bits_to_f32(_le16(b[..., 0], b[..., 1]))


_DECODERS = {F16: decode_f16, BF16: decode_bf16, Q8_0: decode_q8_0,
             Q4_0: decode_q4_0, Q4_K: decode_q4_k, Q4_1: decode_q4_1,
             Q5_0: decode_q5_0, Q5_1: decode_q5_1, Q5_K: decode_q5_k,
             Q6_K: decode_q6_k, F32: decode_f32, Q2_K: decode_q2_k, Q3_K: decode_q3_k,
             MXFP4: decode_mxfp4, NVFP4: decode_nvfp4}


def dequant(wtype: int, W, N: int, K: int) -> np.ndarray:
    """deq(W) as F32 [N, K] (the value rg_dequant must reproduce bit for bit)."""
    if wtype not in _DECODERS:
        raise ValueError(f"unknown weight type {wtype}")
    return _DECODERS[wtype](W, N, K)


# ----------------------------------------------------------------------------
# the contraction

def out_prod(wtype: int, W, N: int, K: int, dY, T: int, dX0=None, beta: float = 0.0,
             Wd=None) -> np.ndarray:
    """F64 [T, K]: beta*dX0 + dY @ deq(W), contracted over the N rows of W."""
    if Wd is None:
        Wd = dequant(wtype, W, N, K)
    dY = np.asarray(dY, dtype=np.float32).reshape(T, N)
    ref = dY.astype(np.float64) @ Wd.astype(np.float64)
    if beta != 0.0:
        ref = ref + float(np.float32(beta)) * np.asarray(dX0, dtype=np.float32).reshape(T, K).astype(np.float64)
    return ref


def batch_weight(i2: int, i3: int, n2: int, n3: int, w_n2: int, w_n3: int):
    """Which weight (j2, j3) batch (i2, i3) of a batched OUT_PROD reads when
    there are w_n2 x w_n3 weights for n2 x n3 gradient batches: ggml's
    broadcast rule for out_prod, each weight serving a run of consecutive
    batches, j = i / (n / w_n) per dimension (the batched OUT_PROD whose
    broadcasting cases the llama.cpp fork's PR "cuda: out_prod accepts a
    quantized src0", section "Measured", reports skipped)."""
    if n2 % w_n2 or n3 % w_n3:
        raise ValueError("weight batch counts must divide the gradient's")
    return i2 // (n2 // w_n2), i3 // (n3 // w_n3)


def out_prod_batched(wtype: int, Ws, N: int, K: int, dYs, T: int, dX0s=None,
                     beta: float = 0.0):
    """F64 [n3][n2][T, K]: every batch (i2, i3) as out_prod with the weight
    batch_weight picks.  Ws[j3][j2] are the stored weights, dYs[i3][i2] the
    [T, N] gradients, dX0s[i3][i2] the old outputs (beta != 0)."""
    n3, n2 = len(dYs), len(dYs[0])
    w_n3, w_n2 = len(Ws), len(Ws[0])
    out = []
    for i3 in range(n3):
        row = []
        for i2 in range(n2):
            j2, j3 = batch_weight(i2, i3, n2, n3, w_n2, w_n3)
            row.append(out_prod(wtype, Ws[j3][j2], N, K, dYs[i3][i2], T,
                                None if dX0s is None else dX0s[i3][i2], beta))
        out.append(row)
    return out


def mul_mat(wtype: int, W, N: int, K: int, X, T: int, Y0=None, beta: float = 0.0,
            Wd=None) -> np.ndarray:
    """F64 [T, N]: beta*Y0 + X @ deq(W)^T, the forward mul_mat(W, x) whose
    backward OUT_PROD computes (llama.cpp fork PR "cuda: out_prod accepts a
    quantized src0", commit message): Y[t, n] = sum_k X[t, k] * deq(W)[n, k],
    contracted over the K values of each row of W."""
    if Wd is None:
        Wd = dequant(wtype, W, N, K)
    X = np.asarray(X, dtype=np.float32).reshape(T, K)
    ref = X.astype(np.float64) @ Wd.astype(np.float64).T
    if beta != 0.0:
        ref = ref + float(np.float32(beta)) * np.asarray(Y0, dtype=np.float32).reshape(T, N).astype(np.float64)
    return ref


def mul_mat_bound(X, Wd) -> np.ndarray:
    """F64 [T, N]: sum_k |X[t, k]| * |deq(W)[n, k]|."""
    return np.abs(np.asarray(X, dtype=np.float64)) @ np.abs(np.asarray(Wd, dtype=np.float64)).T


def abs_bound(dY, Wd) -> np.ndarray:
    """F64 [T, K]: sum_n |dY[t, n]| * |deq(W)[n, k]|."""
    return np.abs(np.asarray(dY, dtype=np.float64)) @ np.abs(np.asarray(Wd, dtype=np.float64))


def out_prod_lora(wtype: int, W, N: int, K: int, dY, T: int, lora_a, lora_b, r: int,
                  scale: float, dX0=None, beta: float = 0.0, Wd=None) -> np.ndarray:
    """F64 [T, K]: the input gradient through the resident base weight AND a
    low-rank adapter beside it,

        dX = beta*dX0 + dY @ deq(W) + scale * (dY @ B) @ A,

    for the forward y = x deq(W)^T + scale * (x A^T) B^T with A [r, K] (the
    adapter's down projection) and B [N, r] (its up projection).  The pages
    name the use (llama.cpp fork PR "cuda: out_prod accepts a quantized src0",
    commit message: a LoRA training on a resident Q4_K_M base) without the
    adapter's formula; this is the plain low-rank-adapter reading.

    Steps, in this order: (1) the base term as out_prod; (2) U = dY @ B over
    the N outputs, F64 (every F32 x F32 product exact); (3) scale * U @ A over
    the r ranks, F64, added to (1)."""
    ref = out_prod(wtype, W, N, K, dY, T, dX0, beta, Wd)
    if r == 0:
        return ref
    dY64 = np.asarray(dY, dtype=np.float32).reshape(T, N).astype(np.float64)
    A = np.asarray(lora_a, dtype=np.float32).reshape(r, K).astype(np.float64)
    B = np.asarray(lora_b, dtype=np.float32).reshape(N, r).astype(np.float64)
    U = dY64 @ B
    return ref + float(np.float32(scale)) * (U @ A)


def lora_bound(dY, lora_a, lora_b, scale: float) -> np.ndarray:
    """F64 [T, K]: |scale| * sum_j (sum_n |dY[t, n]| |B[n, j]|) |A[j, k]|, the
    adapter term's share of the acceptance bound."""
    dY = np.abs(np.asarray(dY, dtype=np.float64))
    A = np.abs(np.asarray(lora_a, dtype=np.float64))
    B = np.abs(np.asarray(lora_b, dtype=np.float64))
    return abs(float(np.float32(scale))) * ((dY @ B) @ A)


def out_prod_at(Wd, dY, ts, ks, dX0=None, beta: float = 0.0):
    """Selected outputs one by one: (ref, bound) at pairs (ts[i], ks[i]).

    Each is the F64 dot product of row ts[i] of dY with column ks[i] of deq(W)
    (plus beta*dX0 there), for parity checks on sizes whose full product is
    too large to form on the CPU."""
    ts = np.asarray(ts, dtype=np.int64)
    ks = np.asarray(ks, dtype=np.int64)
    rows = np.asarray(dY, dtype=np.float32)[ts].astype(np.float64)   # [S, N]
    cols = np.asarray(Wd, dtype=np.float32)[:, ks].T.astype(np.float64)  # [S, N]
    ref = np.einsum("sn,sn->s", rows, cols)
    bnd = np.einsum("sn,sn->s", np.abs(rows), np.abs(cols))
    if beta != 0.0:
        ref = ref + float(np.float32(beta)) * np.asarray(dX0, dtype=np.float32)[ts, ks].astype(np.float64)
    return ref, bnd


def mul_mat_at(Wd, X, ts, ns, Y0=None, beta: float = 0.0):
    """Selected outputs of the forward one by one: (ref, bound) at pairs
    (ts[i], ns[i]), each the F64 dot product of row ts[i] of X with row ns[i]
    of deq(W) (plus beta*Y0 there; see mul_mat), and sum_k |X| |deq(W)|, for
    parity checks on sizes whose full product is too large to form."""
    ts = np.asarray(ts, dtype=np.int64)
    ns = np.asarray(ns, dtype=np.int64)
    rows = np.asarray(X, dtype=np.float32)[ts].astype(np.float64)    # [S, K]
    wrow = np.asarray(Wd, dtype=np.float32)[ns].astype(np.float64)   # [S, K]
    ref = np.einsum("sk,sk->s", rows, wrow)
    bnd = np.einsum("sk,sk->s", np.abs(rows), np.abs(wrow))
    if beta != 0.0:
        ref = ref + float(np.float32(beta)) * np.asarray(Y0, dtype=np.float32)[ts, ns].astype(np.float64)
    return ref, bnd


def lora_at(dY, lora_a, lora_b, scale: float, ts, ks):
    """The adapter term at pairs (ts[i], ks[i]) one by one: (value, bound) of
    scale * sum_j (dY[t] . B[:, j]) A[j, k] and of its absolute terms, F64,
    for parity checks on sizes whose full product is too large to form."""
    ts = np.asarray(ts, dtype=np.int64)
    ks = np.asarray(ks, dtype=np.int64)
    sc = float(np.float32(scale))
    rows = np.asarray(dY, dtype=np.float32)[ts].astype(np.float64)          # [S, N]
    B = np.asarray(lora_b, dtype=np.float32).astype(np.float64)             # [N, r]
    cols = np.asarray(lora_a, dtype=np.float32)[:, ks].T.astype(np.float64)  # [S, r]
    U = rows @ B                                                             # [S, r]
    Ua = np.abs(rows) @ np.abs(B)
    return sc * np.einsum("sr,sr->s", U, cols), abs(sc) * np.einsum("sr,sr->s", Ua, np.abs(cols))

