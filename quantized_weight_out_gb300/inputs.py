"""Seeded synthetic inputs for the quantized-weight OUT_PROD.

This module only *produces* bytes and F32 arrays; it holds none of the
operation's arithmetic (no decode, no contraction).  Both the CPU oracle and
the CUDA path are fed from here, so the two always see identical inputs.

Random numbers
--------------
Every value is a pure function of (seed, stream, field, index):

* ``splitmix64`` - the output mix of SplitMix64 (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).  The i-th
  draw of a stream is the (i+1)-th SplitMix64 output from the stream's key,
  i.e. ``mix(key + (i + 1) * GAMMA)``.
* uniforms in (0, 1] take the top 53 bits: ``((x >> 11) + 1) * 2**-53``.
* normals use the cosine branch of Box and Muller (1958) on draws 2i and 2i+1.

Formats written (little-endian, the block layouts of ggml's GGUF types):

* Q8_0  34 B / 32 values: fp16 ``d`` then 32 int8 ``qs``.
* Q4_0  18 B / 32 values: fp16 ``d`` then 16 bytes; value j<16 sits in the low
  nibble of byte j, value j+16 in the high nibble.
* Q4_K 144 B / 256 values: fp16 ``d``, fp16 ``dmin``, 12 bytes of 6-bit
  (scale, min) pairs for 8 sub-blocks, 128 bytes of nibbles.
* Q4_1  20 B / 32 values: fp16 ``d``, fp16 ``m``, 16 bytes of nibbles (as Q4_0).
* Q5_0  22 B / 32 values: fp16 ``d``, 4 bytes ``qh`` (bit i of the
  little-endian word = fifth bit of value i), 16 bytes of nibbles.
* Q5_1  24 B / 32 values: fp16 ``d``, fp16 ``m``, ``qh``, 16 bytes of nibbles.
* Q5_K 176 B / 256 values: the Q4_K header, 32 bytes ``qh`` (bit 2c / 2c+1 of
  ``qh[l]`` = fifth bit of value 64c+l / 64c+32+l), 128 bytes of nibbles.
* Q6_K 210 B / 256 values: ``ql[128]`` (low 4 bits), ``qh[64]`` (2 high bits
  each), 16 int8 ``scales``, fp16 ``d``.
* Q2_K  84 B / 256 values: 16 bytes of (scale | min << 4), ``qs[64]`` (2 bits
  each: value 128h + 32j + 16s + l in bits 2j..2j+1 of ``qs[32h + 16s + l]``),
  fp16 ``d``, fp16 ``dmin``.
* Q3_K 110 B / 256 values: ``hmask[32]`` (bit 4h + j of ``hmask[16s + l]``:
  the value's third bit), ``qs[64]`` (low 2 bits as Q2_K), 12 bytes of
  sixteen 6-bit scales, fp16 ``d``.
* MXFP4 17 B / 32 values: E8M0 scale byte, 16 bytes of E2M1 nibbles (as Q4_0).
* NVFP4 36 B / 64 values: four E4M3 scale bytes (one per 16 values), 32
  bytes of E2M1 nibbles; the 16 values of scale s in bytes 8s .. 8s+7,
  value 16s + j (j < 8) in the low nibble of byte 8s + j, 16s + j + 8 in
  its high nibble.
* F16 / BF16: 2 B per value; F32: 4 B per value.

The generator recipes follow the workload descriptions of the llama.cpp fork's
PR "cuda: out_prod accepts a quantized src0" (the shapes a LoRA backward sees)
as restated in the workload table below.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional

import numpy as np

# ----------------------------------------------------------------------------
# weight type codes (the C ABI uses the same integers)
F16, BF16, Q8_0, Q4_0, Q4_K = 1, 2, 3, 4, 5
Q4_1, Q5_0, Q5_1, Q5_K, Q6_K, F32 = 6, 7, 8, 9, 10, 11
Q2_K, Q3_K, MXFP4, NVFP4 = 12, 13, 14, 15
TYPE_NAMES = {F16: "f16", BF16: "bf16", Q8_0: "q8_0", Q4_0: "q4_0", Q4_K: "q4_k",
              Q4_1: "q4_1", Q5_0: "q5_0", Q5_1: "q5_1", Q5_K: "q5_k", Q6_K: "q6_k", F32: "f32",
              Q2_K: "q2_k", Q3_K: "q3_k", MXFP4: "mxfp4", NVFP4: "nvfp4"}
NAME_TO_TYPE = {v: k for k, v in TYPE_NAMES.items()}
ALL_TYPES = [Q8_0, Q4_0, Q4_K, F16, BF16, Q4_1, Q5_0, Q5_1, Q5_K, Q6_K, F32, Q2_K, Q3_K, MXFP4,
             NVFP4]

# (values per block, bytes per block)
BLOCK = {F16: (1, 2), BF16: (1, 2), Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144),
         Q4_1: (32, 20), Q5_0: (32, 22), Q5_1: (32, 24), Q5_K: (256, 176),
         Q6_K: (256, 210), F32: (1, 4), Q2_K: (256, 84), Q3_K: (256, 110),
         MXFP4: (32, 17), NVFP4: (64, 36)}


def row_bytes(wtype: int, K: int) -> int:
    """Bytes of one stored row of K values (0 when K does not fit the type)."""
    if wtype not in BLOCK or K <= 0:
        return 0
    bs, bb = BLOCK[wtype]
    if K % bs:
        return 0
    return K // bs * bb


# ----------------------------------------------------------------------------
# counter-based random numbers

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)


def _mix(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int, field: int = 0) -> np.uint64:
    """Key of one (seed, stream, field) sequence."""
    with np.errstate(over="ignore"):
        k = _mix(np.array([seed], dtype=np.uint64))[0]
        k = _mix(np.array([k ^ (np.uint64(stream) * _STREAM_MUL)], dtype=np.uint64))[0]
        k = _mix(np.array([k ^ (np.uint64(field + 1) * _GAMMA)], dtype=np.uint64))[0]
    return np.uint64(k)


def draws_u64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Draws start..start+count-1 of the sequence with this key."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + idx * _GAMMA)


def uniform01(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Uniforms in (0, 1] (float64)."""
    x = draws_u64(key, start, count)
    return ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


_CHUNK = 1 << 20
_THREADS = max(1, min(32, os.cpu_count() or 1))


def _chunked(count: int, fill) -> None:
    """Run fill(start, n) over chunks of [0, count) on a thread pool (numpy
    releases the GIL inside its loops).  Results do not depend on chunking."""
    spans = [(s, min(_CHUNK, count - s)) for s in range(0, count, _CHUNK)]
    if len(spans) <= 1 or _THREADS == 1:
        for s, n in spans:
            fill(s, n)
        return
    with ThreadPoolExecutor(_THREADS) as ex:
        list(ex.map(lambda sn: fill(*sn), spans))


def normal_f32(seed: int, stream: int, count: int, sigma: float, field: int = 0) -> np.ndarray:
    """``count`` draws of N(0, sigma^2), rounded to float32."""
    key = stream_key(seed, stream, field)
    out = np.empty(count, dtype=np.float32)

    def fill(s, n):
        u = uniform01(key, 2 * s, 2 * n)
        u1, u2 = u[0::2], u[1::2]
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        out[s:s + n] = (sigma * z).astype(np.float32)
    _chunked(count, fill)
    return out


def uniform_int(seed: int, stream: int, count: int, modulus: int, field: int) -> np.ndarray:
    """``count`` integers uniform on {0..modulus-1}; modulus divides 2**64."""
    assert modulus & (modulus - 1) == 0
    key = stream_key(seed, stream, field)
    out = np.empty(count, dtype=np.int64)

    def fill(s, n):
        out[s:s + n] = (draws_u64(key, s, n) & np.uint64(modulus - 1)).astype(np.int64)
    _chunked(count, fill)
    return out


# ----------------------------------------------------------------------------
# encoders (F32 -> stored bits).  Round-to-nearest-even throughout.

def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE binary16 bits of x, round to nearest even (numpy's cast)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bfloat16 bits of finite x, round to nearest even."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def _round_half_away(v: np.ndarray) -> np.ndarray:
    return np.sign(v) * np.floor(np.abs(v) + np.float32(0.5))


def _f16_le(bits: np.ndarray) -> np.ndarray:
    """uint16 array [...] -> uint8 array [..., 2] little-endian."""
    b = bits.astype(np.uint16)
    return np.stack([(b & 0xFF).astype(np.uint8), (b >> 8).astype(np.uint8)], axis=-1)


def quantize_q8_0(x: np.ndarray, N: int, K: int) -> np.ndarray:
    """Q8_0 blocks of x [N, K]: d = amax/127 stored fp16, q = round(x/d)."""
    xb = np.asarray(x, dtype=np.float32).reshape(N, K // 32, 32)
    amax = np.max(np.abs(xb), axis=-1)
    d32 = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(d32[..., None] > 0, xb / d32[..., None], np.float32(0))
    q = np.clip(_round_half_away(v.astype(np.float32)), -127, 127).astype(np.int8)
    out = np.empty((N, K // 32, 34), dtype=np.uint8)
    out[..., 0:2] = _f16_le(f32_to_f16_bits(d32))
    out[..., 2:34] = q.view(np.uint8)
    return out.reshape(-1)


def quantize_q4_0(x: np.ndarray, N: int, K: int) -> np.ndarray:
    """Q4_0 blocks: d = mx/-8 (mx the signed value of largest magnitude, first
    on ties), q = clamp(round(x/d) + 8, 0, 15)."""
    xb = np.asarray(x, dtype=np.float32).reshape(N, K // 32, 32)
    idx = np.argmax(np.abs(xb), axis=-1)
    mx = np.take_along_axis(xb, idx[..., None], axis=-1)[..., 0]
    d32 = (mx / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(d32[..., None] != 0, xb / d32[..., None], np.float32(0))
    q = np.clip(_round_half_away(v.astype(np.float32)) + 8, 0, 15).astype(np.uint8)
    out = np.empty((N, K // 32, 18), dtype=np.uint8)
    out[..., 0:2] = _f16_le(f32_to_f16_bits(d32))
    out[..., 2:18] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(-1)


def pack_q4_k(d_bits, dmin_bits, sc, m, q) -> np.ndarray:
    """Pack Q4_K super-blocks from their fields.

    d_bits, dmin_bits: [B] uint16; sc, m: [B, 8] ints in 0..63; q: [B, 256]
    ints in 0..15 (value index order).  Returns uint8 [B, 144]."""
    B = d_bits.shape[0]
    sc = np.asarray(sc, dtype=np.uint8)
    m = np.asarray(m, dtype=np.uint8)
    q = np.asarray(q, dtype=np.uint8)
    S = np.zeros((B, 12), dtype=np.uint8)
    for j in range(4):
        # sub-blocks 0..3: 6 bits in S[j] / S[j+4]; their top bits carry the
        # 2 high bits of sub-blocks 4..7.
        S[:, j] = (sc[:, j] & 63) | ((sc[:, j + 4] >> 4) << 6)
        S[:, j + 4] = (m[:, j] & 63) | ((m[:, j + 4] >> 4) << 6)
        S[:, j + 8] = (sc[:, j + 4] & 15) | ((m[:, j + 4] & 15) << 4)
    qs = np.zeros((B, 128), dtype=np.uint8)
    for c in range(4):
        lo = q[:, 64 * c: 64 * c + 32]
        hi = q[:, 64 * c + 32: 64 * c + 64]
        qs[:, 32 * c: 32 * c + 32] = lo | (hi << 4)
    out = np.empty((B, 144), dtype=np.uint8)
    out[:, 0:2] = _f16_le(d_bits)
    out[:, 2:4] = _f16_le(dmin_bits)
    out[:, 4:16] = S
    out[:, 16:144] = qs
    return out


def _pack_nibbles_32(q: np.ndarray) -> np.ndarray:
    """[B, 32] values 0..15 -> [B, 16] bytes: value j < 16 in the low nibble
    of byte j, value j + 16 in the high nibble."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, :16] & 15) | ((q[:, 16:] & 15) << 4)


def _pack_fifth_bits_32(q: np.ndarray) -> np.ndarray:
    """[B, 32] values 0..31 -> [B, 4] bytes of the little-endian word whose
    bit i is bit 4 of value i."""
    hb = (np.asarray(q, dtype=np.uint64) >> np.uint64(4)) & np.uint64(1)
    word = np.zeros(hb.shape[0], dtype=np.uint64)
    for i in range(32):
        word |= hb[:, i] << np.uint64(i)
    return np.stack([((word >> np.uint64(8 * b)) & np.uint64(0xFF)).astype(np.uint8)
                     for b in range(4)], axis=-1)


def pack_q4_1(d_bits, m_bits, q) -> np.ndarray:
    """Q4_1 blocks [B, 20] from fp16 d, fp16 m and values q [B, 32] in 0..15."""
    B = len(d_bits)
    out = np.empty((B, 20), dtype=np.uint8)
    out[:, 0:2] = _f16_le(np.asarray(d_bits, dtype=np.uint16))
    out[:, 2:4] = _f16_le(np.asarray(m_bits, dtype=np.uint16))
    out[:, 4:20] = _pack_nibbles_32(q)
    return out


def pack_q5_0(d_bits, q) -> np.ndarray:
    """Q5_0 blocks [B, 22] from fp16 d and values q [B, 32] in 0..31."""
    B = len(d_bits)
    out = np.empty((B, 22), dtype=np.uint8)
    out[:, 0:2] = _f16_le(np.asarray(d_bits, dtype=np.uint16))
    out[:, 2:6] = _pack_fifth_bits_32(q)
    out[:, 6:22] = _pack_nibbles_32(np.asarray(q) & 15)
    return out


def pack_q5_1(d_bits, m_bits, q) -> np.ndarray:
    """Q5_1 blocks [B, 24] from fp16 d, fp16 m and values q [B, 32] in 0..31."""
    B = len(d_bits)
    out = np.empty((B, 24), dtype=np.uint8)
    out[:, 0:2] = _f16_le(np.asarray(d_bits, dtype=np.uint16))
    out[:, 2:4] = _f16_le(np.asarray(m_bits, dtype=np.uint16))
    out[:, 4:8] = _pack_fifth_bits_32(q)
    out[:, 8:24] = _pack_nibbles_32(np.asarray(q) & 15)
    return out


def pack_q5_k(d_bits, dmin_bits, sc, m, q) -> np.ndarray:
    """Q5_K super-blocks [B, 176]: the Q4_K packing of (d, dmin, sc, m) and of
    the low nibbles of q [B, 256] (values 0..31), plus qh[32] whose bit 2c of
    byte l is bit 4 of value 64c+l and bit 2c+1 that of value 64c+32+l."""
    q = np.asarray(q, dtype=np.uint8)
    k4 = pack_q4_k(d_bits, dmin_bits, sc, m, q & 15)
    B = k4.shape[0]
    qh = np.zeros((B, 32), dtype=np.uint8)
    for c in range(4):
        qh |= ((q[:, 64 * c: 64 * c + 32] >> 4) & 1) << (2 * c)
        qh |= ((q[:, 64 * c + 32: 64 * c + 64] >> 4) & 1) << (2 * c + 1)
    out = np.empty((B, 176), dtype=np.uint8)
    out[:, 0:16] = k4[:, 0:16]
    out[:, 16:48] = qh
    out[:, 48:176] = k4[:, 16:144]
    return out


def pack_q6_k(d_bits, sc, q) -> np.ndarray:
    """Q6_K super-blocks [B, 210] from fp16 d, int8 scales sc [B, 16] and
    values q [B, 256] in 0..63 (value 128h + 32i + l: low bits in the low
    (i < 2) or high nibble of ql[64h + 32(i % 2) + l], high bits in bits
    2i..2i+1 of qh[32h + l])."""
    q = np.asarray(q, dtype=np.uint8)
    B = q.shape[0]
    ql = np.zeros((B, 128), dtype=np.uint8)
    qh = np.zeros((B, 64), dtype=np.uint8)
    for h in range(2):
        for i in range(4):
            v = q[:, 128 * h + 32 * i: 128 * h + 32 * i + 32]
            at = 64 * h + 32 * (i % 2)
            ql[:, at: at + 32] |= (v & 15) << (4 if i >= 2 else 0)
            qh[:, 32 * h: 32 * h + 32] |= ((v >> 4) & 3) << (2 * i)
    out = np.empty((B, 210), dtype=np.uint8)
    out[:, 0:128] = ql
    out[:, 128:192] = qh
    out[:, 192:208] = np.asarray(sc, dtype=np.int8).view(np.uint8)
    out[:, 208:210] = _f16_le(np.asarray(d_bits, dtype=np.uint16))
    return out


def pack_q2_k(d_bits, dmin_bits, sc, m, q) -> np.ndarray:
    """Q2_K super-blocks [B, 84] from fp16 d and dmin, 4-bit scales sc and
    mins m [B, 16] and values q [B, 256] in 0..3 (value 128h + 32j + 16s + l
    in bits 2j..2j+1 of qs[32h + 16s + l]; its scales byte 8h + 2j + s)."""
    q = np.asarray(q, dtype=np.uint8)
    B = q.shape[0]
    qs = np.zeros((B, 64), dtype=np.uint8)
    for h in range(2):
        for j in range(4):
            for s in range(2):
                v0 = 128 * h + 32 * j + 16 * s
                qs[:, 32 * h + 16 * s: 32 * h + 16 * s + 16] |= (q[:, v0: v0 + 16] & 3) << (2 * j)
    out = np.empty((B, 84), dtype=np.uint8)
    out[:, 0:16] = (np.asarray(sc, dtype=np.uint8) & 15) | (np.asarray(m, dtype=np.uint8) << 4)
    out[:, 16:80] = qs
    out[:, 80:82] = _f16_le(np.asarray(d_bits, dtype=np.uint16))
    out[:, 82:84] = _f16_le(np.asarray(dmin_bits, dtype=np.uint16))
    return out


def pack_q3_k(d_bits, sc6, q) -> np.ndarray:
    """Q3_K super-blocks [B, 110] from fp16 d, 6-bit scales sc6 [B, 16] in
    0..63 (the scale used is sc6 - 32) and values q [B, 256] in -4..3 (low
    2 bits as Q2_K, hmask bit set when q >= 0)."""
    q = np.asarray(q, dtype=np.int64)
    B = q.shape[0]
    low = (q & 3).astype(np.uint8)            # q + 4 = low + 4 * bit: low = q mod 4
    bit = (q >= 0).astype(np.uint8)
    hm = np.zeros((B, 32), dtype=np.uint8)
    qs = np.zeros((B, 64), dtype=np.uint8)
    for h in range(2):
        for j in range(4):
            for s in range(2):
                v0 = 128 * h + 32 * j + 16 * s
                qs[:, 32 * h + 16 * s: 32 * h + 16 * s + 16] |= low[:, v0: v0 + 16] << (2 * j)
                hm[:, 16 * s: 16 * s + 16] |= bit[:, v0: v0 + 16] << (4 * h + j)
    sc6 = np.asarray(sc6, dtype=np.uint8)
    S = np.zeros((B, 12), dtype=np.uint8)
    for i in range(16):
        if i < 8:
            S[:, i] |= sc6[:, i] & 15
        else:
            S[:, i - 8] |= (sc6[:, i] & 15) << 4
        S[:, 8 + i % 4] |= (sc6[:, i] >> 4) << (2 * (i // 4))
    out = np.empty((B, 110), dtype=np.uint8)
    out[:, 0:32] = hm
    out[:, 32:96] = qs
    out[:, 96:108] = S
    out[:, 108:110] = _f16_le(np.asarray(d_bits, dtype=np.uint16))
    return out


def pack_mxfp4(e, q) -> np.ndarray:
    """MXFP4 blocks [nb, 17] from E8M0 scale bytes e [nb] and 4-bit E2M1
    codes q [nb, 32] (value j < 16 in the low nibble of byte j, value j + 16
    in its high nibble)."""
    e = np.asarray(e, dtype=np.uint8)
    out = np.zeros((e.shape[0], 17), dtype=np.uint8)
    out[:, 0] = e
    out[:, 1:17] = _pack_nibbles_32(q)
    return out


def pack_nvfp4(d, q) -> np.ndarray:
    """NVFP4 blocks [nb, 36] from E4M3 scale bytes d [nb, 4] and 4-bit E2M1
    codes q [nb, 64]: the 16 codes of scale s go to bytes 4 + 8s .. 11 + 8s,
    code 16s + j (j < 8) in the low nibble, 16s + j + 8 in the high one."""
    d = np.asarray(d, dtype=np.uint8)
    q = np.asarray(q, dtype=np.uint8).reshape(-1, 4, 16)
    out = np.zeros((d.shape[0], 36), dtype=np.uint8)
    out[:, 0:4] = d
    out[:, 4:36] = (q[..., :8] | (q[..., 8:] << 4)).reshape(-1, 32)
    return out


# ----------------------------------------------------------------------------
# weights and activations for one call

def gen_weight(wtype: int, N: int, K: int, seed: int, stream: int) -> np.ndarray:
    """Stored bytes of an N x K weight, uint8 [N * row_bytes(wtype, K)]."""
    if row_bytes(wtype, K) == 0:
        raise ValueError(f"K={K} does not fit type {wtype}")
    if wtype == Q4_K:
        nb = N * K // 256
        d = np.abs(normal_f32(seed, stream, nb, 1e-3, field=1))
        dmin = np.abs(normal_f32(seed, stream, nb, 1e-3, field=2))
        sc = uniform_int(seed, stream, nb * 8, 64, field=3).reshape(nb, 8)
        m = uniform_int(seed, stream, nb * 8, 64, field=4).reshape(nb, 8)
        q = uniform_int(seed, stream, nb * 256, 16, field=5).reshape(nb, 256)
        return pack_q4_k(f32_to_f16_bits(d), f32_to_f16_bits(dmin), sc, m, q).reshape(-1)
    if wtype == Q5_K:
        nb = N * K // 256
        d = np.abs(normal_f32(seed, stream, nb, 1e-3, field=1))
        dmin = np.abs(normal_f32(seed, stream, nb, 1e-3, field=2))
        sc = uniform_int(seed, stream, nb * 8, 64, field=3).reshape(nb, 8)
        m = uniform_int(seed, stream, nb * 8, 64, field=4).reshape(nb, 8)
        q = uniform_int(seed, stream, nb * 256, 32, field=5).reshape(nb, 256)
        return pack_q5_k(f32_to_f16_bits(d), f32_to_f16_bits(dmin), sc, m, q).reshape(-1)
    if wtype == Q6_K:
        # fields drawn directly: |d * sc * (q - 32)| ~ 2e-5 * 64 * 16 ~ 0.02
        nb = N * K // 256
        d = np.abs(normal_f32(seed, stream, nb, 2e-5, field=1))
        sc = uniform_int(seed, stream, nb * 16, 256, field=3).reshape(nb, 16) - 128
        q = uniform_int(seed, stream, nb * 256, 64, field=5).reshape(nb, 256)
        return pack_q6_k(f32_to_f16_bits(d), sc, q).reshape(-1)
    if wtype == Q2_K:
        # fields drawn directly: |d * sc * q| ~ 5e-4 * 15 * 3 ~ 0.02
        nb = N * K // 256
        d = np.abs(normal_f32(seed, stream, nb, 5e-4, field=1))
        dmin = np.abs(normal_f32(seed, stream, nb, 5e-4, field=2))
        sc = uniform_int(seed, stream, nb * 16, 16, field=3).reshape(nb, 16)
        m = uniform_int(seed, stream, nb * 16, 16, field=4).reshape(nb, 16)
        q = uniform_int(seed, stream, nb * 256, 4, field=5).reshape(nb, 256)
        return pack_q2_k(f32_to_f16_bits(d), f32_to_f16_bits(dmin), sc, m, q).reshape(-1)
    if wtype == Q3_K:
        # fields drawn directly, d signed: |d * (sc - 32) * q| ~ 2e-4 * 32 * 4
        nb = N * K // 256
        d = normal_f32(seed, stream, nb, 2e-4, field=1)
        sc6 = uniform_int(seed, stream, nb * 16, 64, field=3).reshape(nb, 16)
        q = uniform_int(seed, stream, nb * 256, 8, field=5).reshape(nb, 256) - 4
        return pack_q3_k(f32_to_f16_bits(d), sc6, q).reshape(-1)
    if wtype == MXFP4:
        # fields drawn directly: a scale 2^(e - 127) with e in 118..121 and
        # uniform codes give |y| <= 6 * 2^-6 ~ 0.09 (most near 0.01), every
        # nonzero value a normal fp16 (the tensor-core operand)
        nb = N * K // 32
        e = 118 + uniform_int(seed, stream, nb, 4, field=1)
        q = uniform_int(seed, stream, nb * 32, 16, field=5).reshape(nb, 32)
        return pack_mxfp4(e, q).reshape(-1)
    if wtype == NVFP4:
        # fields drawn directly: E4M3 scale bytes 0x00..0x0f (zero, the
        # subnormals m/8 * 2^-6 and the first binade 2^-6 (1 + m/8)) and
        # uniform E2M1 codes give |y| <= 6 * 0.0293 ~ 0.18 (most near 0.02)
        nb = N * K // 64
        d = uniform_int(seed, stream, nb * 4, 16, field=1).reshape(nb, 4)
        q = uniform_int(seed, stream, nb * 64, 16, field=5).reshape(nb, 64)
        return pack_nvfp4(d, q).reshape(-1)
    if wtype in (Q4_1, Q5_0, Q5_1):
        # fields drawn directly (the pages give no workload of these types):
        # a block of N(0, 0.02) weights spans about 0.08, so d ~ 0.08 / levels
        nb = N * K // 32
        levels = 16 if wtype == Q4_1 else 32
        dsig = 0.08 / (levels - 1)
        q = uniform_int(seed, stream, nb * 32, levels, field=5).reshape(nb, 32)
        if wtype == Q5_0:
            d = normal_f32(seed, stream, nb, dsig, field=1)          # signed, like Q4_0's mx/-8
            return pack_q5_0(f32_to_f16_bits(d), q).reshape(-1)
        d = np.abs(normal_f32(seed, stream, nb, dsig, field=1))
        m = normal_f32(seed, stream, nb, 0.04, field=2)
        if wtype == Q4_1:
            return pack_q4_1(f32_to_f16_bits(d), f32_to_f16_bits(m), q).reshape(-1)
        return pack_q5_1(f32_to_f16_bits(d), f32_to_f16_bits(m), q).reshape(-1)
    x = normal_f32(seed, stream, N * K, 0.02)
    if wtype == Q8_0:
        return quantize_q8_0(x, N, K)
    if wtype == Q4_0:
        return quantize_q4_0(x, N, K)
    if wtype == F16:
        return f32_to_f16_bits(x).view(np.uint8).copy()
    if wtype == BF16:
        return f32_to_bf16_bits(x).view(np.uint8).copy()
    if wtype == F32:
        return x.astype("<f4").view(np.uint8).copy()
    raise ValueError(f"unknown weight type {wtype}")


@dataclasses.dataclass
class Problem:
    """One OUT_PROD call: dX[T,K] = beta*dX0 + dY[T,N] . deq(W)[N,K]."""
    name: str
    wtype: int
    N: int
    K: int
    T: int
    dy_sigma: float
    beta: float = 0.0
    stream_base: int = 0     # added to the W / dY / dX0 stream ids (1, 2, 3)
    seed: int = 0

    @property
    def flops(self) -> int:
        return 2 * self.T * self.N * self.K

    @property
    def w_bytes(self) -> int:
        return self.N * row_bytes(self.wtype, self.K)

    def algorithmic_bytes(self) -> int:
        """bytes(W) + 4T(N+K) (+4TK when beta != 0)."""
        b = self.w_bytes + 4 * self.T * (self.N + self.K)
        if self.beta != 0.0:
            b += 4 * self.T * self.K
        return b

    # Every generator is counter-based in row-major order, so the first `rows`
    # rows of an input are exactly what a smaller call would generate.

    def weight(self, rows: Optional[int] = None) -> np.ndarray:
        n = self.N if rows is None else min(rows, self.N)
        return gen_weight(self.wtype, n, self.K, self.seed, 1 + self.stream_base)

    def dy(self, rows: Optional[int] = None) -> np.ndarray:
        t = self.T if rows is None else min(rows, self.T)
        return normal_f32(self.seed, 2 + self.stream_base, t * self.N,
                          self.dy_sigma).reshape(t, self.N)

    def dx0(self, rows: Optional[int] = None) -> Optional[np.ndarray]:
        if self.beta == 0.0:
            return None
        t = self.T if rows is None else min(rows, self.T)
        return normal_f32(self.seed, 3 + self.stream_base, t * self.K,
                          1e-3).reshape(t, self.K)


def _layer_sweep(T: int = 8192) -> List[Problem]:
    shapes = [("q", Q4_K, 4096, 4096), ("k", Q4_K, 1024, 4096), ("v", Q4_K, 1024, 4096),
              ("o", Q4_K, 4096, 4096), ("gate", Q4_K, 14336, 4096),
              ("up", Q4_K, 14336, 4096), ("down", Q8_0, 4096, 14336)]
    return [Problem(f"layer7b_{nm}", wt, n, k, T, 1e-3, 0.0, 16 * i)
            for i, (nm, wt, n, k) in enumerate(shapes)]


# The workloads: each is a list of independent calls.
WORKLOADS = {
    "q8_0_256x256_t32": [Problem("q8_0_256x256_t32", Q8_0, 256, 256, 32, 1.0)],
    "q4_0_4096x4096_t512": [Problem("q4_0_4096x4096_t512", Q4_0, 4096, 4096, 512, 1e-3)],
    "q4_k_14336x4096_t2048": [Problem("q4_k_14336x4096_t2048", Q4_K, 14336, 4096, 2048, 1e-3)],
    "f16_5120x17408_t4096_beta1": [Problem("f16_5120x17408_t4096_beta1", F16, 5120, 17408, 4096, 1e-3, 1.0)],
    "bf16_5120x17408_t4096_beta1": [Problem("bf16_5120x17408_t4096_beta1", BF16, 5120, 17408, 4096, 1e-3, 1.0)],
    "layer7b_t8192": _layer_sweep(8192),
    # the sweep's largest call alone (profiling a full-size launch)
    "layer7b_gate_t8192": [_layer_sweep(8192)[4]],
    # one row of dY (a decode-time gradient): the weight-streaming small-T path
    "smallt_q4_k_14336x4096_t1": [Problem("smallt_q4_k_14336x4096_t1", Q4_K, 14336, 4096, 1, 1e-3)],
    "smallt_q8_0_4096x14336_t1": [Problem("smallt_q8_0_4096x14336_t1", Q8_0, 4096, 14336, 1, 1e-3)],
    # the other quantized types on the sweep's q/o shape, one call each
    "types_4096x4096_t8192": [Problem(f"{TYPE_NAMES[wt]}_4096x4096_t8192", wt, 4096, 4096, 8192,
                                      1e-3, 0.0, 16 * i)
                              for i, wt in enumerate([Q4_1, Q5_0, Q5_1, Q5_K, Q6_K, F32, Q2_K, Q3_K,
                                                      MXFP4, NVFP4])],
}
