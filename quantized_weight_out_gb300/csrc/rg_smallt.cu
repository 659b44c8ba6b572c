// rg_smallt.cu - the small-T variant of
//   dX[t, k] = beta * dX[t, k] + sum_n dY[t, n] * deq(W)[n, k]
// for a handful of rows of dY, where the bytes of W bound the product (the
// role of the in-place decoder the Retrograd page "CUDA status", section
// "Limitations", keeps for small outputs).
//
// Every weight value is read from memory once per pass of up to 8 dY rows.
//  * A producer warp streams the CTA's rows of W (its 256-value tile of each
//    row) with TMA into a shared-memory ring of row stages, so enough bytes
//    are in flight without holding them in registers.
//  * Eight consumer warps decode from shared memory: Q4_K and Q8_0 through
//    the warp-level tensor-core MMA with the weight integers themselves as
//    exact fp16 operands (consume_mma); other quantized types at one or two dY rows
//    a block per warp and a row per lane in F32 (consume_rows); the rest
//    eight values a lane, decoded exactly to F32, F32 FMAs.
//  * The rows are split over many CTAs (grid.y) so that the whole GPU streams
//    W; each CTA writes its partial tile to a workspace, and a second kernel
//    adds the partials in split order together with beta * dX:
//    deterministic, no atomics.  With at most 256 rows of W one CTA per tile
//    takes them all and writes beta * dX + sum into dX itself.
#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {
namespace smt {

constexpr int THREADS = 256;   // 8 consumer warps (plus one producer warp)

// Raw bytes one lane needs from a row for its 8 values (a 256-value tile).
template <int WT>
struct Raw {
  uint32_t v[WT == RG_Q5_K || WT == RG_F32 ? 8
             : WT == RG_Q4_K                  ? 6
             : WT == RG_Q6_K || WT == RG_Q3_K ? 5
             : (WT == RG_Q8_0 || WT == RG_Q4_0 || WT == RG_Q4_1 || WT == RG_MXFP4 ||
                WT == RG_NVFP4)                                                       ? 3
                                                                                    : 4];
};

// The bytes one lane needs for its 8 values, from a row tile staged in
// shared memory (tile: the row's 256-value tile, 16-byte aligned).
template <int WT>
__device__ __forceinline__ void load_raw_smem(const uint8_t* tile, int lane, Raw<WT>& r) {
  if constexpr (WT == RG_F32) {
    const uint4 a = reinterpret_cast<const uint4*>(tile)[2 * lane];
    const uint4 b = reinterpret_cast<const uint4*>(tile)[2 * lane + 1];
    r.v[0] = a.x; r.v[1] = a.y; r.v[2] = a.z; r.v[3] = a.w;
    r.v[4] = b.x; r.v[5] = b.y; r.v[6] = b.z; r.v[7] = b.w;
  } else if constexpr (WT == RG_F16 || WT == RG_BF16) {
    const uint4 q = reinterpret_cast<const uint4*>(tile)[lane];
    r.v[0] = q.x; r.v[1] = q.y; r.v[2] = q.z; r.v[3] = q.w;
  } else if constexpr (WT == RG_Q8_0 || WT == RG_Q4_0) {
    constexpr int BB = WT == RG_Q8_0 ? 34 : 18;
    const uint8_t* blk = tile + BB * (lane >> 2);
    const uint8_t* q = blk + 2 + 8 * (WT == RG_Q8_0 ? (lane & 3) : (lane & 1));
    const uint16_t* q16 = reinterpret_cast<const uint16_t*>(q);
    r.v[0] = *reinterpret_cast<const uint16_t*>(blk);
    r.v[1] = static_cast<uint32_t>(q16[0]) | (static_cast<uint32_t>(q16[1]) << 16);
    r.v[2] = static_cast<uint32_t>(q16[2]) | (static_cast<uint32_t>(q16[3]) << 16);
  } else if constexpr (WT == RG_MXFP4) {
    // values 8(lane & 3) .. +7 of block lane >> 2 (17-byte blocks from an
    // 8-byte aligned tile): the scale byte and 8 bytes of nibbles
    const uint8_t* blk = tile + 17 * (lane >> 2);
    const uint8_t* q = blk + 1 + 8 * (lane & 1);
    r.v[0] = blk[0];
    r.v[1] = static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 8) |
             (static_cast<uint32_t>(q[2]) << 16) | (static_cast<uint32_t>(q[3]) << 24);
    r.v[2] = static_cast<uint32_t>(q[4]) | (static_cast<uint32_t>(q[5]) << 8) |
             (static_cast<uint32_t>(q[6]) << 16) | (static_cast<uint32_t>(q[7]) << 24);
  } else if constexpr (WT == RG_NVFP4) {
    // values 8 lane .. +7: micro-block s = (lane & 7) >> 1 of block lane >> 3
    // (36-byte blocks from a 16-byte aligned tile): its scale byte and its 8
    // code bytes (low nibbles for even lanes, high for odd)
    const uint8_t* blk = tile + 36 * (lane >> 3);
    const int s = (lane & 7) >> 1;
    const uint32_t* q = reinterpret_cast<const uint32_t*>(blk + 4 + 8 * s);
    r.v[0] = blk[s];
    r.v[1] = q[0];
    r.v[2] = q[1];
  } else if constexpr (WT == RG_Q4_1) {
    const uint8_t* blk = tile + 20 * (lane >> 2);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(blk + 4 + 8 * (lane & 1));
    r.v[0] = *reinterpret_cast<const uint32_t*>(blk);  // d | m << 16
    r.v[1] = q[0];
    r.v[2] = q[1];
  } else if constexpr (WT == RG_Q5_0) {
    const uint8_t* blk = tile + 22 * (lane >> 2);
    const uint16_t* h16 = reinterpret_cast<const uint16_t*>(blk + 2);
    const uint16_t* q16 = reinterpret_cast<const uint16_t*>(blk + 6 + 8 * (lane & 1));
    r.v[0] = *reinterpret_cast<const uint16_t*>(blk);
    r.v[1] = static_cast<uint32_t>(h16[0]) | (static_cast<uint32_t>(h16[1]) << 16);
    r.v[2] = static_cast<uint32_t>(q16[0]) | (static_cast<uint32_t>(q16[1]) << 16);
    r.v[3] = static_cast<uint32_t>(q16[2]) | (static_cast<uint32_t>(q16[3]) << 16);
  } else if constexpr (WT == RG_Q5_1) {
    const uint8_t* blk = tile + 24 * (lane >> 2);
    const uint2 q = *reinterpret_cast<const uint2*>(blk + 8 + 8 * (lane & 1));
    r.v[0] = *reinterpret_cast<const uint32_t*>(blk);      // d | m << 16
    r.v[1] = *reinterpret_cast<const uint32_t*>(blk + 4);  // qh
    r.v[2] = q.x;
    r.v[3] = q.y;
  } else if constexpr (WT == RG_Q6_K) {
    // values 8*lane .. +7 = 128h + 32i + l0 .. +7 (tile: the super-block's
    // first byte, 2-byte aligned): 8 bytes of ql, 8 of qh, one scale, d
    const int h = lane >> 4, i = (lane >> 2) & 3, l0 = 8 * (lane & 3);
    const uint16_t* ql = reinterpret_cast<const uint16_t*>(tile + 64 * h + 32 * (i & 1) + l0);
    const uint16_t* qh = reinterpret_cast<const uint16_t*>(tile + 128 + 32 * h + l0);
    r.v[0] = static_cast<uint32_t>(ql[0]) | (static_cast<uint32_t>(ql[1]) << 16);
    r.v[1] = static_cast<uint32_t>(ql[2]) | (static_cast<uint32_t>(ql[3]) << 16);
    r.v[2] = static_cast<uint32_t>(qh[0]) | (static_cast<uint32_t>(qh[1]) << 16);
    r.v[3] = static_cast<uint32_t>(qh[2]) | (static_cast<uint32_t>(qh[3]) << 16);
    r.v[4] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(tile + 208)) |
             (static_cast<uint32_t>(tile[192 + (lane >> 1)]) << 16);
  } else if constexpr (WT == RG_Q2_K || WT == RG_Q3_K) {
    // values 8*lane .. +7 = 128h + 32j + 16s + l0 .. +7 (tile: the
    // super-block's first byte, 2-byte aligned): 8 bytes of qs (and of
    // hmask), the sub-block's scale byte(s), d (and dmin)
    const int h = lane >> 4, j = (lane >> 2) & 3, sb = (lane >> 1) & 1, l0 = 8 * (lane & 1);
    constexpr int QS = WT == RG_Q2_K ? 16 : 32;
    const uint16_t* q = reinterpret_cast<const uint16_t*>(tile + QS + 32 * h + 16 * sb + l0);
    r.v[0] = static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 16);
    r.v[1] = static_cast<uint32_t>(q[2]) | (static_cast<uint32_t>(q[3]) << 16);
    const int si = 8 * h + 2 * j + sb;
    if constexpr (WT == RG_Q2_K) {
      r.v[2] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(tile + 80)) |
               (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(tile + 82)) << 16);
      r.v[3] = tile[si];
    } else {
      const uint16_t* hm = reinterpret_cast<const uint16_t*>(tile + 16 * sb + l0);
      r.v[2] = static_cast<uint32_t>(hm[0]) | (static_cast<uint32_t>(hm[1]) << 16);
      r.v[3] = static_cast<uint32_t>(hm[2]) | (static_cast<uint32_t>(hm[3]) << 16);
      // d, the byte with the scale's low nibble, the byte with its high bits
      r.v[4] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(tile + 108)) |
               (static_cast<uint32_t>(tile[96 + (si & 7)]) << 16) |
               (static_cast<uint32_t>(tile[104 + (si & 3)]) << 24);
    }
  } else {
    // Q4_K, Q5_K: the header, this lane's 8 bytes of nibbles (and of qh)
    constexpr int QS = WT == RG_Q5_K ? 48 : 16;
    const uint4 h = *reinterpret_cast<const uint4*>(tile);
    const int c = lane >> 3, l0 = 8 * (lane & 3);
    const uint2 q = *reinterpret_cast<const uint2*>(tile + QS + 32 * c + l0);
    r.v[0] = h.x; r.v[1] = h.y; r.v[2] = h.z; r.v[3] = h.w; r.v[4] = q.x; r.v[5] = q.y;
    if constexpr (WT == RG_Q5_K) {
      const uint2 qh = *reinterpret_cast<const uint2*>(tile + 16 + l0);
      r.v[6] = qh.x;
      r.v[7] = qh.y;
    }
  }
}

__device__ __forceinline__ int byte_at(const uint32_t* w, int i) {
  return static_cast<int>((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
}

// Exact F32 decode of the lane's 8 values: the same products and single
// rounding as the format definitions (signed zeros kept).
template <int WT>
__device__ __forceinline__ void decode_raw(const Raw<WT>& r, int lane, float (&w)[8]) {
  if constexpr (WT == RG_F32) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __uint_as_float(r.v[i]);
  } else if constexpr (WT == RG_F16 || WT == RG_BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = static_cast<uint16_t>(r.v[i] & 0xFFFFu);
      const uint16_t hi = static_cast<uint16_t>(r.v[i] >> 16);
      w[2 * i] = WT == RG_F16 ? f16_to_f32(lo) : bf16_to_f32(lo);
      w[2 * i + 1] = WT == RG_F16 ? f16_to_f32(hi) : bf16_to_f32(hi);
    }
  } else if constexpr (WT == RG_Q8_0) {
    // int8 q as the byte q + 128, then d * q: an exact product
    const float d = f16_to_f32(static_cast<uint16_t>(r.v[0]));
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t x = r.v[1 + j] ^ 0x80808080u;
      w[4 * j + 0] = d * byte_minus<0>(x, kTwo23 + 128.0f);
      w[4 * j + 1] = d * byte_minus<1>(x, kTwo23 + 128.0f);
      w[4 * j + 2] = d * byte_minus<2>(x, kTwo23 + 128.0f);
      w[4 * j + 3] = d * byte_minus<3>(x, kTwo23 + 128.0f);
    }
  } else if constexpr (WT == RG_Q4_0) {
    const float d = f16_to_f32(static_cast<uint16_t>(r.v[0]));
    const int shift = (lane & 2) ? 4 : 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t x = (r.v[1 + j] >> shift) & 0x0F0F0F0Fu;
      w[4 * j + 0] = d * byte_minus<0>(x, kTwo23 + 8.0f);
      w[4 * j + 1] = d * byte_minus<1>(x, kTwo23 + 8.0f);
      w[4 * j + 2] = d * byte_minus<2>(x, kTwo23 + 8.0f);
      w[4 * j + 3] = d * byte_minus<3>(x, kTwo23 + 8.0f);
    }
  } else if constexpr (WT == RG_MXFP4) {
    // E2M1(code) * 2^(e - 127): exact (low nibbles for the first 16 values
    // of the block, high nibbles for the rest)
    const float sc = e8m0_f32(r.v[0]);
    const int shift = (lane & 2) ? 4 : 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t x = r.v[1 + j] >> shift;
#pragma unroll
      for (int b = 0; b < 4; ++b) w[4 * j + b] = e2m1_f32((x >> (8 * b)) & 15u) * sc;
    }
  } else if constexpr (WT == RG_NVFP4) {
    // E2M1(code) * E4M3(scale): exact
    const float sc = e4m3_f32(r.v[0]);
    const int shift = (lane & 1) ? 4 : 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t x = r.v[1 + j] >> shift;
#pragma unroll
      for (int b = 0; b < 4; ++b) w[4 * j + b] = e2m1_f32((x >> (8 * b)) & 15u) * sc;
    }
  } else if constexpr (WT == RG_Q6_K) {
    // (d * sc) * (q - 32), every step exact
    const int i = (lane >> 2) & 3;
    const float ds = f16_to_f32(static_cast<uint16_t>(r.v[4] & 0xFFFFu)) *
                     static_cast<float>(static_cast<int8_t>((r.v[4] >> 16) & 0xFFu));
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint32_t x = ((r.v[jj] >> (i >= 2 ? 4 : 0)) & 0x0F0F0F0Fu) |
                         (((r.v[2 + jj] >> (2 * i)) & 0x03030303u) << 4);
      w[4 * jj + 0] = ds * byte_minus<0>(x, kTwo23 + 32.0f);
      w[4 * jj + 1] = ds * byte_minus<1>(x, kTwo23 + 32.0f);
      w[4 * jj + 2] = ds * byte_minus<2>(x, kTwo23 + 32.0f);
      w[4 * jj + 3] = ds * byte_minus<3>(x, kTwo23 + 32.0f);
    }
  } else if constexpr (WT == RG_Q2_K) {
    // (d * sc) * q exact, minus dmin * m: one rounding, like the definition
    const int j = (lane >> 2) & 3;
    const float ds = f16_to_f32(static_cast<uint16_t>(r.v[2] & 0xFFFFu)) * static_cast<float>(r.v[3] & 15u);
    const float ndm = -(f16_to_f32(static_cast<uint16_t>(r.v[2] >> 16)) * static_cast<float>(r.v[3] >> 4));
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint32_t x = (r.v[jj] >> (2 * j)) & 0x03030303u;
      w[4 * jj + 0] = fmaf(ds, byte_minus<0>(x, kTwo23), ndm);
      w[4 * jj + 1] = fmaf(ds, byte_minus<1>(x, kTwo23), ndm);
      w[4 * jj + 2] = fmaf(ds, byte_minus<2>(x, kTwo23), ndm);
      w[4 * jj + 3] = fmaf(ds, byte_minus<3>(x, kTwo23), ndm);
    }
  } else if constexpr (WT == RG_Q3_K) {
    // q + 4 = low bits | third bit << 2; (d * (sc - 32)) * q, all exact
    const int h = lane >> 4, j = (lane >> 2) & 3, sb = (lane >> 1) & 1;
    const int si = 8 * h + 2 * j + sb;
    const uint32_t lob = (r.v[4] >> 16) & 0xFFu, hib = r.v[4] >> 24;
    const int sc = static_cast<int>(((si < 8 ? lob : lob >> 4) & 15u) | (((hib >> (2 * (si >> 2))) & 3u) << 4)) - 32;
    const float ds = f16_to_f32(static_cast<uint16_t>(r.v[4] & 0xFFFFu)) * static_cast<float>(sc);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint32_t x = ((r.v[jj] >> (2 * j)) & 0x03030303u) |
                         (((r.v[2 + jj] >> (4 * h + j)) & 0x01010101u) << 2);
      w[4 * jj + 0] = ds * byte_minus<0>(x, kTwo23 + 4.0f);
      w[4 * jj + 1] = ds * byte_minus<1>(x, kTwo23 + 4.0f);
      w[4 * jj + 2] = ds * byte_minus<2>(x, kTwo23 + 4.0f);
      w[4 * jj + 3] = ds * byte_minus<3>(x, kTwo23 + 4.0f);
    }
  } else if constexpr (WT == RG_Q4_1 || WT == RG_Q5_0 || WT == RG_Q5_1) {
    // values 8(lane & 3) .. +7 of block lane >> 2: nibbles (low for the
    // first 16 values of the block, high for the rest) and the fifth bits
    constexpr int Q0 = WT == RG_Q4_1 ? 1 : 2;
    const float d = f16_to_f32(static_cast<uint16_t>(r.v[0] & 0xFFFFu));
    const float m = WT == RG_Q5_0 ? 0.0f : f16_to_f32(static_cast<uint16_t>(r.v[0] >> 16));
    const int j0 = 8 * (lane & 3);
    const int shift = j0 >= 16 ? 4 : 0;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      uint32_t x = (r.v[Q0 + jj] >> shift) & 0x0F0F0F0Fu;
      if constexpr (WT != RG_Q4_1) x |= fifth_bits4(r.v[1] >> (j0 + 4 * jj));
      if constexpr (WT == RG_Q5_0) {
        w[4 * jj + 0] = d * byte_minus<0>(x, kTwo23 + 16.0f);
        w[4 * jj + 1] = d * byte_minus<1>(x, kTwo23 + 16.0f);
        w[4 * jj + 2] = d * byte_minus<2>(x, kTwo23 + 16.0f);
        w[4 * jj + 3] = d * byte_minus<3>(x, kTwo23 + 16.0f);
      } else {  // exact product, one rounding of the sum
        w[4 * jj + 0] = fmaf(d, byte_minus<0>(x, kTwo23), m);
        w[4 * jj + 1] = fmaf(d, byte_minus<1>(x, kTwo23), m);
        w[4 * jj + 2] = fmaf(d, byte_minus<2>(x, kTwo23), m);
        w[4 * jj + 3] = fmaf(d, byte_minus<3>(x, kTwo23), m);
      }
    }
  } else {
    const float d = f16_to_f32(static_cast<uint16_t>(r.v[0] & 0xFFFFu));
    const float dmin = f16_to_f32(static_cast<uint16_t>(r.v[0] >> 16));
    const int c = lane >> 3, half = (lane >> 2) & 1;
    const int j = 2 * c + half;  // sub-block
    const uint32_t* S = &r.v[1];
    int sc, m;
    if (j < 4) {
      sc = byte_at(S, j) & 63;
      m = byte_at(S, j + 4) & 63;
    } else {
      sc = (byte_at(S, j + 4) & 15) | ((byte_at(S, j - 4) >> 6) << 4);
      m = (byte_at(S, j + 4) >> 4) | ((byte_at(S, j) >> 6) << 4);
    }
    // (d * sc) * q - dmin * m: the product is exact (at most 21 bits), so the
    // fused form rounds once, like the definition
    const float ds = d * static_cast<float>(sc);
    const float ndm = -(dmin * static_cast<float>(m));
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      uint32_t x = (r.v[4 + jj] >> (4 * half)) & 0x0F0F0F0Fu;
      if constexpr (WT == RG_Q5_K) x |= ((r.v[6 + jj] >> j) & 0x01010101u) << 4;
      w[4 * jj + 0] = fmaf(ds, byte_minus<0>(x, kTwo23), ndm);
      w[4 * jj + 1] = fmaf(ds, byte_minus<1>(x, kTwo23), ndm);
      w[4 * jj + 2] = fmaf(ds, byte_minus<2>(x, kTwo23), ndm);
      w[4 * jj + 3] = fmaf(ds, byte_minus<3>(x, kTwo23), ndm);
    }
  }
}

// Bytes of one row's 256-value tile.
template <int WT>
__host__ __device__ constexpr int tile_bytes();

// Tiles that are not a multiple of 16 bytes (the super-blocks of Q6_K 210,
// Q3_K 110, Q2_K 84; eight MXFP4 blocks, 136) start at an even offset of a
// 16-byte grain: a stage row holds a window from the grain before
// (window_offset bytes in), 16-byte multiple wide.
template <int WT>
__host__ __device__ constexpr bool windowed() {
  return WT == RG_Q6_K || WT == RG_Q3_K || WT == RG_Q2_K || WT == RG_MXFP4;
}
// Bytes a stage holds per row: the 256-value tile, or its window.
template <int WT>
__host__ __device__ constexpr int stage_row_bytes() {
  return WT == RG_Q6_K ? 224 : WT == RG_Q3_K ? 128 : WT == RG_Q2_K ? 96 : WT == RG_MXFP4 ? 144
                                                                                            : tile_bytes<WT>();
}
template <int WT>
__host__ __device__ constexpr int64_t window_start(int64_t kt) {
  return windowed<WT>() ? ((kt * tile_bytes<WT>()) & ~int64_t{15}) : kt * tile_bytes<WT>();
}
template <int WT>
__host__ __device__ constexpr int window_offset(int64_t kt) {
  return windowed<WT>() ? static_cast<int>((kt * tile_bytes<WT>()) & 15) : 0;
}

template <int WT>
__host__ __device__ constexpr int tile_bytes() {
  return (256 / block_values(WT)) * block_bytes(WT);
}

// The row-per-lane consumers (quantized W, one or two rows of dY) take 64
// rows per stage (two per lane) in a 4-deep ring; the row-per-warp consumers
// 32 rows in an 8-deep ring (4-deep for F32 W, whose rows are four times
// wider than the quantized ones).
// Q4_K and Q8_0 at up to eight rows of dY go through the warp-level MMA
// consumer (consume_mma), also with 64-row stages in a 4-deep ring.
template <int WT, int TB>
constexpr bool mma_path() { return WT == RG_Q4_K || WT == RG_Q8_0; }
template <int WT, int TB>
constexpr bool rows_path() {
  // (NVFP4's 16-value scales do not fit the block-per-warp layout: it takes
  // the eight-values-a-lane consumer)
  return TB <= 2 && is_quant(WT) && !windowed<WT>() && !mma_path<WT, TB>() && WT != RG_NVFP4;
}
template <int WT, int TB>
constexpr int stage_rows() { return rows_path<WT, TB>() || mma_path<WT, TB>() ? 64 : 32; }
template <int WT, int TB>
constexpr int n_stages() {
  return rows_path<WT, TB>() || mma_path<WT, TB>() || WT == RG_F32 ? 4 : 8;
}
constexpr int CONSUMERS = 8; // consumer warps; warp 8 is the TMA producer
constexpr int MAX_ROWS = 512;

// Where a CTA's sums go: partial sums p[(split * T + t) * ld + k] for the
// reduction kernel (beta 0), or, when one CTA holds all N rows, dX itself
// (ld = dX's row stride) with beta * dX added.
struct SmtOut {
  float* p;
  int64_t ld;
  float beta;
};
__device__ __forceinline__ void smt_store(const SmtOut& o, int split, int T, int t, int k, float v) {
  float* q = o.p + (static_cast<int64_t>(split) * T + t) * o.ld + k;
  if (o.beta != 0.0f) v = fmaf(o.beta, *q, v);
  *q = v;
}

// Shared memory after the staged dY slice: the MMA consumer's scaled dY
// table (two stage buffers of [sub-block][dY row][64 rows + 16 pad] fp16,
// rows in fragment order, see table_pos),
// its min-term partials [warp][4][2][TB] and the per-row maxima [8]; the
// row-per-warp consumers' reduction buffer [4][TB][256].
constexpr int YDS_STRIDE = 80;  // 40 words: lines 8 banks apart
template <int TB>
constexpr int yds_elems() { return 2 * 8 * TB * YDS_STRIDE; }
template <int WT, int TB>
constexpr int aux_bytes() {
  return rows_path<WT, TB>() ? 0
         : mma_path<WT, TB>() ? 2 * yds_elems<TB>() + 4 * (CONSUMERS * 4 * 2 * TB) + 4 * 8
                              : 4 * 4 * TB * 256;
}

// --- one and two rows of dY: a block per warp, a row per lane ---------------
// Warp g of the eight consumers owns block g of every row's 256-value tile
// (the g-th Q8_0 or Q4_0 block, the g-th Q4_K sub-block, values 32g .. 32g+31
// of F16/BF16) and lane l takes row l of each 32-row stage.  Every offset
// inside a row is then a compile-time constant: the block's bytes come out
// of 16-byte shared loads with constant shifts, its scale is folded into dY
// once per row (F32 products; the acceptance bound covers the reassociation),
// and a value costs one byte permute plus half a packed F32 add and half a
// packed F32 fused multiply-add per row of dY.  The 32 lanes' partial sums of
// the block's 32 values are combined by a fixed butterfly at the end.

typedef unsigned long long f32x2;  // two F32 values in one 64-bit register
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Two bytes (B, B+1) of x as the F32 pair (u - bias, u' - bias), exactly.
template <int B>
__device__ __forceinline__ f32x2 bytes2(uint32_t x, f32x2 neg_two23_bias) {
  return add2(pack2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u | B)),
                    __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u | (B + 1)))),
              neg_two23_bias);
}

// Add one row's block g (its 32 values times each dY row) into acc; Q4_K's
// min term goes to msum, subtracted once at the end.  g is the warp's index,
// uniform over the warp: one code path serves all eight warps.
template <int WT, int TB>
__device__ __forceinline__ void row_block(const uint8_t* row, int g, const float (&y)[TB],
                                          f32x2 (&acc)[TB][16], float (&msum)[TB]) {
  static_assert(is_quant(WT), "quantized types only");
  if constexpr (WT == RG_Q8_0 || WT == RG_Q4_0) {
    // the block starts at byte X = g * (34 or 18), an even offset: read the
    // aligned words around it; off2 = the block starts 2 bytes into a word
    constexpr int BB = WT == RG_Q8_0 ? 34 : 18, NQ = WT == RG_Q8_0 ? 8 : 4;
    const int X = BB * g;
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + (X & ~3));
    const bool off2 = (X & 2) != 0;
    uint32_t w[NQ + 1];
#pragma unroll
    for (int i = 0; i <= NQ; ++i) w[i] = wp[i];
    const float d = f16_to_f32(static_cast<uint16_t>(off2 ? (w[0] >> 16) : (w[0] & 0xFFFFu)));
    // quant word j = the 4 bytes at X + 2 + 4j
    uint32_t q[NQ];
#pragma unroll
    for (int j = 0; j < NQ; ++j) q[j] = off2 ? w[j + 1] : __funnelshift_r(w[j], w[j + 1], 16);
    f32x2 yd[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) yd[t] = pack2(y[t] * d, y[t] * d);
    if constexpr (WT == RG_Q8_0) {
      const f32x2 nb = pack2(-(kTwo23 + 128.0f), -(kTwo23 + 128.0f));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t x = q[j] ^ 0x80808080u;  // int8 q -> byte q + 128
        const f32x2 q01 = bytes2<0>(x, nb), q23 = bytes2<2>(x, nb);
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          acc[t][2 * j] = fma2(yd[t], q01, acc[t][2 * j]);
          acc[t][2 * j + 1] = fma2(yd[t], q23, acc[t][2 * j + 1]);
        }
      }
    } else {
      const f32x2 nb = pack2(-(kTwo23 + 8.0f), -(kTwo23 + 8.0f));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = q[j] & 0x0F0F0F0Fu, hi = (q[j] >> 4) & 0x0F0F0F0Fu;  // values 4j.., 16+4j..
        const f32x2 l01 = bytes2<0>(lo, nb), l23 = bytes2<2>(lo, nb);
        const f32x2 h01 = bytes2<0>(hi, nb), h23 = bytes2<2>(hi, nb);
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          acc[t][2 * j] = fma2(yd[t], l01, acc[t][2 * j]);
          acc[t][2 * j + 1] = fma2(yd[t], l23, acc[t][2 * j + 1]);
          acc[t][8 + 2 * j] = fma2(yd[t], h01, acc[t][8 + 2 * j]);
          acc[t][9 + 2 * j] = fma2(yd[t], h23, acc[t][9 + 2 * j]);
        }
      }
    }
  } else if constexpr (WT == RG_Q4_1 || WT == RG_Q5_0 || WT == RG_Q5_1) {
    // block g at byte X = g * (20, 22 or 24): d (and m), qh (Q5), 16 bytes
    // of nibbles.  Q5_0's X is even only: off2 = it starts 2 bytes into a word.
    constexpr int BB = block_bytes(WT);
    const int X = BB * g;
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + (X & ~3));
    const bool off2 = WT == RG_Q5_0 && (X & 2) != 0;
    constexpr int NW = WT == RG_Q4_1 ? 5 : 6;
    uint32_t w[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = wp[i];
    float d, m = 0.0f;
    uint32_t qh = 0, q[4];
    if constexpr (WT == RG_Q5_0) {
      d = f16_to_f32(static_cast<uint16_t>(off2 ? (w[0] >> 16) : (w[0] & 0xFFFFu)));
      qh = off2 ? w[1] : __funnelshift_r(w[0], w[1], 16);
#pragma unroll
      for (int j = 0; j < 4; ++j) q[j] = off2 ? w[2 + j] : __funnelshift_r(w[1 + j], w[2 + j], 16);
    } else {
      d = f16_to_f32(static_cast<uint16_t>(w[0] & 0xFFFFu));
      m = f16_to_f32(static_cast<uint16_t>(w[0] >> 16));
      constexpr int Q0 = WT == RG_Q4_1 ? 1 : 2;
      if constexpr (WT == RG_Q5_1) qh = w[1];
#pragma unroll
      for (int j = 0; j < 4; ++j) q[j] = w[Q0 + j];
    }
    // y * (d*q + m) = (y*d)*q + y*m; the y*m terms go to msum (subtracted, so negated)
    f32x2 yd[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      yd[t] = pack2(y[t] * d, y[t] * d);
      if constexpr (WT != RG_Q5_0) msum[t] = fmaf(y[t], -m, msum[t]);
    }
    const float bias = WT == RG_Q5_0 ? 16.0f : 0.0f;
    const f32x2 nb = pack2(-(kTwo23 + bias), -(kTwo23 + bias));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t lo = q[j] & 0x0F0F0F0Fu, hi = (q[j] >> 4) & 0x0F0F0F0Fu;  // values 4j.., 16+4j..
      if constexpr (WT != RG_Q4_1) {
        lo |= fifth_bits4(qh >> (4 * j));
        hi |= fifth_bits4(qh >> (16 + 4 * j));
      }
      const f32x2 l01 = bytes2<0>(lo, nb), l23 = bytes2<2>(lo, nb);
      const f32x2 h01 = bytes2<0>(hi, nb), h23 = bytes2<2>(hi, nb);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        acc[t][2 * j] = fma2(yd[t], l01, acc[t][2 * j]);
        acc[t][2 * j + 1] = fma2(yd[t], l23, acc[t][2 * j + 1]);
        acc[t][8 + 2 * j] = fma2(yd[t], h01, acc[t][8 + 2 * j]);
        acc[t][9 + 2 * j] = fma2(yd[t], h23, acc[t][9 + 2 * j]);
      }
    }
  } else {
    // sub-block g = 2c + h: nibble h of bytes 32c .. 32c+31 of the quants
    // (Q5_K: plus bit g of qh[l] as the fifth bit)
    constexpr int QS = WT == RG_Q5_K ? 48 : 16;
    const int c = g >> 1, h = g & 1;
    const uint4 hd = *reinterpret_cast<const uint4*>(row);
    const uint4 qa = *reinterpret_cast<const uint4*>(row + QS + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(row + QS + 16 + 32 * c);
    uint32_t hw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if constexpr (WT == RG_Q5_K) {
      const uint4 ha = *reinterpret_cast<const uint4*>(row + 16);
      const uint4 hb2 = *reinterpret_cast<const uint4*>(row + 32);
      hw[0] = ha.x; hw[1] = ha.y; hw[2] = ha.z; hw[3] = ha.w;
      hw[4] = hb2.x; hw[5] = hb2.y; hw[6] = hb2.z; hw[7] = hb2.w;
    }
    const float d = f16_to_f32(static_cast<uint16_t>(hd.x & 0xFFFFu));
    const float dmin = f16_to_f32(static_cast<uint16_t>(hd.x >> 16));
    // the 6-bit scale and min of sub-block g from header bytes 4..15
    auto hb = [&](int i) {
      const uint32_t wd = i < 4 ? hd.y : (i < 8 ? hd.z : hd.w);
      return (wd >> (8 * (i & 3))) & 0xFFu;
    };
    uint32_t sc, m;
    if (g < 4) {
      sc = hb(g) & 63u;
      m = hb(g + 4) & 63u;
    } else {
      sc = (hb(g + 4) & 15u) | ((hb(g - 4) >> 6) << 4);
      m = (hb(g + 4) >> 4) | ((hb(g) >> 6) << 4);
    }
    const float ds = d * static_cast<float>(sc), dm = dmin * static_cast<float>(m);
    const f32x2 nb = pack2(-kTwo23, -kTwo23);
    f32x2 yd[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      yd[t] = pack2(y[t] * ds, y[t] * ds);
      msum[t] = fmaf(y[t], dm, msum[t]);
    }
    const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t x = (qw[j] >> (4 * h)) & 0x0F0F0F0Fu;
      if constexpr (WT == RG_Q5_K) x |= ((hw[j] >> g) & 0x01010101u) << 4;
      const f32x2 q01 = bytes2<0>(x, nb), q23 = bytes2<2>(x, nb);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        acc[t][2 * j] = fma2(yd[t], q01, acc[t][2 * j]);
        acc[t][2 * j + 1] = fma2(yd[t], q23, acc[t][2 * j + 1]);
      }
    }
  }
}

// The consumer warp of block g: every stage's rows (row = lane, then lane +
// 32), then the butterfly over lanes and the block's partial sums to part.
template <int WT, int TB, int TBYTES, int BR, int STAGES_>
__device__ __forceinline__ void consume_rows(int g, const uint8_t* stage_buf, const float* ys,
                                             uint32_t bar0,
                                             int n_tiles, int nrows, int lane, int kt, int K,
                                             int t0, int T, int split, SmtOut out, WaitCtl ctl,
                                             volatile int* abort_flag) {
  f32x2 acc[TB][16];
  float msum[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    msum[t] = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[t][i] = 0ull;  // (+0.0f, +0.0f)
  }
  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % STAGES_;
    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * s, static_cast<uint32_t>(i / STAGES_) & 1u,
                                           ctl, abort_flag)))
      break;
#pragma unroll 1
    for (int u = 0; u < BR / 32; ++u) {
      const int r = i * BR + 32 * u + lane;  // this lane's rows within the CTA's slice
      if (r < nrows) {
        float y[TB];
#pragma unroll
        for (int t = 0; t < TB; ++t) y[t] = ys[t * MAX_ROWS + r];
        row_block<WT, TB>(stage_buf + (s * BR + 32 * u + lane) * TBYTES, g, y, acc, msum);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar0 + 8u * (STAGES_ + s));
  }
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      unpack2(acc[t][i], v[2 * i], v[2 * i + 1]);
      if constexpr (WT != RG_Q8_0 && WT != RG_Q4_0 && WT != RG_Q5_0) {
        v[2 * i] -= msum[t];
        v[2 * i + 1] -= msum[t];
      }
    }
    // reduce-scatter over the 32 lanes: afterwards lane l holds value l
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < o; ++j) {
        const float send = up ? v[j] : v[j + o];
        const float keep = up ? v[j + o] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    const int gt = t0 + t, gk = kt * 256 + 32 * g + lane;
    if (gt < T && gk < K) smt_store(out, split, T, gt, gk, v[0]);
  }
}

// --- Q4_K, one to eight rows of dY: the warp-level tensor-core MMA ---------
// mma.m16n8k16 computes D[k][t] += sum over 16 rows n of A[k][n] * B[n][t]
// with A = the nibbles q of W (a 32-bit register holds the fp16 values of
// rows n and n + 1 in one column k) and B = fp16(y * 2^s * d * sc), the dY row t times the
// sub-block's scale; the min term sum_n y * dmin * m stays in F32.
//  * A nibble q in the low bits of an fp16 is the subnormal q * 2^-24,
//    exactly; a high nibble left in place is 16q * 2^-24.  So the operand
//    pair of two rows costs one byte permute (one byte of each row) and one
//    AND per nibble, 0.75 integer instructions a value, against about 2.5
//    for an F32 value; the MMA takes the multiply-adds off the FMA pipe.
//  * 2^s puts max|y| of the CTA's slice in [2, 4), so the largest row's
//    y * d * sc stays in fp16's range wherever d * sc * q does (the
//    tensor-core variant's precondition); the result is scaled back exactly.
//    Rows whose |y| lies many octaves below the slice's maximum give fp16
//    subnormal operands and keep fewer significant bits: a term q * y * d * sc
//    then carries an absolute error up to q * 2^-25 * 2^-s, which the
//    bound's sum of |y| |deq W| covers through the slice's large rows.
//  * Warp w owns the 32 columns k = 64 (w >> 1) + 32 h + 4 g + 2 (w & 1) + j
//    (g = 0..7, h, j = 0, 1): bytes 2 (w & 1) and 2 (w & 1) + 1 of word g
//    of the 64-value chunk w >> 1, both nibbles, i.e. two accumulator tiles.
//  * Per stage, the CTA first decodes each row's eight scales and mins
//    (thread 4r + q: sub-blocks q and q + 4 of stage row r) into the fp16
//    table B is loaded from, then every warp runs its MMAs over the 64 rows.
//
// Q8_0 takes the same path with its eight 32-value blocks in place of the
// sub-blocks: B = fp16(y * 2^s * d) per (row, block), no min term, and A the
// int8 values as fp16 integers (1024 + 128 + q from one XOR into the
// exponent bits, less 1152 in one packed subtraction: exact for every q, so
// the only rounding before the F32 sums is B's).  Warp w owns block w.

// D += A * B for one m16n8k16 tile (fp16 operands, F32 accumulation).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^s of dY row t from the bits of the slice's max|y| (clamped to F32's
// normal powers; zero rows get 2^127, whose products are still zero), and
// 2^-s, exactly (2^-127 is the subnormal 1 << 22).
__device__ __forceinline__ int row_scale_exp(int max_bits) {
  return min(max(255 - ((max_bits >> 23) & 255), 1), 254);
}
__device__ __forceinline__ float row_scale(int max_bits) {
  return __int_as_float(row_scale_exp(max_bits) << 23);
}
__device__ __forceinline__ float row_unscale(int max_bits) {
  const int fe = row_scale_exp(max_bits);
  return __int_as_float(fe < 254 ? (254 - fe) << 23 : 1 << 22);
}
// Position of stage row r in its 16-row group of the scaled dY table: rows
// 2c, 2c + 1, 2c + 8, 2c + 9 at 4c .. 4c + 3, so that fragment thread c loads
// both of its B registers with one 8-byte read.
__device__ __forceinline__ int table_pos(int r) {
  return (r & ~15) | (4 * ((r & 7) >> 1) + (r & 1) + 2 * ((r >> 3) & 1));
}

// Named barrier 1 over the consumer warps that also returns, to every one of
// them, whether any thread passed `any` true: a decision they all share (the
// producer may set the abort flag between two warps' own reads of it).
__device__ __forceinline__ bool consumers_sync_any(bool any) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(any)), "n"(THREADS)
      : "memory");
  return r != 0;
}

// Q8_0's int8 q into the fp16 pair of one operand register: x holds byte q
// of row n in bits 0..7 and of row n + 1 in bits 16..23 (other bits zero);
// 0x6400 | (q ^ 0x80) is the fp16 value 1024 + 128 + q, exactly, and one
// packed subtraction of 1152 leaves q.
__device__ __forceinline__ uint32_t q8_pair(uint32_t x) {
  const uint32_t biased = x ^ 0x64806480u;
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x64806480u));
  return r;
}

template <int WT, int TB, int BR, int STAGES_>
__device__ __forceinline__ void consume_mma(int warp, int lane, const uint8_t* stage_buf,
                                            float* ys, uint8_t* aux, uint32_t bar0,
                                            int n_tiles, int nrows, int kt, int K, int t0, int T,
                                            int split, SmtOut out, WaitCtl ctl,
                                            volatile int* abort_flag) {
  static_assert(WT == RG_Q4_K || WT == RG_Q8_0, "the MMA consumer takes Q4_K and Q8_0");
  constexpr bool K4 = WT == RG_Q4_K;
  // Q4_K super-block: d, dmin, 12 scale bytes, 128 nibble bytes; Q8_0: eight
  // blocks of d and 32 int8 values
  constexpr int TBYTES = K4 ? 144 : 272;
  static_assert(BR == 64, "64-row stages: one scale-pass thread per (row, q), four MMA row groups");
  uint16_t* yds = reinterpret_cast<uint16_t*>(aux);
  float* mred = reinterpret_cast<float*>(aux + 2 * yds_elems<TB>());
  int* smax = reinterpret_cast<int*>(mred + CONSUMERS * 4 * 2 * TB);
  const int tid = warp * 32 + lane;

  // the slice's max|y| per dY row (NaN ignored), then y *= 2^s in place
  {
    float mx[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      mx[t] = 0.0f;
      for (int r = tid; r < MAX_ROWS; r += THREADS) mx[t] = fmaxf(mx[t], fabsf(ys[t * MAX_ROWS + r]));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx[t] = fmaxf(mx[t], __shfl_xor_sync(0xffffffffu, mx[t], o));
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < TB; ++t) atomicMax(smax + t, __float_as_int(mx[t]));  // non-negative: int order
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    const float f = row_scale(smax[t]);
    for (int r = tid; r < MAX_ROWS; r += THREADS) ys[t * MAX_ROWS + r] *= f;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");

  const int srow = tid >> 2, q = tid & 3;        // scale pass: sub-blocks q, q + 4 of row srow
  const int c4 = warp >> 1, bp = warp & 1;       // MMA: chunk c4, bytes 2bp and 2bp + 1 of a word
  const int g = lane >> 2, c = lane & 3;         // the fragment's group and thread in group
  // byte b of x into the low half, byte b of y into the high half
  const uint32_t sel0 = static_cast<uint32_t>(2 * bp) * 0x0011u + static_cast<uint32_t>(4 + 2 * bp) * 0x1100u;
  const uint32_t sel1 = sel0 + 0x1111u;
  float acc[2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[h][e] = 0.0f;
  float msum[TB][2];
#pragma unroll
  for (int t = 0; t < TB; ++t) msum[t][0] = msum[t][1] = 0.0f;
  bool aborted = false;  // taken by every consumer warp alike

  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % STAGES_;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8u * s, static_cast<uint32_t>(i / STAGES_) & 1u,
                                                      ctl, abort_flag));
    uint16_t* Y = yds + (i & 1) * (8 * TB * YDS_STRIDE);
    const uint8_t* stage = stage_buf + s * BR * TBYTES;
    if (ok && !K4) {
      // the scales of blocks q and q + 4; a row past the slice (the next
      // slice's, or TMA's zero fill past N) gets zero entries
      const bool live = i * BR + srow < nrows;
      const uint8_t* rowp = stage + srow * TBYTES;
      const float d0 = live ? f16_to_f32(*reinterpret_cast<const uint16_t*>(rowp + 34 * q)) : 0.0f;
      const float d1 = live ? f16_to_f32(*reinterpret_cast<const uint16_t*>(rowp + 34 * (q + 4))) : 0.0f;
      const float* yr = ys + i * BR + srow;
      const int pos = table_pos(srow);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const float y = yr[t * MAX_ROWS];
        Y[(q * TB + t) * YDS_STRIDE + pos] = __half_as_ushort(__float2half_rn(y * d0));
        Y[((q + 4) * TB + t) * YDS_STRIDE + pos] = __half_as_ushort(__float2half_rn(y * d1));
      }
    }
    if (ok && K4) {
      // scales and mins of sub-blocks q and q + 4; a row past the slice (the
      // next slice's, or TMA's zero fill past N) gets zero entries
      const bool live = i * BR + srow < nrows;
      uint4 hd = *reinterpret_cast<const uint4*>(stage + srow * TBYTES);
      if (!live) hd = make_uint4(0u, 0u, 0u, 0u);
      const float d = f16_to_f32(static_cast<uint16_t>(hd.x & 0xFFFFu));
      const float dmin = f16_to_f32(static_cast<uint16_t>(hd.x >> 16));
      const uint32_t b0 = hd.y >> (8 * q), b1 = hd.z >> (8 * q), b2 = hd.w >> (8 * q);
      const float ds0 = d * static_cast<float>(b0 & 63u);
      const float ds1 = d * static_cast<float>((b2 & 15u) | ((b0 >> 2) & 48u));
      const float dm0 = dmin * static_cast<float>(b1 & 63u);
      const float dm1 = dmin * static_cast<float>(((b2 >> 4) & 15u) | ((b1 >> 2) & 48u));
      const float* yr = ys + i * BR + srow;
      const int pos = table_pos(srow);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const float y = yr[t * MAX_ROWS];
        Y[(q * TB + t) * YDS_STRIDE + pos] = __half_as_ushort(__float2half_rn(y * ds0));
        Y[((q + 4) * TB + t) * YDS_STRIDE + pos] = __half_as_ushort(__float2half_rn(y * ds1));
        msum[t][0] = fmaf(y, dm0, msum[t][0]);
        msum[t][1] = fmaf(y, dm1, msum[t][1]);
      }
    }
    // every consumer warp arrives, with or without its stage, and all take
    // the same abort decision
    if (consumers_sync_any(!ok || *abort_flag != 0)) {
      aborted = true;
      break;
    }
    if constexpr (!K4) {
      // warp w: block w; M row g is column 2g + h of the block, M row g + 8
      // column 16 + 2g + h (h: the accumulator tile); 16-bit loads of the
      // byte pairs (the blocks' values sit at even, not 4-byte, offsets)
      const uint8_t* wq = stage + 34 * warp + 2 + 2 * g;
#pragma unroll
      for (int grp = 0; grp < BR / 16; ++grp) {
        const int R = 16 * grp + 2 * c;
        uint32_t x[8];  // rows R, R + 1, R + 8, R + 9, low and high pair each
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint8_t* rp = wq + (R + (r & 1) + 8 * (r >> 1)) * TBYTES;
          x[2 * r] = *reinterpret_cast<const uint16_t*>(rp);
          x[2 * r + 1] = *reinterpret_cast<const uint16_t*>(rp + 16);
        }
        uint2 yv = make_uint2(0u, 0u);  // B: rows R, R + 1 and R + 8, R + 9 at dY row g
        if (g < TB) yv = *reinterpret_cast<const uint2*>(Y + (warp * TB + g) * YDS_STRIDE + 16 * grp + 4 * c);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // byte h of each row's pair into the two halves (bytes 2 and 6: zero)
          const uint32_t sel = h ? 0x6521u : 0x6420u;
          mma_16816(acc[h], q8_pair(__byte_perm(x[0], x[2], sel)), q8_pair(__byte_perm(x[1], x[3], sel)),
                    q8_pair(__byte_perm(x[4], x[6], sel)), q8_pair(__byte_perm(x[5], x[7], sel)), yv.x, yv.y);
        }
      }
    } else {
    const uint8_t* wq = stage + 16 + 32 * c4 + 4 * g;
#pragma unroll
    for (int grp = 0; grp < BR / 16; ++grp) {
      const int R = 16 * grp + 2 * c;  // rows R, R + 1 (k-pair 2c) and R + 8, R + 9 (2c + 8)
      const uint32_t wa = *reinterpret_cast<const uint32_t*>(wq + R * TBYTES);
      const uint32_t wb = *reinterpret_cast<const uint32_t*>(wq + (R + 1) * TBYTES);
      const uint32_t wc = *reinterpret_cast<const uint32_t*>(wq + (R + 8) * TBYTES);
      const uint32_t wd = *reinterpret_cast<const uint32_t*>(wq + (R + 9) * TBYTES);
      const uint32_t p0 = __byte_perm(wa, wb, sel0), p1 = __byte_perm(wa, wb, sel1);
      const uint32_t r0 = __byte_perm(wc, wd, sel0), r1 = __byte_perm(wc, wd, sel1);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t M = h ? 0x00F000F0u : 0x000F000Fu;
        uint2 yv = make_uint2(0u, 0u);  // B: rows R, R + 1 and R + 8, R + 9 at dY row g
        if (g < TB)
          yv = *reinterpret_cast<const uint2*>(Y + ((2 * c4 + h) * TB + g) * YDS_STRIDE + 16 * grp + 4 * c);
        mma_16816(acc[h], p0 & M, p1 & M, r0 & M, r1 & M, yv.x, yv.y);
      }
    }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar0 + 8u * (STAGES_ + s));
  }

  // a wait that gave up: no partial sums reach `out` (all consumer warps
  // leave here together, so the named barriers below stay matched)
  if (aborted) return;
  if constexpr (!K4) {
    // this lane's outputs: dY rows 2c, 2c + 1 at M rows g and g + 8 of both tiles
    const float inv0 = 2 * c < TB ? row_unscale(smax[2 * c]) : 0.0f;
    const float inv1 = 2 * c + 1 < TB ? row_unscale(smax[2 * c + 1]) : 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = 2 * c + (e & 1);
        const int gk = kt * 256 + 32 * warp + 16 * (e >> 1) + 2 * g + h;
        if (t < TB && t0 + t < T && gk < K)
          smt_store(out, split, T, t0 + t, gk, acc[h][e] * ((e & 1) ? inv1 : inv0));
      }
    return;
  } else {
  // the min terms of each sub-block over the slice's rows, in a fixed order:
  // lanes of one q (xor 4, 8, 16), then the eight warps
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int o = 4; o <= 16; o <<= 1) msum[t][jj] += __shfl_xor_sync(0xffffffffu, msum[t][jj], o);
  if (lane < 4) {
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) mred[((warp * 4 + lane) * 2 + jj) * TB + t] = msum[t][jj];
  }
  asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
  // one thread per (sub-block j, dY row t) adds the eight warps in order
  // (the table's space is free now)
  float* mtot = reinterpret_cast<float*>(aux);
  if (tid < 8 * TB) {
    const int j = tid / TB, t = tid - j * TB;  // sub-block j: scale-pass thread q = j & 3, slot j >> 2
    float m = 0.0f;
#pragma unroll
    for (int w = 0; w < CONSUMERS; ++w) m += mred[((w * 4 + (j & 3)) * 2 + (j >> 2)) * TB + t];
    mtot[j * TB + t] = m;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
  // this lane's outputs: dY rows 2c, 2c + 1 at columns k and k + 1 of each tile
  const float inv0 = 2 * c < TB ? row_unscale(smax[2 * c]) : 0.0f;
  const float inv1 = 2 * c + 1 < TB ? row_unscale(smax[2 * c + 1]) : 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = 2 * c4 + h;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 2 * c + (e & 1);
      const int gk = kt * 256 + 64 * c4 + 32 * h + 4 * g + 2 * bp + (e >> 1);
      if (t < TB && t0 + t < T && gk < K) {
        const float v = (acc[h][e] * (h ? 1048576.0f : 16777216.0f) - mtot[j * TB + t]) *  // 2^20, 2^24
                        ((e & 1) ? inv1 : inv0);
        smt_store(out, split, T, t0 + t, gk, v);
      }
    }
  }
  }
}

// grid (ceil(K/256), n_splits, ceil(T/TB)); the sums over rows
// [split * rows_per_split, +rows_per_split) to `out` (partial sums, or dX).
// A producer warp streams the CTA's rows of W, tile by tile of BR rows, into
// an 8-stage ring with TMA; eight consumer warps decode from shared memory.
template <int WT, int TB>
__global__ void __launch_bounds__(THREADS + 32, mma_path<WT, TB>() ? (TB <= 4 ? 3 : 2)
                                                : rows_path<WT, TB>() && TB == 1 ? 3
                                                : TB >= 8                        ? 1
                                                                                 : 2)
    smallt_kernel(const __grid_constant__ CUtensorMap map_w, int N, int K,
                  const float* __restrict__ dY, int64_t dy_t, int64_t dy_n, int T,
                  SmtOut out, int rows_per_split, WaitCtl ctl, int inject_stall) {
  constexpr int TBYTES = stage_row_bytes<WT>();
  constexpr int BR = stage_rows<WT, TB>(), STAGES = n_stages<WT, TB>();
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* stage_buf = sm;                                              // STAGES x BR x TBYTES
  float* ys = reinterpret_cast<float*>(sm + STAGES * BR * TBYTES);      // [TB][MAX_ROWS]
  float* red = ys + TB * MAX_ROWS;                                      // aux_bytes<WT, TB>()
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) +
                                               aux_bytes<WT, TB>());    // full[S], empty[S]
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;
  // the reduction kernel after this one may be scheduled now (it waits for
  // this grid to complete before reading the partial sums)
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, split = blockIdx.y;
  const int t0 = blockIdx.z * TB;
  const int nbeg = split * rows_per_split;
  const int nrows = max(0, min(N, nbeg + rows_per_split) - nbeg);
  const int n_tiles = (nrows + BR - 1) / BR;
  const uint32_t bar0 = smem_addr(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };

  // the producer's lane initialises the ring and starts its first copies
  // before the block-wide barrier (fresh slots need no wait)
  const bool producer = threadIdx.x == THREADS;
  uint32_t pend = 0;                         // slots with a copy started
  const int n_pre = min(STAGES, n_tiles);
  if (producer) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), CONSUMERS);
    }
    abort_flag_s = 0;
    if constexpr (mma_path<WT, TB>()) {
      int* smax = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(red) + aux_bytes<WT, TB>() - 32);
      for (int t = 0; t < 8; ++t) smax[t] = 0;
    }
    fence_mbar_init();
    for (int i = 0; i < n_pre; ++i) {
      if (i == 0 && inject_stall != 0) continue;  // fault injection: the first stage never fills
      mbar_arrive_expect_tx(full(i), BR * TBYTES);
      tma_load_2d(smem_addr(stage_buf + i * BR * TBYTES), &map_w, full(i),
                  static_cast<int>(window_start<WT>(kt) / 4), nbeg + i * BR);
      pend |= 1u << i;
    }
  }
  if (warp < CONSUMERS) {
    // this CTA's slice of dY, [TB][nrows], staged by the consumers while the
    // producer sets up the ring and starts its first copies
    for (int idx = threadIdx.x; idx < TB * MAX_ROWS; idx += THREADS) {
      const int t = idx / MAX_ROWS, r = idx - t * MAX_ROWS;
      ys[idx] = (t0 + t < T && r < nrows)
                    ? __ldg(dY + static_cast<int64_t>(t0 + t) * dy_t + static_cast<int64_t>(nbeg + r) * dy_n)
                    : 0.0f;
    }
  }
  __syncthreads();  // the ring's barriers and the staged slice of dY

  if (warp == CONSUMERS) {
    // ---------------- producer ----------------
    if (lane == 0) {
      // the copies after the first STAGES (which started before the barrier,
      // phase 0), each into a slot its consumers have released
      uint32_t ph = n_pre == STAGES ? 1u : 0u, pend_ph = 0;  // the phase of each started copy
      for (int i = n_pre; i < n_tiles; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(empty(s), ph ^ 1u, ctl, abort_flag)) break;
        mbar_arrive_expect_tx(full(s), BR * TBYTES);
        tma_load_2d(smem_addr(stage_buf + s * BR * TBYTES), &map_w, full(s),
                    static_cast<int>(window_start<WT>(kt) / 4), nbeg + i * BR);
        pend |= 1u << s;
        pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
        if (s == STAGES - 1) ph ^= 1u;
      }
      // drain: every copy started lands before the CTA leaves (a consumed
      // one's phase is past, and its wait returns at once)
      volatile int no_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if (pend & (1u << s)) (void)mbar_wait(full(s), (pend_ph >> s) & 1u, ctl, &no_abort);
    }
    __syncwarp();
  }

  if constexpr (mma_path<WT, TB>()) {
    if (warp < CONSUMERS)
      consume_mma<WT, TB, BR, STAGES>(warp, lane, stage_buf, ys, reinterpret_cast<uint8_t*>(red), bar0,
                                      n_tiles, nrows, kt, K, t0, T, split, out, ctl, abort_flag);
    return;
  } else if constexpr (rows_path<WT, TB>()) {
    // quantized, one and two rows of dY: a block per warp, a row per lane
    if (warp < CONSUMERS)
      consume_rows<WT, TB, TBYTES, BR, STAGES>(warp, stage_buf, ys, bar0, n_tiles, nrows, lane, kt,
                                               K, t0, T, split, out, ctl, abort_flag);
    return;
  } else {
  float acc[TB][8];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[t][i] = 0.0f;

  if (warp < CONSUMERS) {
    const bool kvalid = kt * 256 + 8 * lane < K;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(full(s), static_cast<uint32_t>(i / STAGES) & 1u, ctl,
                                             abort_flag)))
        break;
      if (kvalid) {
        const uint8_t* tile = stage_buf + s * BR * TBYTES + window_offset<WT>(kt);
        Raw<WT> raw[BR / CONSUMERS];
#pragma unroll
        for (int u = 0; u < BR / CONSUMERS; ++u) load_raw_smem<WT>(tile + (warp + CONSUMERS * u) * TBYTES, lane, raw[u]);
#pragma unroll
        for (int u = 0; u < BR / CONSUMERS; ++u) {
          const int r = i * BR + warp + CONSUMERS * u;  // row within the CTA's slice
          if (r < nrows) {
            float w[8];
            decode_raw<WT>(raw[u], lane, w);
#pragma unroll
            for (int t = 0; t < TB; ++t) {
              const float y = ys[t * MAX_ROWS + r];
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[t][q] = fmaf(y, w[q], acc[t][q]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));
    }
  }

  // the CTA's eight consumer warps, summed in a fixed order: (w + 4) into w, then 0..3
  if (warp >= 4 && warp < CONSUMERS) {
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int q = 0; q < 8; ++q) red[((warp - 4) * TB + t) * 256 + 8 * lane + q] = acc[t][q];
  }
  __syncthreads();
  if (warp < 4) {
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int q = 0; q < 8; ++q) red[(warp * TB + t) * 256 + 8 * lane + q] += acc[t][q];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < TB * 256; idx += THREADS + 32) {
    const int t = idx >> 8, kk = idx & 255;
    const int gt = t0 + t, gk = kt * 256 + kk;
    if (gt < T && gk < K) {
      const float sum = ((red[(0 * TB + t) * 256 + kk] + red[(1 * TB + t) * 256 + kk]) +
                         red[(2 * TB + t) * 256 + kk]) + red[(3 * TB + t) * 256 + kk];
      smt_store(out, split, T, gt, gk, sum);
    }
  }
  }
}

template <int WT, int TB>
constexpr size_t smem_bytes() {
  return static_cast<size_t>(n_stages<WT, TB>()) * stage_rows<WT, TB>() * stage_row_bytes<WT>() +
         sizeof(float) * TB * MAX_ROWS + aux_bytes<WT, TB>() + 16 * n_stages<WT, TB>();
}

// --- the forward at a few rows of X -----------------------------------------
// Y[t, n] = beta * Y[t, n] + sum_k X[t, k] * deq(W)[n, k], up to four rows
// of X a pass (rg_mul_mat's route for one or two rows): every weight value
// is read once a pass, so the call streams W like the small-T OUT_PROD,
// with the roles of the two axes swapped.  A CTA owns a
// block of rows (8, 16 or 32) along the whole of K: a producer warp copies,
// tile by tile, the block's 256-value tiles (or their 16-byte windows) into
// a ring; consumer warp w takes rows w, w + 8, ... of the block, each lane
// decodes its 8 values of a row exactly to F32 and multiplies them with its
// 8 values of each row of X, and the 32 lanes' partial sums of a row meet in
// a fixed butterfly at the end: no partial sums in memory, no second kernel
// and no 16-bit copy of X.
template <int WT>
constexpr int fwd_rows() { return WT == RG_F32 ? 16 : 32; }
template <int WT>
constexpr int fwd_stages() {
  return stage_row_bytes<WT>() * fwd_rows<WT>() * 8 <= 72 * 1024 ? 8 : 4;
}
template <int WT>
constexpr size_t fwd_smem_bytes() {
  return static_cast<size_t>(fwd_stages<WT>()) * fwd_rows<WT>() * stage_row_bytes<WT>() + 16 * fwd_stages<WT>();
}

// grid (ceil(N / rows), ceil(T / TB)); rows = the tensor map's box height
// (8, 16 or 32, at most fwd_rows<WT>()), a multiple of 8.
template <int WT, int TB>
__global__ void __launch_bounds__(THREADS + 32, 3)
    smallt_fwd_kernel(const __grid_constant__ CUtensorMap map_w, int N, int K,
                      const float* __restrict__ X, int T, float* __restrict__ Y, float beta, int rows,
                      WaitCtl ctl) {
  constexpr int TBYTES = stage_row_bytes<WT>();
  constexpr int RMAX = fwd_rows<WT>(), STAGES = fwd_stages<WT>(), UMAX = RMAX / CONSUMERS;
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* stage_buf = sm;  // STAGES x RMAX x TBYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + STAGES * RMAX * TBYTES);  // full[S], empty[S]
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * rows, t0 = blockIdx.y * TB;
  const int n_kt = (K + 255) / 256;
  const uint32_t bar0 = smem_addr(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t stage_tx = static_cast<uint32_t>(rows) * TBYTES;

  // the producer's lane initialises the ring and starts its first copies
  // before the block-wide barrier (fresh slots need no wait)
  const bool producer = threadIdx.x == THREADS;
  uint32_t pend = 0;
  const int n_pre = min(STAGES, n_kt);
  if (producer) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), CONSUMERS);
    }
    abort_flag_s = 0;
    fence_mbar_init();
    for (int i = 0; i < n_pre; ++i) {
      mbar_arrive_expect_tx(full(i), stage_tx);
      tma_load_2d(smem_addr(stage_buf + i * RMAX * TBYTES), &map_w, full(i),
                  static_cast<int>(window_start<WT>(i) / 4), n0);
      pend |= 1u << i;
    }
  }
  __syncthreads();  // the ring's barriers

  if (warp == CONSUMERS) {
    if (lane == 0) {
      uint32_t ph = n_pre == STAGES ? 1u : 0u, pend_ph = 0;  // the phase of each started copy
      for (int i = n_pre; i < n_kt; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(empty(s), ph ^ 1u, ctl, abort_flag)) break;
        mbar_arrive_expect_tx(full(s), stage_tx);
        tma_load_2d(smem_addr(stage_buf + s * RMAX * TBYTES), &map_w, full(s),
                    static_cast<int>(window_start<WT>(i) / 4), n0);
        pend |= 1u << s;
        pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
        if (s == STAGES - 1) ph ^= 1u;
      }
      // every copy started lands before the CTA leaves
      volatile int no_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if (pend & (1u << s)) (void)mbar_wait(full(s), (pend_ph >> s) & 1u, ctl, &no_abort);
    }
    __syncwarp();
    return;
  }

  const int upw = rows / CONSUMERS;  // rows of the block this warp takes
  float acc[UMAX][TB];
#pragma unroll
  for (int u = 0; u < UMAX; ++u)
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[u][t] = 0.0f;
  bool ok = true;
  for (int i = 0; i < n_kt; ++i) {
    const int s = i % STAGES;
    // this lane's 8 values of each row of X in tile i (zeros past K and T;
    // K is a multiple of 8, so a lane's 8 values are all in or all out)
    const int k0 = i * 256 + 8 * lane;
    const bool kv = k0 < K;
    float x[TB][8];
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f), b = a;
      if (kv && t0 + t < T) {
        const float4* p = reinterpret_cast<const float4*>(X + static_cast<int64_t>(t0 + t) * K + k0);
        a = __ldg(p);
        b = __ldg(p + 1);
      }
      x[t][0] = a.x; x[t][1] = a.y; x[t][2] = a.z; x[t][3] = a.w;
      x[t][4] = b.x; x[t][5] = b.y; x[t][6] = b.z; x[t][7] = b.w;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(full(s), static_cast<uint32_t>(i / STAGES) & 1u, ctl,
                                           abort_flag))) {
      ok = false;
      break;
    }
    if (kv) {
      const uint8_t* tile = stage_buf + s * RMAX * TBYTES + window_offset<WT>(i);
#pragma unroll
      for (int u = 0; u < UMAX; ++u) {
        if (u < upw) {
          Raw<WT> raw;
          load_raw_smem<WT>(tile + (warp + CONSUMERS * u) * TBYTES, lane, raw);
          float w[8];
          decode_raw<WT>(raw, lane, w);
#pragma unroll
          for (int t = 0; t < TB; ++t)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[u][t] = fmaf(x[t][q], w[q], acc[u][t]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }
  if (!ok) return;  // a wait that gave up: Y is left as it was (rg_check reports it)
  // the 32 lanes' partial sums of each row in a fixed butterfly (every lane
  // ends with the same bits); lane 0 writes
#pragma unroll
  for (int u = 0; u < UMAX; ++u) {
    if (u < upw) {
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        float v = acc[u][t];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        const int n = n0 + warp + CONSUMERS * u;
        if (lane == 0 && n < N && t0 + t < T) {
          float* y = Y + static_cast<int64_t>(t0 + t) * N + n;
          *y = beta != 0.0f ? fmaf(beta, *y, v) : v;
        }
      }
    }
  }
}

// dX = beta * dX + sum over splits (in split order), four values per thread.
// dX offset of element i of a [T, K] slab, dX rows ldx floats apart
__device__ __forceinline__ int64_t dx_at(int64_t i, int64_t K, int64_t ldx) {
  if (ldx == K) return i;
  const int64_t t = i / K;
  return t * ldx + (i - t * K);
}

__global__ void __launch_bounds__(256) smallt_reduce(const float* __restrict__ part, int n_splits,
                                                     int64_t TK, int64_t K, int64_t ldx,
                                                     float* __restrict__ dX, float beta) {
  pdl_wait();  // the partial sums come from the kernel before this one
  for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * 4; i < TK;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x * 4) {
    float4 s = *reinterpret_cast<const float4*>(part + i);
    int p = 1;
    // eight loads in flight, then the adds in split order
    for (; p + 8 <= n_splits; p += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = *reinterpret_cast<const float4*>(part + static_cast<int64_t>(p + u) * TK + i);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w;
      }
    }
    for (; p < n_splits; ++p) {
      const float4 v = *reinterpret_cast<const float4*>(part + static_cast<int64_t>(p) * TK + i);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    float4* o = reinterpret_cast<float4*>(dX + dx_at(i, K, ldx));
    if (beta != 0.0f) {
      const float4 x = *o;
      s.x = fmaf(beta, x.x, s.x); s.y = fmaf(beta, x.y, s.y);
      s.z = fmaf(beta, x.z, s.z); s.w = fmaf(beta, x.w, s.w);
    }
    *o = s;
  }
}

// The same sum for few outputs and many splits, where one thread per output
// would wait out its loads one after another: a warp per four outputs, lane
// p loading split p0 + p; each group of 32 splits is added by a fixed xor
// tree and the groups in order.
__global__ void __launch_bounds__(256) smallt_reduce_wide(const float* __restrict__ part,
                                                          int n_splits, int64_t TK, int64_t K,
                                                          int64_t ldx, float* __restrict__ dX,
                                                          float beta) {
  pdl_wait();  // the partial sums come from the kernel before this one
  const int lane = threadIdx.x & 31;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t q = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; q * 4 < TK;
       q += nw) {
    const int64_t i = q * 4;
    float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int p0 = 0; p0 < n_splits; p0 += 32) {
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (p0 + lane < n_splits)
        v = *reinterpret_cast<const float4*>(part + static_cast<int64_t>(p0 + lane) * TK + i);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
        v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
      }
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    if (lane == 0) {
      float4* o = reinterpret_cast<float4*>(dX + dx_at(i, K, ldx));
      if (beta != 0.0f) {
        const float4 x = *o;
        s.x = fmaf(beta, x.x, s.x); s.y = fmaf(beta, x.y, s.y);
        s.z = fmaf(beta, x.z, s.z); s.w = fmaf(beta, x.w, s.w);
      }
      *o = s;
    }
  }
}

}  // namespace smt

// Resident CTAs per SM of smallt_kernel<WT, TB> on this device (queried once).
template <int WT, int TB>
static int smallt_residency(const DevInfo& dev) {
  // per device; threads that race on the first call store the same value
  static std::atomic<int> cache[64];
  std::atomic<int>& slot = cache[dev.device & 63];
  int c = slot.load(std::memory_order_relaxed);
  if (c == 0) {
    auto kern = smt::smallt_kernel<WT, TB>;
    constexpr size_t smem = smt::smem_bytes<WT, TB>();
    int n = 0;
    if (ensure_smem_attr(reinterpret_cast<const void*>(kern), static_cast<int>(smem)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, smt::THREADS + 32, smem) != cudaSuccess ||
        n <= 0)
      n = 1;
    slot.store(n, std::memory_order_relaxed);
    c = n;
  }
  return c;
}

template <int WT>
static int smallt_residency_tb(int tb, const DevInfo& dev) {
  switch (tb) {
    case 1: return smallt_residency<WT, 1>(dev);
    case 2: return smallt_residency<WT, 2>(dev);
    case 4: return smallt_residency<WT, 4>(dev);
    default: return smallt_residency<WT, 8>(dev);
  }
}

// At most this many rows of W, one CTA per tile takes them all.
constexpr int64_t kOneSliceRows = 256;

SmalltPlan plan_smallt(int wtype, int64_t N, int64_t K, int64_t T, const DevInfo& dev) {
  SmalltPlan p{};
  const int tb_max = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
  p.n_ktiles = static_cast<int>((K + 255) / 256);
  auto capacity_at = [&](int tb) {
    const int per_sm = with_wtype(wtype, 1, [&](auto wt) {
      return smallt_residency_tb<decltype(wt)::value>(tb, dev);
    });
    return static_cast<int64_t>(dev.num_sms) * per_sm;
  };
  if (N <= kOneSliceRows) {
    // few rows of W: one CTA takes all of them for its tile and writes dX
    // itself (no partial sums, no second kernel), with as few dY rows per
    // pass as keep the tiles within one wave
    int tb = 1;
    while (tb < tb_max && static_cast<int64_t>(p.n_ktiles) * ((T + tb - 1) / tb) > capacity_at(tb)) tb *= 2;
    p.tb = tb;
    p.n_tchunks = static_cast<int>((T + tb - 1) / tb);
    p.rows_per_split = static_cast<int>((N + 7) / 8 * 8);
    p.n_splits = 1;
    p.workspace = 0;
    return p;
  }
  p.tb = tb_max;
  p.n_tchunks = static_cast<int>((T + p.tb - 1) / p.tb);
  // one wave of resident CTAs; rows split no finer than 64 per CTA and no
  // coarser than the staged slice of dY allows
  const int64_t capacity = capacity_at(p.tb);
  const int64_t tiles = static_cast<int64_t>(p.n_ktiles) * p.n_tchunks;
  int64_t splits = std::max<int64_t>(1, capacity / tiles);
  splits = std::min<int64_t>(splits, (N + 63) / 64);
  splits = std::max<int64_t>(splits, (N + smt::MAX_ROWS - 1) / smt::MAX_ROWS);
  int64_t rows = (N + splits - 1) / splits;
  rows = (rows + 7) / 8 * 8;
  p.rows_per_split = static_cast<int>(rows);
  p.n_splits = static_cast<int>((N + rows - 1) / rows);
  // a single slice writes dX directly
  p.workspace = p.n_splits == 1 ? 0
                                : static_cast<size_t>(p.n_splits) * static_cast<size_t>(T) *
                                      static_cast<size_t>(K) * 4;
  return p;
}

template <int WT, int TB>
static cudaError_t launch_smallt_t(const void* W, int64_t N, int64_t K, const float* dY,
                                   int64_t T, float* dX, float beta, const Layout& lay, float* part,
                                   const SmalltPlan& p, const DevInfo& dev, cudaStream_t stream,
                                   int inject_stall) {
  auto kern = smt::smallt_kernel<WT, TB>;
  constexpr size_t smem = smt::smem_bytes<WT, TB>();
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // W as rows of 32-bit words; one box = a stage of rows x one 256-value tile
  const uint64_t rb = static_cast<uint64_t>(K / block_values(WT) * block_bytes(WT));
  CUtensorMap map;
  if (encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rb / 4, static_cast<uint64_t>(N), rb,
                   smt::stage_row_bytes<WT>() / 4, smt::stage_rows<WT, TB>(),
                   CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(p.n_ktiles), static_cast<unsigned>(p.n_splits),
                  static_cast<unsigned>(p.n_tchunks));
  WaitCtl ctl{dev.status, dev.wait_limit_ns};
  // one slice of rows: the sums are dX itself; else partial sums for the
  // reduction kernel
  const smt::SmtOut out = p.n_splits == 1 ? smt::SmtOut{dX, lay.dx_t, beta} : smt::SmtOut{part, K, 0.0f};
  kern<<<grid, smt::THREADS + 32, smem, stream>>>(map, static_cast<int>(N), static_cast<int>(K), dY,
                                                   lay.dy_t, lay.dy_n, static_cast<int>(T), out,
                                                   p.rows_per_split, ctl, inject_stall);
  return counted(cudaGetLastError());
}

template <int WT>
static cudaError_t launch_smallt_w(const void* W, int64_t N, int64_t K, const float* dY,
                                   int64_t T, float* dX, float beta, const Layout& lay, float* part,
                                   const SmalltPlan& p, const DevInfo& dev, cudaStream_t stream,
                                   int inject_stall) {
  switch (p.tb) {
    case 1: return launch_smallt_t<WT, 1>(W, N, K, dY, T, dX, beta, lay, part, p, dev, stream, inject_stall);
    case 2: return launch_smallt_t<WT, 2>(W, N, K, dY, T, dX, beta, lay, part, p, dev, stream, inject_stall);
    case 4: return launch_smallt_t<WT, 4>(W, N, K, dY, T, dX, beta, lay, part, p, dev, stream, inject_stall);
    default: return launch_smallt_t<WT, 8>(W, N, K, dY, T, dX, beta, lay, part, p, dev, stream, inject_stall);
  }
}

cudaError_t launch_smallt(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, const Layout& lay, float* part,
                          const SmalltPlan& p, const DevInfo& dev, cudaStream_t stream,
                          int inject_stall) {
  if (p.n_tchunks > 65535 || p.n_splits > 65535) return cudaErrorInvalidConfiguration;
  const cudaError_t e = with_wtype(wtype, cudaErrorInvalidValue, [&](auto wt) {
    return launch_smallt_w<decltype(wt)::value>(W, N, K, dY, T, dX, beta, lay, part, p, dev, stream,
                                                inject_stall);
  });
  if (e != cudaSuccess || p.n_splits == 1) return e;  // one slice: the kernel wrote dX
  return launch_reduce_partials(part, p.n_splits, T, K, dX, lay.dx_t, beta, dev, stream);
}

template <int WT, int TB>
static cudaError_t launch_smallt_fwd_t(const void* W, int64_t N, int64_t K, const float* X, int64_t T,
                                       float* Y, float beta, const DevInfo& dev, cudaStream_t stream) {
  auto kern = smt::smallt_fwd_kernel<WT, TB>;
  constexpr size_t smem = smt::fwd_smem_bytes<WT>();
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // per device; threads that race on the first call store the same value
  static std::atomic<int> cache[64];
  std::atomic<int>& slot = cache[dev.device & 63];
  int per_sm = slot.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, smt::THREADS + 32, smem) != cudaSuccess ||
        per_sm <= 0)
      per_sm = 1;
    slot.store(per_sm, std::memory_order_relaxed);
  }
  // blocks of rows: the largest of 32 (16 for F32), 16 and 8 rows that still
  // gives at least half a wave of CTAs
  const int64_t n_tchunks = (T + TB - 1) / TB;
  const int64_t half_wave = static_cast<int64_t>(dev.num_sms) * per_sm / 2;
  int rows = smt::fwd_rows<WT>();
  while (rows > 8 && (N + rows - 1) / rows * n_tchunks < half_wave) rows /= 2;
  const int64_t n_blocks = (N + rows - 1) / rows;
  if (n_blocks > 0x7FFFFFFF || n_tchunks > 65535) return cudaErrorInvalidConfiguration;
  const uint64_t rb = static_cast<uint64_t>(K / block_values(WT) * block_bytes(WT));
  CUtensorMap map;
  if (encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rb / 4, static_cast<uint64_t>(N), rb,
                   smt::stage_row_bytes<WT>() / 4, static_cast<uint32_t>(rows),
                   CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  WaitCtl ctl{dev.status, dev.wait_limit_ns};
  kern<<<dim3(static_cast<unsigned>(n_blocks), static_cast<unsigned>(n_tchunks)), smt::THREADS + 32, smem,
         stream>>>(map, static_cast<int>(N), static_cast<int>(K), X, static_cast<int>(T), Y, beta, rows, ctl);
  return counted(cudaGetLastError());
}

cudaError_t launch_smallt_fwd(int wtype, const void* W, int64_t N, int64_t K, const float* X, int64_t T,
                              float* Y, float beta, const DevInfo& dev, cudaStream_t stream) {
  return with_wtype(wtype, cudaErrorInvalidValue, [&](auto wt) {
    constexpr int WT = decltype(wt)::value;
    return T <= 1   ? launch_smallt_fwd_t<WT, 1>(W, N, K, X, T, Y, beta, dev, stream)
           : T <= 2 ? launch_smallt_fwd_t<WT, 2>(W, N, K, X, T, Y, beta, dev, stream)
                    : launch_smallt_fwd_t<WT, 4>(W, N, K, X, T, Y, beta, dev, stream);
  });
}

cudaError_t launch_reduce_partials(const float* part, int n_splits, int64_t T, int64_t K,
                                   float* dX, int64_t dx_t, float beta, const DevInfo& dev,
                                   cudaStream_t stream) {
  const int64_t TK = T * K;
  // latency regime (a warp per four outputs fits in one wave): the wide form
  const int64_t quads = TK / 4;
  if (n_splits >= 4 && quads * 32 <= static_cast<int64_t>(dev.num_sms) * 2048) {
    const int64_t blocks = (quads * 32 + 255) / 256;
    return counted(launch_after_prev(smt::smallt_reduce_wide,
                                     dim3(static_cast<unsigned>(std::max<int64_t>(1, blocks))),
                                     dim3(256), stream, part, n_splits, TK, K, dx_t, dX, beta));
  }
  const int64_t blocks = std::min<int64_t>((quads + 255) / 256, static_cast<int64_t>(dev.num_sms) * 8);
  return counted(launch_after_prev(smt::smallt_reduce,
                                   dim3(static_cast<unsigned>(std::max<int64_t>(1, blocks))),
                                   dim3(256), stream, part, n_splits, TK, K, dx_t, dX, beta));
}

}  // namespace rg
