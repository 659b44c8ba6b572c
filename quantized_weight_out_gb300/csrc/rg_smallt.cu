// rg_smallt.cu - the small-T variant of
//   dX[t, k] = beta * dX[t, k] + sum_n dY[t, n] * deq(W)[n, k]
// for a handful of rows of dY, where the bytes of W bound the product (the
// role of the in-place decoder the Retrograd page "CUDA status", section
// "Limitations", keeps for small outputs).
//
// Every weight value is read from memory once per pass of up to 8 dY rows,
// decoded exactly to F32 in registers, and multiplied in F32 by each dY row.
//  * A warp walks whole rows of W: lane l owns values 8l .. 8l+7 of a
//    256-value tile, so the 32 lanes read one contiguous row segment (16-byte
//    loads for F16/BF16, 8-byte loads of Q4_K nibbles, 2-byte loads of the
//    34/18-byte Q8_0/Q4_0 blocks) and several rows are in flight per warp.
//  * The rows are split over many CTAs (grid.y) so that the whole GPU streams
//    W; each CTA sums its eight warps in a fixed order and writes its partial
//    tile to a workspace, and a second kernel adds the partials in split
//    order together with beta * dX: deterministic, no atomics.
#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {
namespace smt {

constexpr int THREADS = 256;   // 8 warps
constexpr int ROWS = 256;      // dY columns (= W rows) staged per chunk

// Raw bytes one lane needs from a row for its 8 values (a 256-value tile).
template <int WT>
struct Raw {
  uint32_t v[WT == RG_Q4_K ? 6 : WT == RG_Q8_0 || WT == RG_Q4_0 ? 3 : 4];
};

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t* p) {
  return static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)));
}

// tile: first byte of the row's 256-value tile (16-byte aligned)
template <int WT>
__device__ __forceinline__ void load_raw(const uint8_t* tile, int lane, Raw<WT>& r) {
  if constexpr (WT == RG_F16 || WT == RG_BF16) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(tile) + lane);
    r.v[0] = q.x; r.v[1] = q.y; r.v[2] = q.z; r.v[3] = q.w;
  } else if constexpr (WT == RG_Q8_0) {
    const uint8_t* blk = tile + 34 * (lane >> 2);          // 4 lanes per 32-value block
    const uint8_t* q = blk + 2 + 8 * (lane & 3);
    r.v[0] = ldg_u16(blk);
    r.v[1] = ldg_u16(q) | (ldg_u16(q + 2) << 16);
    r.v[2] = ldg_u16(q + 4) | (ldg_u16(q + 6) << 16);
  } else if constexpr (WT == RG_Q4_0) {
    const uint8_t* blk = tile + 18 * (lane >> 2);
    const uint8_t* q = blk + 2 + 8 * (lane & 1);           // low nibbles for lane&3 < 2, high after
    r.v[0] = ldg_u16(blk);
    r.v[1] = ldg_u16(q) | (ldg_u16(q + 2) << 16);
    r.v[2] = ldg_u16(q + 4) | (ldg_u16(q + 6) << 16);
  } else {  // Q4_K: header (d, dmin, 12 scale bytes) and 8 nibble bytes
    const uint4 h = __ldg(reinterpret_cast<const uint4*>(tile));
    const int c = lane >> 3, l0 = 8 * (lane & 3);
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(tile + 16 + 32 * c + l0));
    r.v[0] = h.x; r.v[1] = h.y; r.v[2] = h.z; r.v[3] = h.w; r.v[4] = q.x; r.v[5] = q.y;
  }
}

__device__ __forceinline__ int byte_at(const uint32_t* w, int i) {
  return static_cast<int>((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
}

// Exact F32 decode of the lane's 8 values: the same products and single
// rounding as the format definitions (signed zeros kept).
template <int WT>
__device__ __forceinline__ void decode_raw(const Raw<WT>& r, int lane, float (&w)[8]) {
  if constexpr (WT == RG_F16 || WT == RG_BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = static_cast<uint16_t>(r.v[i] & 0xFFFFu);
      const uint16_t hi = static_cast<uint16_t>(r.v[i] >> 16);
      w[2 * i] = WT == RG_F16 ? f16_to_f32(lo) : bf16_to_f32(lo);
      w[2 * i + 1] = WT == RG_F16 ? f16_to_f32(hi) : bf16_to_f32(hi);
    }
  } else if constexpr (WT == RG_Q8_0) {
    const float d = f16_to_f32(static_cast<uint16_t>(r.v[0]));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int8_t q = static_cast<int8_t>((r.v[1 + (i >> 2)] >> (8 * (i & 3))) & 0xFFu);
      w[i] = d * static_cast<float>(q);
    }
  } else if constexpr (WT == RG_Q4_0) {
    const float d = f16_to_f32(static_cast<uint16_t>(r.v[0]));
    const int shift = (lane & 2) ? 4 : 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = static_cast<int>((r.v[1 + (i >> 2)] >> (8 * (i & 3) + shift)) & 15u);
      w[i] = d * static_cast<float>(q - 8);
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
    const float ds = d * static_cast<float>(sc);
    const float dm = dmin * static_cast<float>(m);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = static_cast<int>((r.v[4 + (i >> 2)] >> (8 * (i & 3) + 4 * half)) & 15u);
      w[i] = ds * static_cast<float>(q) - dm;
    }
  }
}

// grid (ceil(K/256), n_splits, ceil(T/TB)); partial sums of rows
// [split * rows_per_split, +rows_per_split) to part[(split * T + t) * K + k].
template <int WT, int TB, int RU>
__global__ void __launch_bounds__(THREADS, 2)
    smallt_kernel(const uint8_t* __restrict__ W, int64_t rb, int N, int K,
                  const float* __restrict__ dY, int T, float* __restrict__ part,
                  int rows_per_split) {
  __shared__ float ys[TB][ROWS];
  __shared__ __align__(16) float red[4][TB][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, split = blockIdx.y;
  const int t0 = blockIdx.z * TB;
  const int nbeg = split * rows_per_split;
  const int nend = min(N, nbeg + rows_per_split);
  const bool kvalid = kt * 256 + 8 * lane < K;
  const int64_t tile_off = static_cast<int64_t>(kt) * (256 / block_values(WT)) * block_bytes(WT);

  float acc[TB][8];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[t][i] = 0.0f;

  for (int c0 = nbeg; c0 < nend; c0 += ROWS) {
    const int cn = min(ROWS, nend - c0);
    for (int idx = threadIdx.x; idx < TB * ROWS; idx += THREADS) {
      const int t = idx / ROWS, r = idx - t * ROWS;
      ys[t][r] = (t0 + t < T && r < cn) ? __ldg(dY + static_cast<int64_t>(t0 + t) * N + c0 + r) : 0.0f;
    }
    __syncthreads();
    if (kvalid) {
      for (int r = warp; r < cn; r += 8 * RU) {
        Raw<WT> raw[RU];
#pragma unroll
        for (int u = 0; u < RU; ++u) {
          const int rr = r + 8 * u;
          if (rr < cn) load_raw<WT>(W + static_cast<int64_t>(c0 + rr) * rb + tile_off, lane, raw[u]);
        }
#pragma unroll
        for (int u = 0; u < RU; ++u) {
          const int rr = r + 8 * u;
          if (rr < cn) {
            float w[8];
            decode_raw<WT>(raw[u], lane, w);
#pragma unroll
            for (int t = 0; t < TB; ++t) {
              const float y = ys[t][rr];
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[t][i] = fmaf(y, w[i], acc[t][i]);
            }
          }
        }
      }
    }
    __syncthreads();
  }

  // the CTA's eight warps, summed in a fixed order: (w + 4) into w, then 0..3
  if (warp >= 4) {
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) red[warp - 4][t][8 * lane + i] = acc[t][i];
  }
  __syncthreads();
  if (warp < 4) {
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) red[warp][t][8 * lane + i] += acc[t][i];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < TB * 256; idx += THREADS) {
    const int t = idx >> 8, kk = idx & 255;
    const int gt = t0 + t, gk = kt * 256 + kk;
    if (gt < T && gk < K) {
      const float s = ((red[0][t][kk] + red[1][t][kk]) + red[2][t][kk]) + red[3][t][kk];
      part[(static_cast<int64_t>(split) * T + gt) * K + gk] = s;
    }
  }
}

// dX = beta * dX + sum over splits (in split order), four values per thread.
__global__ void __launch_bounds__(256) smallt_reduce(const float* __restrict__ part, int n_splits,
                                                     int64_t TK, float* __restrict__ dX,
                                                     float beta) {
  for (int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * 4; i < TK;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x * 4) {
    float4 s = *reinterpret_cast<const float4*>(part + i);
    for (int p = 1; p < n_splits; ++p) {
      const float4 v = *reinterpret_cast<const float4*>(part + static_cast<int64_t>(p) * TK + i);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    float4* o = reinterpret_cast<float4*>(dX + i);
    if (beta != 0.0f) {
      const float4 x = *o;
      s.x = fmaf(beta, x.x, s.x); s.y = fmaf(beta, x.y, s.y);
      s.z = fmaf(beta, x.z, s.z); s.w = fmaf(beta, x.w, s.w);
    }
    *o = s;
  }
}

}  // namespace smt

SmalltPlan plan_smallt(int64_t N, int64_t K, int64_t T, const DevInfo& dev) {
  SmalltPlan p{};
  p.tb = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
  p.n_ktiles = static_cast<int>((K + 255) / 256);
  p.n_tchunks = static_cast<int>((T + p.tb - 1) / p.tb);
  const int64_t target = static_cast<int64_t>(dev.num_sms) * 4;
  int64_t splits = (target + p.n_ktiles * p.n_tchunks - 1) / (p.n_ktiles * p.n_tchunks);
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, (N + 63) / 64));
  int64_t rows = (N + splits - 1) / splits;
  rows = (rows + 7) / 8 * 8;
  p.rows_per_split = static_cast<int>(rows);
  p.n_splits = static_cast<int>((N + rows - 1) / rows);
  p.workspace = static_cast<size_t>(p.n_splits) * static_cast<size_t>(T) * static_cast<size_t>(K) * 4;
  return p;
}

template <int WT, int TB>
static cudaError_t launch_smallt_t(const void* W, int64_t N, int64_t K, const float* dY,
                                   int64_t T, float* part, const SmalltPlan& p,
                                   cudaStream_t stream) {
  constexpr int RU = TB <= 4 ? 8 : 4;
  const int64_t rb = K / block_values(WT) * block_bytes(WT);
  const dim3 grid(static_cast<unsigned>(p.n_ktiles), static_cast<unsigned>(p.n_splits),
                  static_cast<unsigned>(p.n_tchunks));
  smt::smallt_kernel<WT, TB, RU><<<grid, smt::THREADS, 0, stream>>>(
      static_cast<const uint8_t*>(W), rb, static_cast<int>(N), static_cast<int>(K), dY,
      static_cast<int>(T), part, p.rows_per_split);
  return cudaGetLastError();
}

template <int WT>
static cudaError_t launch_smallt_w(const void* W, int64_t N, int64_t K, const float* dY,
                                   int64_t T, float* part, const SmalltPlan& p,
                                   cudaStream_t stream) {
  switch (p.tb) {
    case 1: return launch_smallt_t<WT, 1>(W, N, K, dY, T, part, p, stream);
    case 2: return launch_smallt_t<WT, 2>(W, N, K, dY, T, part, p, stream);
    case 4: return launch_smallt_t<WT, 4>(W, N, K, dY, T, part, p, stream);
    default: return launch_smallt_t<WT, 8>(W, N, K, dY, T, part, p, stream);
  }
}

cudaError_t launch_smallt(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, float* part, const SmalltPlan& p,
                          const DevInfo& dev, cudaStream_t stream) {
  if (p.n_tchunks > 65535 || p.n_splits > 65535) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  switch (wtype) {
    case RG_F16: e = launch_smallt_w<RG_F16>(W, N, K, dY, T, part, p, stream); break;
    case RG_BF16: e = launch_smallt_w<RG_BF16>(W, N, K, dY, T, part, p, stream); break;
    case RG_Q8_0: e = launch_smallt_w<RG_Q8_0>(W, N, K, dY, T, part, p, stream); break;
    case RG_Q4_0: e = launch_smallt_w<RG_Q4_0>(W, N, K, dY, T, part, p, stream); break;
    case RG_Q4_K: e = launch_smallt_w<RG_Q4_K>(W, N, K, dY, T, part, p, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  const int64_t TK = T * K;
  const int64_t blocks = std::min<int64_t>((TK / 4 + 255) / 256, static_cast<int64_t>(dev.num_sms) * 8);
  smt::smallt_reduce<<<static_cast<unsigned>(std::max<int64_t>(1, blocks)), 256, 0, stream>>>(
      part, p.n_splits, TK, dX, beta);
  return cudaGetLastError();
}

}  // namespace rg
