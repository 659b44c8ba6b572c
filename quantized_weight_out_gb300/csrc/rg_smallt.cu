// rg_smallt.cu - the small-T variant of
//   dX[t, k] = beta * dX[t, k] + sum_n dY[t, n] * deq(W)[n, k]
// for a handful of rows of dY, where the bytes of W bound the product (the
// role of the in-place decoder the Retrograd page "CUDA status", section
// "Limitations", keeps for small outputs).
//
// Every weight value is read from memory once per pass of up to 8 dY rows,
// decoded exactly to F32 in registers, and multiplied in F32 by each dY row.
//  * A producer warp streams the CTA's rows of W (its 256-value tile of each
//    row) with TMA into an 8-stage shared-memory ring of 32-row tiles, so
//    enough bytes are in flight without holding them in registers.
//  * A consumer warp takes whole rows: lane l owns values 8l .. 8l+7, reads
//    their bytes from shared memory and decodes them in registers.
//  * The rows are split over many CTAs (grid.y) so that the whole GPU streams
//    W; each CTA sums its eight warps in a fixed order and writes its partial
//    tile to a workspace, and a second kernel adds the partials in split
//    order together with beta * dX: deterministic, no atomics.
#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {
namespace smt {

constexpr int THREADS = 256;   // 8 consumer warps (plus one producer warp)

// Raw bytes one lane needs from a row for its 8 values (a 256-value tile).
template <int WT>
struct Raw {
  uint32_t v[WT == RG_Q4_K ? 6 : WT == RG_Q8_0 || WT == RG_Q4_0 ? 3 : 4];
};

// The bytes one lane needs for its 8 values, from a row tile staged in
// shared memory (tile: the row's 256-value tile, 16-byte aligned).
template <int WT>
__device__ __forceinline__ void load_raw_smem(const uint8_t* tile, int lane, Raw<WT>& r) {
  if constexpr (WT == RG_F16 || WT == RG_BF16) {
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
  } else {
    const uint4 h = *reinterpret_cast<const uint4*>(tile);
    const int c = lane >> 3, l0 = 8 * (lane & 3);
    const uint2 q = *reinterpret_cast<const uint2*>(tile + 16 + 32 * c + l0);
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

// Bytes of one row's 256-value tile.
template <int WT>
__host__ __device__ constexpr int tile_bytes() {
  return (256 / block_values(WT)) * block_bytes(WT);
}

constexpr int BR = 32;       // rows of W per pipeline stage
constexpr int STAGES = 8;    // stages in flight per CTA
constexpr int CONSUMERS = 8; // consumer warps; warp 8 is the TMA producer
constexpr int MAX_ROWS = 512;

// grid (ceil(K/256), n_splits, ceil(T/TB)); partial sums of rows
// [split * rows_per_split, +rows_per_split) to part[(split * T + t) * K + k].
// A producer warp streams the CTA's rows of W, tile by tile of BR rows, into
// an 8-stage ring with TMA; eight consumer warps decode from shared memory.
template <int WT, int TB>
__global__ void __launch_bounds__(THREADS + 32, TB >= 8 ? 1 : 2)
    smallt_kernel(const __grid_constant__ CUtensorMap map_w, int N, int K,
                  const float* __restrict__ dY, int T, float* __restrict__ part,
                  int rows_per_split, WaitCtl ctl) {
  constexpr int TBYTES = tile_bytes<WT>();
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* stage_buf = sm;                                              // STAGES x BR x TBYTES
  float* ys = reinterpret_cast<float*>(sm + STAGES * BR * TBYTES);      // [TB][MAX_ROWS]
  float* red = ys + TB * MAX_ROWS;                                      // [4][TB][256]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + 4 * TB * 256);    // full[S], empty[S]
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, split = blockIdx.y;
  const int t0 = blockIdx.z * TB;
  const int nbeg = split * rows_per_split;
  const int nrows = max(0, min(N, nbeg + rows_per_split) - nbeg);
  const int n_tiles = (nrows + BR - 1) / BR;
  const uint32_t bar0 = smem_addr(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), CONSUMERS);
    }
    abort_flag_s = 0;
    fence_mbar_init();
  }
  // this CTA's slice of dY, [TB][nrows]
  for (int idx = threadIdx.x; idx < TB * MAX_ROWS; idx += THREADS + 32) {
    const int t = idx / MAX_ROWS, r = idx - t * MAX_ROWS;
    ys[idx] = (t0 + t < T && r < nrows) ? __ldg(dY + static_cast<int64_t>(t0 + t) * N + nbeg + r) : 0.0f;
  }
  __syncthreads();

  if (warp == CONSUMERS) {
    // ---------------- producer ----------------
    if (lane == 0) {
      uint32_t ph = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(empty(s), ph ^ 1u, ctl, abort_flag)) break;
        mbar_arrive_expect_tx(full(s), BR * TBYTES);
        tma_load_2d(smem_addr(stage_buf + s * BR * TBYTES), &map_w, full(s), kt * (TBYTES / 4),
                    nbeg + i * BR);
        if (s == STAGES - 1) ph ^= 1u;
      }
      // drain: the copies started land before the CTA leaves
      volatile int no_abort = 0;
      for (int i = max(0, n_tiles - STAGES); i < n_tiles; ++i)
        (void)mbar_wait(full(i % STAGES), static_cast<uint32_t>(i / STAGES) & 1u, ctl, &no_abort);
    }
    __syncwarp();
  }

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
        const uint8_t* tile = stage_buf + s * BR * TBYTES;
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
      part[(static_cast<int64_t>(split) * T + gt) * K + gk] = sum;
    }
  }
}

template <int WT, int TB>
constexpr size_t smem_bytes() {
  return static_cast<size_t>(STAGES) * BR * tile_bytes<WT>() + sizeof(float) * TB * MAX_ROWS +
         sizeof(float) * 4 * TB * 256 + 16 * STAGES;
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
  splits = std::max<int64_t>(splits, (N + smt::MAX_ROWS - 1) / smt::MAX_ROWS);
  int64_t rows = (N + splits - 1) / splits;
  rows = (rows + 7) / 8 * 8;
  p.rows_per_split = static_cast<int>(rows);
  p.n_splits = static_cast<int>((N + rows - 1) / rows);
  p.workspace = static_cast<size_t>(p.n_splits) * static_cast<size_t>(T) * static_cast<size_t>(K) * 4;
  return p;
}

template <int WT, int TB>
static cudaError_t launch_smallt_t(const CUtensorMap& map, int64_t N, int64_t K, const float* dY,
                                   int64_t T, float* part, const SmalltPlan& p, const DevInfo& dev,
                                   cudaStream_t stream) {
  auto kern = smt::smallt_kernel<WT, TB>;
  constexpr size_t smem = smt::smem_bytes<WT, TB>();
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.n_ktiles), static_cast<unsigned>(p.n_splits),
                  static_cast<unsigned>(p.n_tchunks));
  WaitCtl ctl{dev.status, dev.wait_limit_ns};
  kern<<<grid, smt::THREADS + 32, smem, stream>>>(map, static_cast<int>(N), static_cast<int>(K), dY,
                                                   static_cast<int>(T), part, p.rows_per_split, ctl);
  return counted(cudaGetLastError());
}

template <int WT>
static cudaError_t launch_smallt_w(const void* W, int64_t N, int64_t K, const float* dY,
                                   int64_t T, float* part, const SmalltPlan& p, const DevInfo& dev,
                                   cudaStream_t stream) {
  // W as rows of 32-bit words; one box = BR rows x one 256-value tile
  const uint64_t rb = static_cast<uint64_t>(K / block_values(WT) * block_bytes(WT));
  CUtensorMap map;
  if (encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rb / 4, static_cast<uint64_t>(N), rb,
                   smt::tile_bytes<WT>() / 4, smt::BR, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  switch (p.tb) {
    case 1: return launch_smallt_t<WT, 1>(map, N, K, dY, T, part, p, dev, stream);
    case 2: return launch_smallt_t<WT, 2>(map, N, K, dY, T, part, p, dev, stream);
    case 4: return launch_smallt_t<WT, 4>(map, N, K, dY, T, part, p, dev, stream);
    default: return launch_smallt_t<WT, 8>(map, N, K, dY, T, part, p, dev, stream);
  }
}

cudaError_t launch_smallt(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, float* part, const SmalltPlan& p,
                          const DevInfo& dev, cudaStream_t stream) {
  if (p.n_tchunks > 65535 || p.n_splits > 65535) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  switch (wtype) {
    case RG_F16: e = launch_smallt_w<RG_F16>(W, N, K, dY, T, part, p, dev, stream); break;
    case RG_BF16: e = launch_smallt_w<RG_BF16>(W, N, K, dY, T, part, p, dev, stream); break;
    case RG_Q8_0: e = launch_smallt_w<RG_Q8_0>(W, N, K, dY, T, part, p, dev, stream); break;
    case RG_Q4_0: e = launch_smallt_w<RG_Q4_0>(W, N, K, dY, T, part, p, dev, stream); break;
    case RG_Q4_K: e = launch_smallt_w<RG_Q4_K>(W, N, K, dY, T, part, p, dev, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_reduce_partials(part, p.n_splits, T * K, dX, beta, dev, stream);
}

cudaError_t launch_reduce_partials(const float* part, int n_splits, int64_t TK, float* dX,
                                   float beta, const DevInfo& dev, cudaStream_t stream) {
  const int64_t blocks = std::min<int64_t>((TK / 4 + 255) / 256, static_cast<int64_t>(dev.num_sms) * 8);
  smt::smallt_reduce<<<static_cast<unsigned>(std::max<int64_t>(1, blocks)), 256, 0, stream>>>(
      part, n_splits, TK, dX, beta);
  return counted(cudaGetLastError());
}

}  // namespace rg
