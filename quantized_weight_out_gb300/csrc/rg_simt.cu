// rg_simt.cu - the two CUDA-core variants of the OUT_PROD
//   dX[t, k] = beta * dX[t, k] + sum_n dY[t, n] * deq(W)[n, k].
//
// simt32: exact F32 decode and F32 FMA, accumulated in 32-row partial sums
//   that are then added together (blocked summation keeps the F32 error far
//   below the sequential worst case over N up to ~17k rows).
// smallt: for a handful of rows of dY the product is bound by the bytes of W,
//   as the Retrograd page "CUDA status" (section "Limitations") notes when it
//   keeps an in-place decoder for small outputs.  Each weight value is decoded
//   once, in registers, and multiplied by up to 8 dY rows held in shared
//   memory; the N rows are split over a thread-block cluster whose partial
//   sums are added through distributed shared memory (deterministic, no
//   scratch memory, no atomics).
#include <cooperative_groups.h>

#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace cg = cooperative_groups;

namespace rg {

// ---------------------------------------------------------------------------
// simt32: one CTA per 64(t) x 64(k) output tile, 256 threads, 4x4 outputs each

constexpr int S32_TT = 64, S32_TK = 64, S32_TN = 32;

template <int WT>
__global__ void __launch_bounds__(256) simt32_kernel(const uint8_t* __restrict__ W, int64_t rb,
                                                     int N, int K,
                                                     const float* __restrict__ dY, int T,
                                                     float* __restrict__ dX, float beta) {
  __shared__ float ys[S32_TN][S32_TT + 1];              // [n][t]
  __shared__ __align__(16) float ws[S32_TN][S32_TK];    // [n][k]
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * S32_TT;
  const int k0 = blockIdx.x * S32_TK;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int n0 = 0; n0 < N; n0 += S32_TN) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + 256 * i;
      const int r = idx >> 5, c = idx & 31;
      const int64_t t = t0 + r;
      const int n = n0 + c;
      ys[c][r] = (t < T && n < N) ? dY[t * N + n] : 0.0f;
    }
    {
      const int r = tid >> 3, kk = 8 * (tid & 7);
      const int n = n0 + r, k = k0 + kk;
      float v[8];
      if (n < N && k < K) {
        decode8_f32<WT>(W + static_cast<int64_t>(n) * rb, k, v);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ws[r][kk + i] = v[i];
    }
    __syncthreads();
    float p[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) p[i][j] = 0.0f;
#pragma unroll 8
    for (int c = 0; c < S32_TN; ++c) {
      float y[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) y[i] = ys[c][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = ws[c][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) p[i][j] = fmaf(y[i], w[j], p[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] += p[i][j];
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + ty + 16 * i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + tx + 16 * j;
      if (k >= K) continue;
      float* o = dX + t * K + k;
      *o = beta != 0.0f ? fmaf(beta, *o, acc[i][j]) : acc[i][j];
    }
  }
}

cudaError_t launch_simt32(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, const DevInfo& dev,
                          cudaStream_t stream) {
  (void)dev;
  const int64_t rb = K / block_values(wtype) * block_bytes(wtype);
  const dim3 grid(static_cast<unsigned>((K + S32_TK - 1) / S32_TK),
                  static_cast<unsigned>((T + S32_TT - 1) / S32_TT));
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const int n = static_cast<int>(N), k = static_cast<int>(K), t = static_cast<int>(T);
  switch (wtype) {
    case RG_F16: simt32_kernel<RG_F16><<<grid, 256, 0, stream>>>(w, rb, n, k, dY, t, dX, beta); break;
    case RG_BF16: simt32_kernel<RG_BF16><<<grid, 256, 0, stream>>>(w, rb, n, k, dY, t, dX, beta); break;
    case RG_Q8_0: simt32_kernel<RG_Q8_0><<<grid, 256, 0, stream>>>(w, rb, n, k, dY, t, dX, beta); break;
    case RG_Q4_0: simt32_kernel<RG_Q4_0><<<grid, 256, 0, stream>>>(w, rb, n, k, dY, t, dX, beta); break;
    case RG_Q4_K: simt32_kernel<RG_Q4_K><<<grid, 256, 0, stream>>>(w, rb, n, k, dY, t, dX, beta); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// smallt
//
// grid (ceil(K/256), C, ceil(T/TB)), cluster (1, C, 1).  A CTA covers 256
// values of k and rows [rank*R, rank*R + R) of W.  Warp w: k-quarter w & 3
// (64 values), row phase w >> 2; lane l: 8 values of k at 8*(l >> 2), row
// slot l & 3, so a thread visits the rows congruent to its (phase, slot)
// mod 8.  Partial sums are reduced over the row slots by warp shuffles, over
// the two row phases in shared memory, and over the cluster through DSMEM.

constexpr int ST_TB = 8;        // dY rows per pass
constexpr int ST_ROWS = 128;    // W rows staged per chunk of dY

template <int WT>
__global__ void __launch_bounds__(256) smallt_kernel(const uint8_t* __restrict__ W, int64_t rb,
                                                     int N, int K,
                                                     const float* __restrict__ dY, int T,
                                                     float* __restrict__ dX, float beta,
                                                     int rows_per_cta) {
  cg::cluster_group cluster = cg::this_cluster();
  const int csize = static_cast<int>(cluster.num_blocks());
  const int crank = static_cast<int>(cluster.block_rank());

  __shared__ float ys[ST_TB][ST_ROWS];
  __shared__ __align__(16) float red[ST_TB * 256];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kq = warp & 3, rp = warp >> 2, kg = lane >> 2, rs = lane & 3;
  const int kl = 64 * kq + 8 * kg;
  const int k = blockIdx.x * 256 + kl;
  const bool kvalid = k < K;
  const int64_t t0 = static_cast<int64_t>(blockIdx.z) * ST_TB;
  const int nbeg = crank * rows_per_cta;
  const int nend = min(N, nbeg + rows_per_cta);

  float acc[ST_TB][8];
#pragma unroll
  for (int t = 0; t < ST_TB; ++t)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[t][i] = 0.0f;

  for (int c0 = nbeg; c0 < nend; c0 += ST_ROWS) {
    const int cn = min(ST_ROWS, nend - c0);
    for (int idx = tid; idx < ST_TB * ST_ROWS; idx += 256) {
      const int r = idx / ST_ROWS, c = idx % ST_ROWS;
      const int64_t t = t0 + r;
      ys[r][c] = (t < T && c < cn) ? dY[t * N + c0 + c] : 0.0f;
    }
    __syncthreads();
    if (kvalid) {
      for (int rr = rp * 4 + rs; rr < cn; rr += 8) {
        float w[8];
        decode8_f32<WT>(W + static_cast<int64_t>(c0 + rr) * rb, k, w);
#pragma unroll
        for (int t = 0; t < ST_TB; ++t) {
          const float y = ys[t][rr];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[t][i] = fmaf(y, w[i], acc[t][i]);
        }
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int t = 0; t < ST_TB; ++t)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc[t][i] += __shfl_xor_sync(0xffffffffu, acc[t][i], 1);
      acc[t][i] += __shfl_xor_sync(0xffffffffu, acc[t][i], 2);
    }
  if (rp == 1 && rs == 0) {
#pragma unroll
    for (int t = 0; t < ST_TB; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) red[t * 256 + kl + i] = acc[t][i];
  }
  __syncthreads();
  if (rp == 0 && rs == 0) {
#pragma unroll
    for (int t = 0; t < ST_TB; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) red[t * 256 + kl + i] += acc[t][i];
  }
  cluster.sync();

  // rank r of the cluster finishes outputs [r*per, (r+1)*per) of the TB x 256 tile
  const int per = ST_TB * 256 / csize;
  for (int idx = crank * per + tid; idx < (crank + 1) * per; idx += 256) {
    float s = 0.0f;
    for (int r = 0; r < csize; ++r) s += cluster.map_shared_rank(red, r)[idx];
    const int64_t gt = t0 + idx / 256;
    const int gk = blockIdx.x * 256 + (idx & 255);
    if (gt < T && gk < K) {
      float* o = dX + gt * K + gk;
      *o = beta != 0.0f ? fmaf(beta, *o, s) : s;
    }
  }
  cluster.sync();
}

cudaError_t launch_smallt(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, const DevInfo& dev,
                          cudaStream_t stream) {
  (void)dev;
  int csize = 1;
  while (csize < 8 && N / (2 * csize) >= 64) csize *= 2;
  const int rows_per_cta = static_cast<int>((N + csize - 1) / csize);
  const int64_t rb = K / block_values(wtype) * block_bytes(wtype);
  const int64_t tchunks = (T + ST_TB - 1) / ST_TB;
  if (tchunks > 65535) return cudaErrorInvalidConfiguration;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((K + 255) / 256), static_cast<unsigned>(csize),
                     static_cast<unsigned>(tchunks));
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(csize);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;

  const uint8_t* w = static_cast<const uint8_t*>(W);
  const int n = static_cast<int>(N), k = static_cast<int>(K), t = static_cast<int>(T);
  switch (wtype) {
    case RG_F16: return cudaLaunchKernelEx(&cfg, smallt_kernel<RG_F16>, w, rb, n, k, dY, t, dX, beta, rows_per_cta);
    case RG_BF16: return cudaLaunchKernelEx(&cfg, smallt_kernel<RG_BF16>, w, rb, n, k, dY, t, dX, beta, rows_per_cta);
    case RG_Q8_0: return cudaLaunchKernelEx(&cfg, smallt_kernel<RG_Q8_0>, w, rb, n, k, dY, t, dX, beta, rows_per_cta);
    case RG_Q4_0: return cudaLaunchKernelEx(&cfg, smallt_kernel<RG_Q4_0>, w, rb, n, k, dY, t, dX, beta, rows_per_cta);
    case RG_Q4_K: return cudaLaunchKernelEx(&cfg, smallt_kernel<RG_Q4_K>, w, rb, n, k, dY, t, dX, beta, rows_per_cta);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rg
