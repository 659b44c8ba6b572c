// rg_simt.cu - the full-F32 CUDA-core variant of the OUT_PROD
//   dX[t, k] = beta * dX[t, k] + sum_n dY[t, n] * deq(W)[n, k]:
// exact F32 decode and F32 FMA, accumulated in 32-row partial sums that are
// then added together (blocked summation keeps the F32 error far below the
// sequential worst case over N up to ~17k rows).
#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {

// ---------------------------------------------------------------------------
// simt32: one CTA per 64(t) x 64(k) output tile, 256 threads, 4x4 outputs each

constexpr int S32_TT = 64, S32_TK = 64, S32_TN = 32;

template <int WT>
__global__ void __launch_bounds__(256) simt32_kernel(const uint8_t* __restrict__ W, int64_t rb,
                                                     int N, int K,
                                                     const float* __restrict__ dY, int T,
                                                     float* __restrict__ dX, float beta,
                                                     int64_t dy_t, int64_t dy_n, int64_t dx_t) {
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
      ys[c][r] = (t < T && n < N) ? dY[t * dy_t + n * dy_n] : 0.0f;
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
      float* o = dX + t * dx_t + k;
      *o = beta != 0.0f ? fmaf(beta, *o, acc[i][j]) : acc[i][j];
    }
  }
}

cudaError_t launch_simt32(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, const Layout& lay, const DevInfo& dev,
                          cudaStream_t stream) {
  (void)dev;
  const int64_t rb = K / block_values(wtype) * block_bytes(wtype);
  const dim3 grid(static_cast<unsigned>((K + S32_TK - 1) / S32_TK),
                  static_cast<unsigned>((T + S32_TT - 1) / S32_TT));
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const int n = static_cast<int>(N), k = static_cast<int>(K), t = static_cast<int>(T);
  return with_wtype(wtype, cudaErrorInvalidValue, [&](auto wt) {
    simt32_kernel<decltype(wt)::value><<<grid, 256, 0, stream>>>(w, rb, n, k, dY, t, dX, beta,
                                                                 lay.dy_t, lay.dy_n, lay.dx_t);
    return counted(cudaGetLastError());
  });
}

}  // namespace rg
