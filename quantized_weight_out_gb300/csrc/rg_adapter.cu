// rg_adapter.cu - the low-rank adapter's share of the input gradient,
//
//     dX += scale * (dY . B) . A,     A [rank, K], B [N, rank], F32,
//
// beside the resident base weight (llama.cpp fork PR "cuda: out_prod accepts
// a quantized src0", commit message: a LoRA training on a resident
// quantized base).  Two routes:
//   * tensor cores: U = dY . B runs as an OUT_PROD over B's 16-bit copy, and
//     adapter_pack_kernel writes U after dY's own columns in the 16-bit dY
//     copy, so the base product's kernel takes the adapter as extra
//     contraction chunks (A's rows come in by TMA, already scaled);
//   * F32 (the SIMT and small-T variants): adapter_down_kernel forms U in
//     partial sums over ranges of n, adapter_up_kernel adds
//     scale * U . A to dX after the base product.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {

namespace {

// out[t, c] for c in [c_gap, c_end) of each row: zeros before c_ad (the gap
// between dY's own columns and the chunk boundary), U[t, c - c_ad] rounded
// to 16 bits for c - c_ad < rank, zeros after.  Eight columns per thread
// (c_gap, c_ad and ld are multiples of 8).
template <bool BF16>
__global__ void __launch_bounds__(256) adapter_pack_kernel(const float* __restrict__ U,
                                                           int64_t ldu, int64_t T, int64_t rank,
                                                           int64_t c_gap, int64_t c_ad,
                                                           int64_t c_end, int64_t ld,
                                                           uint16_t* __restrict__ out) {
  const int64_t groups = (c_end - c_gap) >> 3;
  const int64_t total = T * groups;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = g / groups;
    const int64_t c0 = c_gap + ((g - t * groups) << 3);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t j = c0 + 2 * i + h - c_ad;
        v[h] = (j >= 0 && j < rank) ? U[t * ldu + j] : 0.0f;
      }
      if constexpr (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[0], v[1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __half2 h = __floats2half2_rn(v[0], v[1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
    *reinterpret_cast<uint4*>(out + t * ld + c0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// part[s, t, j] = sum over n in range s of dY[t, n] * B[n, j] (F32).  Block
// (t, 32 ranks, range s); warp w takes n = n0 + w, n0 + w + 8, ...; lane l
// rank j0 + l, so B's row segment is one coalesced read and dY's value a
// broadcast.  The eight warps' sums are added in a fixed order.
__global__ void __launch_bounds__(256) adapter_down_kernel(const float* __restrict__ dY,
                                                           const float* __restrict__ B,
                                                           int64_t N, int64_t rank,
                                                           int64_t n_per, int64_t T,
                                                           float* __restrict__ part) {
  __shared__ float red[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = blockIdx.x;
  const int64_t j = static_cast<int64_t>(blockIdx.y) * 32 + lane;
  const int64_t n0 = static_cast<int64_t>(blockIdx.z) * n_per;
  const int64_t n1 = n0 + n_per < N ? n0 + n_per : N;
  const float* y = dY + t * N;
  float acc = 0.0f;
  if (j < rank)
    for (int64_t n = n0 + warp; n < n1; n += 8) acc = fmaf(__ldg(y + n), __ldg(B + n * rank + j), acc);
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && j < rank) {
    float s = red[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) s += red[w][lane];
    part[(static_cast<int64_t>(blockIdx.z) * T + t) * rank + j] = s;
  }
}

// dX[t, k] += scale * sum_j U[t, j] * A[j, k], U[t, j] the n ranges' partial
// sums added in order.  Block (t, 1024 values of k); four k per thread.
__global__ void __launch_bounds__(256) adapter_up_kernel(const float* __restrict__ part,
                                                         int n_parts, int64_t T, int64_t rank,
                                                         const float* __restrict__ A, int64_t K,
                                                         float scale, float* __restrict__ dX,
                                                         int64_t dx_t) {
  extern __shared__ float u[];  // [rank]
  const int64_t t = blockIdx.x;
  for (int64_t j = threadIdx.x; j < rank; j += blockDim.x) {
    float s = part[t * rank + j];
    for (int p = 1; p < n_parts; ++p) s += part[(static_cast<int64_t>(p) * T + t) * rank + j];
    u[j] = s;
  }
  __syncthreads();
  const int64_t k = (static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x) * 4;
  if (k >= K) return;  // K is a multiple of 8: four values are all in or all out
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t j = 0; j < rank; ++j) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(A + j * K + k));
    const float uj = u[j];
    acc.x = fmaf(uj, a.x, acc.x);
    acc.y = fmaf(uj, a.y, acc.y);
    acc.z = fmaf(uj, a.z, acc.z);
    acc.w = fmaf(uj, a.w, acc.w);
  }
  float4* o = reinterpret_cast<float4*>(dX + t * dx_t + k);
  float4 d = *o;
  d.x = fmaf(scale, acc.x, d.x);
  d.y = fmaf(scale, acc.y, d.y);
  d.z = fmaf(scale, acc.z, d.z);
  d.w = fmaf(scale, acc.w, d.w);
  *o = d;
}

}  // namespace

cudaError_t launch_adapter_pack(const float* U, int64_t ldu, int64_t T, int64_t rank, int64_t N,
                                int64_t ld, bool bf16, uint16_t* out, const DevInfo& dev,
                                cudaStream_t stream) {
  const int64_t c_gap = (N + 7) / 8 * 8;  // dY's conversion wrote up to here
  const int64_t c_ad = (N + 63) / 64 * 64;
  const int64_t c_end = tc_adapter_cols(N, rank);
  const int grid = grid_for(T * ((c_end - c_gap) >> 3), 256, dev);
  if (bf16)
    adapter_pack_kernel<true><<<grid, 256, 0, stream>>>(U, ldu, T, rank, c_gap, c_ad, c_end, ld, out);
  else
    adapter_pack_kernel<false><<<grid, 256, 0, stream>>>(U, ldu, T, rank, c_gap, c_ad, c_end, ld, out);
  return counted(cudaGetLastError());
}

int adapter_down_parts(int64_t N, int64_t T, int64_t rank, const DevInfo& dev) {
  // about two blocks per SM, each range at least 256 values of n
  const int64_t blocks = T * ((rank + 31) / 32);
  int64_t parts = (2 * static_cast<int64_t>(dev.num_sms) + blocks - 1) / blocks;
  parts = std::min<int64_t>(parts, std::max<int64_t>(1, N / 256));
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(parts, 1024)));
}

cudaError_t launch_adapter_f32(const float* dY, int64_t N, int64_t T, const float* A,
                               const float* B, int64_t rank, int64_t K, float scale, float* dX,
                               int64_t dx_t, float* part, int n_parts, const DevInfo& dev,
                               cudaStream_t stream) {
  (void)dev;
  if (T > 2147483647ll || (rank + 31) / 32 > 65535 || (K + 1023) / 1024 > 65535)
    return cudaErrorInvalidConfiguration;
  const int64_t n_per = (N + n_parts - 1) / n_parts;
  adapter_down_kernel<<<dim3(static_cast<unsigned>(T), static_cast<unsigned>((rank + 31) / 32),
                             static_cast<unsigned>(n_parts)),
                        256, 0, stream>>>(dY, B, N, rank, n_per, T, part);
  cudaError_t e = counted(cudaGetLastError());
  if (e != cudaSuccess) return e;
  adapter_up_kernel<<<dim3(static_cast<unsigned>(T), static_cast<unsigned>((K + 1023) / 1024)),
                      256, static_cast<size_t>(rank) * 4, stream>>>(part, n_parts, T, rank, A, K,
                                                                    scale, dX, dx_t);
  return counted(cudaGetLastError());
}

}  // namespace rg
