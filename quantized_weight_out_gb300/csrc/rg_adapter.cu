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

// --- dY's 16-bit copy and U = dY . B in one pass over dY (rank <= 32) ---
//
// Block: 32 rows of dY, 256 threads, the contraction in chunks of 256 values
// of n, two chunks in flight: while the warps multiply chunk c out of shared
// memory, every thread's eight float4 of chunk c + 1 (a warp reads four rows
// x 128 contiguous bytes per instruction) are on their way into registers
// and B^T's chunk c + 1 into the other shared buffer (cp.async, zero-filled
// past N and past the rank).  A chunk's dY values are rounded to 16 bits
// once: written to the copy in HBM and to the MMA's tile.  Warp w multiplies
// rows 16 (w & 1).. by chunk quarter w >> 1 with mma.sync m16n8k16 (F32
// accumulation); the four quarters' U are added in a fixed order at the end
// and written, rounded to 16 bits, after dY's columns.  U is small: the
// legacy warp MMA is plenty for it.
constexpr int AD_TR = 32, AD_NC = 256, AD_LD = AD_NC + 8;  // (+8: conflict-free fragments)

template <int R8>
constexpr int adapter_smem_bytes() {
  constexpr int tiles = 2 * (AD_TR + R8) * AD_LD * 2;  // two buffers of dY's and B^T's chunk
  constexpr int red = 4 * AD_TR * R8 * 4;
  return tiles > red ? tiles : red;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float a, float b) {
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  if constexpr (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16 bytes global -> shared, the first `bytes` (0..16) from src, the rest zero
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// dY [T, N] F32 (rows 16-byte aligned when VEC) -> out [T, ld] 16-bit:
// columns [0, c_ad) dY (zeros from N on), [c_ad, c_ad + 64) U = dY . B for
// ranks < rank, zeros after.  bt: B^T [rank, ldb] 16-bit, ldb % 8 == 0.
template <bool BF16, bool VEC, int R8>
__global__ void __launch_bounds__(256) convert_dy_adapter_kernel(
    const float* __restrict__ dY, int64_t T, int64_t N, const uint16_t* __restrict__ bt,
    int64_t ldb, int rank, int64_t c_ad, int64_t ld, uint16_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t ad_smem[];
  // buffer b: dY's tile [AD_TR][AD_LD], then B^T's [R8][AD_LD]
  uint16_t* const buf0 = reinterpret_cast<uint16_t*>(ad_smem);
  constexpr int BUF = (AD_TR + R8) * AD_LD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * AD_TR;
  const int lr = tid >> 3, l8 = tid & 7;  // load role: row lr, float4 l8 + 8q
  const int64_t t = t0 + lr;
  const bool row_ok = t < T;
  const float* yrow = dY + t * N;
  const int mt = warp & 1, ks = warp >> 1;  // MMA role: rows 16 mt.., chunk quarter ks
  float acc[R8 / 8][4];
#pragma unroll
  for (int i = 0; i < R8 / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

  float4 v[8];
  auto load_y = [&](int64_t n0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int64_t n = n0 + (q * 8 + l8) * 4;
      if (VEC && row_ok && n + 4 <= N) {
        v[q] = __ldcs(reinterpret_cast<const float4*>(yrow + n));
      } else {
        v[q].x = (row_ok && n < N) ? yrow[n] : 0.0f;
        v[q].y = (row_ok && n + 1 < N) ? yrow[n + 1] : 0.0f;
        v[q].z = (row_ok && n + 2 < N) ? yrow[n + 2] : 0.0f;
        v[q].w = (row_ok && n + 3 < N) ? yrow[n + 3] : 0.0f;
      }
    }
  };
  auto load_b = [&](int64_t n0, uint16_t* sB) {
#pragma unroll
    for (int i = 0; i < R8 / 8; ++i) {
      const int e = tid + 256 * i;  // 32 sixteen-byte pieces a row
      const int jj = e >> 5, k = (e & 31) * 8;
      const int64_t n = n0 + k;
      const int64_t left = (jj < rank && n < N) ? (N - n) * 2 : 0;
      const int bytes = left >= 16 ? 16 : static_cast<int>(left);
      // a zero-byte copy still names a valid address: the row's start
      const uint16_t* src = bt + static_cast<int64_t>(jj < rank ? jj : 0) * ldb + (bytes ? n : 0);
      cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(sB + jj * AD_LD + k)), src, bytes);
    }
    cp_async_commit();
  };

  load_y(0);
  load_b(0, buf0 + AD_TR * AD_LD);
  int b = 0;
  for (int64_t n0 = 0; n0 < c_ad; n0 += AD_NC, b ^= 1) {
    uint16_t* const sY = buf0 + b * BUF;
    uint16_t* const sB = sY + AD_TR * AD_LD;
    // chunk n0: rounded once, to the copy and to the tile
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int c = (q * 8 + l8) * 4;
      const uint2 h = make_uint2(pack16<BF16>(v[q].x, v[q].y), pack16<BF16>(v[q].z, v[q].w));
      *reinterpret_cast<uint2*>(sY + lr * AD_LD + c) = h;
      if (row_ok && n0 + c < c_ad) *reinterpret_cast<uint2*>(out + t * ld + n0 + c) = h;
    }
    cp_async_wait_all();  // this thread's pieces of B^T's chunk n0
    __syncthreads();      // every tile of chunk n0 in place; chunk n0 - 256's reads done
    if (n0 + AD_NC < c_ad) {
      load_y(n0 + AD_NC);                         // in flight during the MMAs
      load_b(n0 + AD_NC, buf0 + (b ^ 1) * BUF + AD_TR * AD_LD);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int k0 = ks * 64 + kk * 16 + 2 * tq;
      const uint16_t* ya = sY + (mt * 16 + g) * AD_LD + k0;
      uint32_t a[4];
      a[0] = *reinterpret_cast<const uint32_t*>(ya);
      a[1] = *reinterpret_cast<const uint32_t*>(ya + 8 * AD_LD);
      a[2] = *reinterpret_cast<const uint32_t*>(ya + 8);
      a[3] = *reinterpret_cast<const uint32_t*>(ya + 8 * AD_LD + 8);
#pragma unroll
      for (int nt = 0; nt < R8 / 8; ++nt) {
        const uint16_t* bb = sB + (nt * 8 + g) * AD_LD + k0;
        mma_16816<BF16>(acc[nt], a, *reinterpret_cast<const uint32_t*>(bb),
                        *reinterpret_cast<const uint32_t*>(bb + 8));
      }
    }
  }
  __syncthreads();  // the last chunk's reads are done: the buffers become the reduction's
  // the four chunk quarters' sums, added in order
  float* red = reinterpret_cast<float*>(ad_smem);  // [4][AD_TR][R8]
#pragma unroll
  for (int nt = 0; nt < R8 / 8; ++nt) {
    const int r0 = mt * 16 + g, j = nt * 8 + 2 * tq;
    red[(ks * AD_TR + r0) * R8 + j] = acc[nt][0];
    red[(ks * AD_TR + r0) * R8 + j + 1] = acc[nt][1];
    red[(ks * AD_TR + r0 + 8) * R8 + j] = acc[nt][2];
    red[(ks * AD_TR + r0 + 8) * R8 + j + 1] = acc[nt][3];
  }
  __syncthreads();
  // 64 adapter columns a row, 8 per thread: 32 rows x 8 groups
  {
    const int r = tid >> 3, j0 = (tid & 7) * 8;
    const int64_t tr = t0 + r;
    if (tr < T) {
      float u[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int j = j0 + x;
        float sum = 0.0f;
        if (j < rank && j < R8) {
          sum = red[r * R8 + j];
#pragma unroll
          for (int q = 1; q < 4; ++q) sum += red[(q * AD_TR + r) * R8 + j];
        }
        u[x] = sum;
      }
      *reinterpret_cast<uint4*>(out + tr * ld + c_ad + j0) =
          make_uint4(pack16<BF16>(u[0], u[1]), pack16<BF16>(u[2], u[3]),
                     pack16<BF16>(u[4], u[5]), pack16<BF16>(u[6], u[7]));
    }
  }
}

template <bool BF16, bool VEC, int R8>
cudaError_t launch_cda(const float* dY, int64_t T, int64_t N, const uint16_t* bt, int64_t ldb,
                       int rank, int64_t c_ad, int64_t ld, uint16_t* out, cudaStream_t stream) {
  auto kern = convert_dy_adapter_kernel<BF16, VEC, R8>;
  constexpr int smem = adapter_smem_bytes<R8>();
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>((T + AD_TR - 1) / AD_TR), 256, smem, stream>>>(dY, T, N, bt, ldb,
                                                                              rank, c_ad, ld, out);
  return counted(cudaGetLastError());
}

template <bool BF16, bool VEC>
cudaError_t launch_cda_r(const float* dY, int64_t T, int64_t N, const uint16_t* bt, int64_t ldb,
                         int rank, int64_t c_ad, int64_t ld, uint16_t* out, cudaStream_t stream) {
  if (rank <= 8) return launch_cda<BF16, VEC, 8>(dY, T, N, bt, ldb, rank, c_ad, ld, out, stream);
  if (rank <= 16) return launch_cda<BF16, VEC, 16>(dY, T, N, bt, ldb, rank, c_ad, ld, out, stream);
  return launch_cda<BF16, VEC, 32>(dY, T, N, bt, ldb, rank, c_ad, ld, out, stream);
}

}  // namespace

cudaError_t launch_convert_dy_adapter(const float* dY, int64_t T, int64_t N, const uint16_t* bt,
                                      int64_t ldb, int64_t rank, int64_t ld, bool bf16,
                                      uint16_t* out, cudaStream_t stream) {
  if (rank < 1 || rank > kAdapterFusedRank || ldb % 8 || ld % 8 || T > 2147483647ll * AD_TR)
    return cudaErrorInvalidValue;
  const int64_t c_ad = (N + 63) / 64 * 64;
  const bool vec = (N & 3) == 0;
  const int r = static_cast<int>(rank);
  if (bf16)
    return vec ? launch_cda_r<true, true>(dY, T, N, bt, ldb, r, c_ad, ld, out, stream)
               : launch_cda_r<true, false>(dY, T, N, bt, ldb, r, c_ad, ld, out, stream);
  return vec ? launch_cda_r<false, true>(dY, T, N, bt, ldb, r, c_ad, ld, out, stream)
             : launch_cda_r<false, false>(dY, T, N, bt, ldb, r, c_ad, ld, out, stream);
}

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
