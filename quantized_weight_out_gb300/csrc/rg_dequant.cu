// rg_dequant.cu - elementwise kernels: the bit-exact block decode to F32
// (rg_dequant), the dY -> fp16/bf16 operand conversion of the tensor-core
// path, the N == 0 scale, and the bounded-wait probe.
//
// The decode is the role of the converters that the llama.cpp fork's PR
// "cuda: out_prod accepts a quantized src0" (section "What") runs before its
// SGEMM (ggml_get_to_fp32_cuda); here it is a stand-alone call whose output
// must equal the format definition bit for bit.
#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {

// Bytes of a 256-value segment of a stored row (a whole number of blocks).
template <int WT>
__host__ __device__ constexpr int seg_bytes() {
  return 256 / block_values(WT) * block_bytes(WT);
}

// A warp per group of U rows x one 256-value segment: each lane fetches 16
// bytes of each of the U row segments with one 16-byte load (U loads in
// flight), the warp stages them in shared memory, and every warp-wide store
// writes 512 contiguous bytes of F32.  Segments run fastest along a row, so
// consecutive warps read and write consecutive memory.
constexpr int DQ_U = 4;
template <int WT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ W, int64_t N,
                                                      int64_t K, int64_t rb,
                                                      float* __restrict__ out) {
  constexpr int SB = seg_bytes<WT>();
  static_assert(SB % 16 == 0 && SB <= 512, "a segment is at most one 16-byte load per lane");
  __shared__ __align__(16) uint8_t buf[8][DQ_U][SB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t segs = (K + 255) >> 8;
  const int64_t groups = (N + DQ_U - 1) / DQ_U * segs;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * 8;
  for (int64_t g = blockIdx.x * 8LL + warp; g < groups; g += nwarps) {
    const int64_t rg = g / segs, sg = g - rg * segs;
    const int64_t n0 = rg * DQ_U;
    const int64_t boff = sg * SB + 16 * lane;  // this lane's bytes of the segment
    uint4 v[DQ_U];
#pragma unroll
    for (int u = 0; u < DQ_U; ++u) {
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (16 * lane < SB && n0 + u < N && boff < rb)
        v[u] = __ldcs(reinterpret_cast<const uint4*>(W + (n0 + u) * rb + boff));
    }
#pragma unroll
    for (int u = 0; u < DQ_U; ++u)
      if (16 * lane < SB) *reinterpret_cast<uint4*>(&buf[warp][u][16 * lane]) = v[u];
    __syncwarp();
    // lane l stores values 4l .. 4l+3 and 128+4l .. 128+4l+3 of the segment,
    // so each warp-wide store covers 512 contiguous bytes; it decodes the
    // 8-value groups holding them (lanes 2i and 2i+1 share a group)
    const int hl = lane & 1;
#pragma unroll
    for (int u = 0; u < DQ_U; ++u) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kin = 128 * h + 8 * (lane >> 1);  // the group, inside the segment
        const int64_t k = sg * 256 + kin + 4 * hl;
        if (n0 + u < N && k < K) {
          float x[8];
          decode8_f32<WT>(buf[warp][u], kin, x);
          __stcs(reinterpret_cast<float4*>(out + (n0 + u) * K + k),
                 hl ? make_float4(x[4], x[5], x[6], x[7]) : make_float4(x[0], x[1], x[2], x[3]));
        }
      }
    }
    __syncwarp();
  }
}

// Q6_K, Q3_K, Q2_K and MXFP4 rows (210, 110, 84 and 136 bytes per 256
// values) are not 16-byte aligned in general, and an F32 segment is wider
// than a warp's one 16-byte load per lane: one thread per 8 values, reading
// its bytes directly.
template <int WT>
__global__ void __launch_bounds__(256) dequant_bytes_kernel(const uint8_t* __restrict__ W, int64_t N,
                                                            int64_t K, int64_t rb,
                                                            float* __restrict__ out) {
  const int64_t gpr = K >> 3;  // 8-value groups per row
  const int64_t total = N * gpr;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = g / gpr;
    const int k0 = static_cast<int>(g - n * gpr) << 3;
    float v[8];
    decode8_f32<WT>(W + n * rb, k0, v);
    float4* o = reinterpret_cast<float4*>(out + n * K + k0);
    __stcs(o, make_float4(v[0], v[1], v[2], v[3]));
    __stcs(o + 1, make_float4(v[4], v[5], v[6], v[7]));
  }
}

// deq(W)^T as 16-bit [K, N] (rows ldo values apart): the dense operand of
// the forward mul_mat.  A CTA decodes 32 rows x 256 values of W exactly to
// F32 (warp w: rows w, w+8, ...; lane l: values 8l .. 8l+7), stages them in
// shared memory, and writes the 256 x 32 transposed tile rounded to fp16 (or
// bf16: BF16OUT), one output row of 32 values per warp step.
template <int WT, bool BF16OUT>
__global__ void __launch_bounds__(256) dequant_t16_kernel(const uint8_t* __restrict__ W, int64_t N,
                                                          int64_t K, int64_t rb,
                                                          uint16_t* __restrict__ out, int64_t ldo) {
  __shared__ __align__(16) float tile[32][260];  // [n][k], rows 16-byte aligned
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 256, n0 = static_cast<int64_t>(blockIdx.y) * 32;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int nl = warp + 8 * i;
    const int64_t n = n0 + nl, k = k0 + 8 * lane;
    float v[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if (n < N && k < K) decode8_f32<WT>(W + n * rb, static_cast<int>(k), v);
    float4* t = reinterpret_cast<float4*>(&tile[nl][8 * lane]);
    t[0] = make_float4(v[0], v[1], v[2], v[3]);
    t[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __syncthreads();
  for (int kl = warp; kl < 256; kl += 8) {
    const int64_t k = k0 + kl, n = n0 + lane;
    if (k < K && n < N) {
      const float x = tile[lane][kl];
      if constexpr (BF16OUT) {
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        out[k * ldo + n] = *reinterpret_cast<const uint16_t*>(&h);
      } else {
        const __half h = __float2half_rn(x);
        out[k * ldo + n] = *reinterpret_cast<const uint16_t*>(&h);
      }
    }
  }
}

cudaError_t launch_dequant_t16(int wtype, const void* W, int64_t N, int64_t K, bool bf16,
                               uint16_t* out, int64_t ldo, const DevInfo& dev, cudaStream_t stream) {
  (void)dev;
  const int64_t rb = K / block_values(wtype) * block_bytes(wtype);
  const int64_t gy = (N + 31) / 32;
  if (gy > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>((K + 255) / 256), static_cast<unsigned>(gy));
  const uint8_t* w = static_cast<const uint8_t*>(W);
  return with_wtype(wtype, cudaErrorInvalidValue, [&](auto wt) {
    constexpr int WT = decltype(wt)::value;
    if (bf16)
      dequant_t16_kernel<WT, true><<<grid, 256, 0, stream>>>(w, N, K, rb, out, ldo);
    else
      dequant_t16_kernel<WT, false><<<grid, 256, 0, stream>>>(w, N, K, rb, out, ldo);
    return counted(cudaGetLastError());
  });
}


cudaError_t launch_dequant(int wtype, const void* W, int64_t N, int64_t K, float* out,
                           const DevInfo& dev, cudaStream_t stream) {
  const int64_t rb = K / block_values(wtype) * block_bytes(wtype);
  const int grid = grid_for((N + DQ_U - 1) / DQ_U * ((K + 255) >> 8) * 32, 256, dev);
  const uint8_t* w = static_cast<const uint8_t*>(W);
  return with_wtype(wtype, cudaErrorInvalidValue, [&](auto wt) {
    constexpr int WT = decltype(wt)::value;
    if constexpr (WT == RG_Q6_K || WT == RG_F32 || WT == RG_Q2_K || WT == RG_Q3_K || WT == RG_MXFP4)
      dequant_bytes_kernel<WT><<<grid_for(N * (K >> 3), 256, dev), 256, 0, stream>>>(w, N, K, rb, out);
    else
      dequant_kernel<WT><<<grid, 256, 0, stream>>>(w, N, K, rb, out);
    return counted(cudaGetLastError());
  });
}

// dY [T, N] F32 -> [T, ld] 16-bit of mul * dY, round to nearest even (mul
// is 1 for dY itself: exact).  One thread per 8 values; 16-byte loads when
// every row is 16-byte aligned (N % 4 == 0).
template <bool BF16>
__global__ void __launch_bounds__(256) convert_dy_kernel(const float* __restrict__ dY, int64_t T,
                                                         int64_t N, int64_t ld, float mul,
                                                         uint16_t* __restrict__ out, int* status,
                                                         float* __restrict__ zero, int64_t zk,
                                                         int64_t zld) {
  pdl_launch_dependents();  // the tensor-core kernel may be scheduled now (it waits for us)
  const int64_t cpr = (N + 7) >> 3;
  const int64_t total = T * cpr;
  const bool vec = (N & 3) == 0;
  bool over = false;
  // eight values from row t, columns 8c on (zeros past N)
  auto load8 = [&](int64_t t, int64_t c, float (&v)[8]) {
    const int64_t n0 = c << 3;
    const float* src = dY + t * N + n0;
    if (vec && n0 + 8 <= N) {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(src));
      const float4 b = __ldcs(reinterpret_cast<const float4*>(src) + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (n0 + i < N) ? src[i] : 0.0f;
    }
  };
  auto store8 = [&](int64_t t, int64_t c, float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] *= mul;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      over |= overflowed16<BF16>(v[2 * i], w[i] & 0xFFFFu) | overflowed16<BF16>(v[2 * i + 1], w[i] >> 16);
    }
    *reinterpret_cast<uint4*>(out + t * ld + (c << 3)) = make_uint4(w[0], w[1], w[2], w[3]);
  };
  // a grid-stride walk over the groups of eight, two groups an iteration
  // with both groups' loads in flight; the row and column are carried from
  // one group to the next instead of divided out each time
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t st = stride / cpr, sr = stride - st * cpr;
  auto advance = [&](int64_t& t, int64_t& c) {
    t += st;
    c += sr;
    if (c >= cpr) {
      c -= cpr;
      ++t;
    }
  };
  int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  int64_t t = g / cpr, c = g - t * cpr;
  for (; g < total; g += 2 * stride) {
    int64_t t1 = t, c1 = c;
    advance(t1, c1);
    const bool two = g + stride < total;
    float v0[8], v1[8];
    load8(t, c, v0);
    if (two) load8(t1, c1, v1);
    store8(t, c, v0);
    if (two) store8(t1, c1, v1);
    t = t1;
    c = c1;
    advance(t, c);
  }
  if (over) report_range(status);
  // dX zeroed for a contraction split in two whose halves are both added into
  // it (T rows of zk values, zld apart; zk and zld multiples of 4)
  if (zero != nullptr) {
    const int64_t q4 = zk >> 2;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < T * q4;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int64_t t = g / q4;
      *reinterpret_cast<float4*>(zero + t * zld + 4 * (g - t * q4)) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  }
}

// Strided dY (a row stride other than N, or a column stride other than 1,
// e.g. dY given transposed): 32 x 32 tiles through shared memory; the reads
// run along whichever axis has unit stride (n when dy_n == 1, else t) and
// the 16-bit writes along n.
template <bool BF16>
__global__ void __launch_bounds__(256) convert_dy_tiled_kernel(const float* __restrict__ dY,
                                                               int64_t T, int64_t N, int64_t dy_t,
                                                               int64_t dy_n, int64_t ld,
                                                               uint16_t* __restrict__ out,
                                                               int* status) {
  pdl_launch_dependents();  // the tensor-core kernel may be scheduled now (it waits for us)
  __shared__ float tile[32][33];  // [t][n]
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 32, t0 = static_cast<int64_t>(blockIdx.y) * 32;
  const bool along_n = dy_n == 1 || dy_t != 1;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int a = ty + 8 * j;  // the slow index inside the tile
    const int64_t t = along_n ? t0 + a : t0 + tx, n = along_n ? n0 + tx : n0 + a;
    const float v = (t < T && n < N) ? __ldg(dY + t * dy_t + n * dy_n) : 0.0f;
    if (along_n)
      tile[a][tx] = v;
    else
      tile[tx][a] = v;
  }
  __syncthreads();
  bool over = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int a = ty + 8 * j;
    const int64_t t = t0 + a, n = n0 + tx;
    if (t < T && n < N) {
      uint16_t bits;
      if constexpr (BF16) {
        const __nv_bfloat16 h = __float2bfloat16_rn(tile[a][tx]);
        bits = *reinterpret_cast<const uint16_t*>(&h);
      } else {
        const __half h = __float2half_rn(tile[a][tx]);
        bits = *reinterpret_cast<const uint16_t*>(&h);
      }
      out[t * ld + n] = bits;
      over |= overflowed16<BF16>(tile[a][tx], bits);
    }
  }
  if (over) report_range(status);
}

cudaError_t launch_convert_dy(const float* dY, int64_t T, int64_t N, int64_t dy_t, int64_t dy_n,
                              int64_t ld, bool bf16, uint16_t* out, const DevInfo& dev,
                              cudaStream_t stream, float mul, float* zero, int64_t zk, int64_t zld) {
  if (zero != nullptr && (dy_n != 1 || dy_t != N || (zk & 3) || (zld & 3))) return cudaErrorInvalidValue;
  if (dy_n != 1 || dy_t != N) {
    if (mul != 1.0f) return cudaErrorInvalidValue;  // (strided rows are dY's alone)
    const int64_t gy = (T + 31) / 32;
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>((N + 31) / 32), static_cast<unsigned>(gy));
    if (bf16)
      convert_dy_tiled_kernel<true><<<grid, 256, 0, stream>>>(dY, T, N, dy_t, dy_n, ld, out,
                                                              dev.status);
    else
      convert_dy_tiled_kernel<false><<<grid, 256, 0, stream>>>(dY, T, N, dy_t, dy_n, ld, out,
                                                               dev.status);
    return counted(cudaGetLastError());
  }
  const int grid = grid_for(T * ((N + 7) >> 3), 256, dev);
  if (bf16)
    convert_dy_kernel<true><<<grid, 256, 0, stream>>>(dY, T, N, ld, mul, out, dev.status, zero, zk, zld);
  else
    convert_dy_kernel<false><<<grid, 256, 0, stream>>>(dY, T, N, ld, mul, out, dev.status, zero, zk, zld);
  return counted(cudaGetLastError());
}

__global__ void __launch_bounds__(256) scale_kernel(float* __restrict__ x, int64_t T, int64_t K,
                                                    int64_t ldx, float beta) {
  const int64_t count = T * K;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / K;
    float* p = x + t * ldx + (i - t * K);
    *p = beta == 0.0f ? 0.0f : beta * *p;
  }
}

cudaError_t launch_scale(float* dX, int64_t T, int64_t K, int64_t dx_t, float beta,
                         const DevInfo& dev, cudaStream_t stream) {
  scale_kernel<<<grid_for(T * K, 256, dev), 256, 0, stream>>>(dX, T, K, dx_t, beta);
  return counted(cudaGetLastError());
}

// One thread waits on an mbarrier that nothing arrives on.
__global__ void wait_probe_kernel(WaitCtl ctl) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(smem_addr(&bar), 0, ctl, &abort_flag);
  __syncthreads();
}

cudaError_t launch_wait_probe(const DevInfo& dev, unsigned long long limit_ns,
                              cudaStream_t stream) {
  WaitCtl ctl{dev.status, limit_ns};
  wait_probe_kernel<<<1, 32, 0, stream>>>(ctl);
  return counted(cudaGetLastError());
}

}  // namespace rg
