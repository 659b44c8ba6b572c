// rg_tc.cu - fused decode + tcgen05 GEMM for
//   dX[t, k] = beta * dX[t, k] + sum_n dY[t, n] * deq(W)[n, k].
//
// The llama.cpp fork's PR "cuda: out_prod accepts a quantized src0" (section
// "What") reaches this product by writing deq(W) to a dense F32 pool copy and
// running cuBLAS SGEMM on it, and names a fused dequant-GEMM as the follow-on.
// This kernel is that fused GEMM, built for sm_103a:
//
//  * orientation: the tensor core computes D[k, t] = sum_n deq(W)[n, k] *
//    dY[t, n], i.e. A = deq(W)^T (M = 128 values of k, MN-major: k is
//    contiguous in a stored row) and B = dY^T (N = BT values of t, K-major:
//    n is contiguous in a row of dY).  The contraction runs over the rows n
//    of W, so each block's scale belongs to one contraction row and is folded
//    into the operand while decoding.
//  * one CTA per SM (persistent), warp-specialised:
//      warp 0      TMA producer: packed W rows (or F16/BF16 tiles, already
//                  in operand layout) and the 16-bit dY tile, per stage;
//      warp 1      tensor-memory owner and MMA issuer (one thread);
//      warps 4-7   decoders: packed blocks in shared memory -> fp16 operand
//                  tile in the 128-byte-swizzled layout the MMA reads;
//      warps 8-11  epilogue: tcgen05.ld -> beta*dX + acc -> global.
//  * F32 accumulators live in tensor memory, two per CTA (2 x BT columns), so
//    the epilogue of one tile overlaps the main loop of the next.
//  * every wait is bounded; a wait that gives up raises the CTA's abort flag,
//    records RG_ERR_TIMEOUT, and the CTA drains its in-flight copies and MMAs
//    before freeing tensor memory and returning.
#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {
namespace tc {

constexpr int BM = 128;           // k-values per tile (MMA M)
constexpr int BC = 64;            // contraction rows (n) per pipeline stage
constexpr int UMMA_K = 16;        // contraction rows per tcgen05.mma (16-bit inputs)
constexpr int NUM_THREADS = 384;  // 12 warps
constexpr int A_STAGE = BC * BM * 2;      // 16 KB: 64 rows of n x 128 fp16 values of k
constexpr int A_COLBLK = BC * 128;        // 8 KB: one 64-value column block of k

// Bytes of one packed W row that a 128-value tile loads (16-byte multiples):
// Q8_0 4 blocks = 136 B inside a 144 B window, Q4_0 72 B inside 80 B, Q4_K
// the whole 144 B super-block (its header holds every sub-block's scale).
template <int WT>
__host__ __device__ constexpr int p_row_bytes() {
  return WT == RG_Q8_0 ? 144 : WT == RG_Q4_0 ? 80 : WT == RG_Q4_K ? 144 : 0;
}

template <int WT, int BT>
struct Cfg {
  static constexpr bool QUANT = is_quant(WT);
  static constexpr bool BF = WT == RG_BF16;
  static constexpr int B_STAGE = BT * 128;  // BT rows of t x 64 16-bit values of n
  static constexpr int P_STAGE = QUANT ? BC * p_row_bytes<WT>() : 0;
  static constexpr int STAGE = A_STAGE + B_STAGE + ((P_STAGE + 1023) / 1024) * 1024;
  static constexpr int S = std::min(6, (200 * 1024) / STAGE);
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + S * A_STAGE;
  static constexpr int OFF_P = OFF_B + S * B_STAGE;
  static constexpr int OFF_BAR = OFF_P + S * ((P_STAGE + 1023) / 1024) * 1024;
  // barriers: full_tma[S], full_dec[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr int NUM_BARS = 3 * S + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024 B alignment
  static constexpr uint32_t TMA_BYTES = (QUANT ? P_STAGE : A_STAGE) + B_STAGE;
  static constexpr uint32_t TMEM_COLS = 2 * BT;
  static constexpr uint32_t IDESC = idesc_f16(BF, BM, BT, /*A MN-major*/ true, /*B*/ false);
  static_assert(S >= 2, "pipeline needs at least two stages");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// --- operand packing helpers ------------------------------------------------

__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
  return *reinterpret_cast<const __half2*>(&u);
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Bytes 0..3 of `b` are small unsigned integers u (< 256).  Returns the two
// fp16 values 1024 + u of bytes (lo_sel) packed as a half2: 0x64 is the high
// byte of 1024.0 in binary16, whose unit in the last place is 1, so the low
// byte lands in the mantissa exactly.
__device__ __forceinline__ __half2 bytes_to_h2_plus1024(uint32_t b, uint32_t sel) {
  return u32_as_h2(__byte_perm(b, 0x64646464u, sel));
}
constexpr uint32_t SEL_B01 = 0x5140;  // bytes 0,1 -> (lo half, hi half)
constexpr uint32_t SEL_B23 = 0x7362;  // bytes 2,3

// Store a 16-byte chunk (8 fp16 values of k = 8*cidx .. 8*cidx+7 of the tile)
// of contraction row n into the A stage: MN-major, 128-byte swizzle (chunk c
// of a 128-byte row r sits at position c ^ (r mod 8)); column blocks of 64
// values of k are A_COLBLK apart.
__device__ __forceinline__ void st_a_chunk(uint8_t* a, int n, int cidx, uint32_t x, uint32_t y,
                                           uint32_t z, uint32_t w) {
  const int jb = cidx >> 3, cc = cidx & 7;
  *reinterpret_cast<uint4*>(a + jb * A_COLBLK + n * 128 + ((cc ^ (n & 7)) << 4)) =
      make_uint4(x, y, z, w);
}

__device__ __forceinline__ uint32_t ld2_u16(const uint8_t* p) {  // 4 bytes at a 2-byte boundary
  const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
  return static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 16);
}

// Decode one stage: P holds BC packed rows of one 128-value tile (row stride
// p_row_bytes), A receives the fp16 operand.  dtid = 0..127.  kt = the tile's
// index along k (selects the byte offset inside the loaded window, or the
// half of the Q4_K super-block).
template <int WT>
__device__ __forceinline__ void decode_stage(const uint8_t* __restrict__ P, uint8_t* __restrict__ A,
                                             int dtid, int kt) {
  constexpr int PR = p_row_bytes<WT>();
  if constexpr (WT == RG_Q8_0) {
    // unit = (row n, block b of 4, quarter q of 4): 8 values -> one chunk
    const int off = (kt * 136) & 15;
    const __half2 bias = __float2half2_rn(1152.0f);  // 1024 + 128 (int8 sign bias)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int u = dtid + 128 * i;
      const int n = u >> 4, b = (u >> 2) & 3, q = u & 3;
      const uint8_t* blk = P + n * PR + off + 34 * b;
      const __half2 d2 = __half2half2(__ushort_as_half(ld_u16(blk)));
      const uint32_t w0 = ld2_u16(blk + 2 + 8 * q) ^ 0x80808080u;
      const uint32_t w1 = ld2_u16(blk + 6 + 8 * q) ^ 0x80808080u;
      const uint32_t o0 = h2_as_u32(__hmul2(__hsub2(bytes_to_h2_plus1024(w0, SEL_B01), bias), d2));
      const uint32_t o1 = h2_as_u32(__hmul2(__hsub2(bytes_to_h2_plus1024(w0, SEL_B23), bias), d2));
      const uint32_t o2 = h2_as_u32(__hmul2(__hsub2(bytes_to_h2_plus1024(w1, SEL_B01), bias), d2));
      const uint32_t o3 = h2_as_u32(__hmul2(__hsub2(bytes_to_h2_plus1024(w1, SEL_B23), bias), d2));
      st_a_chunk(A, n, 4 * b + q, o0, o1, o2, o3);
    }
  } else if constexpr (WT == RG_Q4_0) {
    // unit = (row n, block b of 4, half h): 16 values (low or high nibbles)
    const int off = (kt * 72) & 15;
    const __half2 bias = __float2half2_rn(1032.0f);  // 1024 + 8 (the Q4_0 zero point)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int u = dtid + 128 * i;
      const int n = u >> 3, b = (u >> 1) & 3, h = u & 1;
      const uint8_t* blk = P + n * PR + off + 18 * b;
      const __half2 d2 = __half2half2(__ushort_as_half(ld_u16(blk)));
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t w = ld2_u16(blk + 2 + 4 * j);
        w = (h ? (w >> 4) : w) & 0x0F0F0F0Fu;
        o[2 * j] = h2_as_u32(__hmul2(__hsub2(bytes_to_h2_plus1024(w, SEL_B01), bias), d2));
        o[2 * j + 1] = h2_as_u32(__hmul2(__hsub2(bytes_to_h2_plus1024(w, SEL_B23), bias), d2));
      }
      st_a_chunk(A, n, 4 * b + 2 * h, o[0], o[1], o[2], o[3]);
      st_a_chunk(A, n, 4 * b + 2 * h + 1, o[4], o[5], o[6], o[7]);
    }
  } else if constexpr (WT == RG_Q4_K) {
    // unit = (row n, chunk cl of 2, part p of 4): qs bytes 8p..8p+7 of chunk
    // c = 2*(kt & 1) + cl give 8 values of sub-block 2c (low nibbles) and 8
    // of sub-block 2c+1 (high nibbles).
    const int h2 = kt & 1;
    const __half2 magic = __float2half2_rn(1024.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int u = dtid + 128 * i;
      const int n = u >> 3, cl = (u >> 2) & 1, p = u & 3;
      const int c = 2 * h2 + cl;
      const uint8_t* sb = P + n * PR;
      const float d = f16_to_f32(ld_u16(sb));
      const float dmin = f16_to_f32(ld_u16(sb + 2));
      int sc0, m0, sc1, m1;
      q4k_scale_min(sb + 4, 2 * c, sc0, m0);
      q4k_scale_min(sb + 4, 2 * c + 1, sc1, m1);
      const __half2 ds0 = __float2half2_rn(d * static_cast<float>(sc0));
      const __half2 nm0 = __float2half2_rn(-(dmin * static_cast<float>(m0)));
      const __half2 ds1 = __float2half2_rn(d * static_cast<float>(sc1));
      const __half2 nm1 = __float2half2_rn(-(dmin * static_cast<float>(m1)));
      const uint2 qv = *reinterpret_cast<const uint2*>(sb + 16 + 32 * c + 8 * p);
      const uint32_t l0 = qv.x & 0x0F0F0F0Fu, l1 = qv.y & 0x0F0F0F0Fu;
      const uint32_t g0 = (qv.x >> 4) & 0x0F0F0F0Fu, g1 = (qv.y >> 4) & 0x0F0F0F0Fu;
      uint32_t lo[4], hi[4];
      lo[0] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(l0, SEL_B01), magic), ds0, nm0));
      lo[1] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(l0, SEL_B23), magic), ds0, nm0));
      lo[2] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(l1, SEL_B01), magic), ds0, nm0));
      lo[3] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(l1, SEL_B23), magic), ds0, nm0));
      hi[0] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(g0, SEL_B01), magic), ds1, nm1));
      hi[1] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(g0, SEL_B23), magic), ds1, nm1));
      hi[2] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(g1, SEL_B01), magic), ds1, nm1));
      hi[3] = h2_as_u32(__hfma2(__hsub2(bytes_to_h2_plus1024(g1, SEL_B23), magic), ds1, nm1));
      st_a_chunk(A, n, 8 * cl + p, lo[0], lo[1], lo[2], lo[3]);
      st_a_chunk(A, n, 8 * cl + 4 + p, hi[0], hi[1], hi[2], hi[3]);
    }
  }
}

// Byte offset (16-byte multiple) of the window a k-tile loads from a packed row.
template <int WT>
__device__ __forceinline__ int p_window_start(int kt) {
  if constexpr (WT == RG_Q8_0) return (kt * 136) & ~15;
  if constexpr (WT == RG_Q4_0) return (kt * 72) & ~15;
  return (kt >> 1) * 144;  // Q4_K: the whole super-block
}

// --- the kernel -----------------------------------------------------------------

template <int WT, int BT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    out_prod_tc_kernel(const __grid_constant__ CUtensorMap map_w,
                       const __grid_constant__ CUtensorMap map_y, float* __restrict__ dX,
                       float beta, int T, int K, int n_ktiles, int n_tiles, int n_chunks,
                       WaitCtl ctl, int inject_stall) {
  using C = Cfg<WT, BT>;
  constexpr int S = C::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sP = smem + C::OFF_P;
  const uint32_t bar0 = smem_addr(smem + C::OFF_BAR);
  auto full_tma = [&](int s) { return bar0 + 8u * s; };
  auto full_dec = [&](int s) { return bar0 + 8u * (S + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto acc_full = [&](int a) { return bar0 + 8u * (3 * S + a); };
  auto acc_empty = [&](int a) { return bar0 + 8u * (3 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (3 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_tma(s), 1);
      mbar_init(full_dec(s), 4);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&map_w);
    tma_prefetch_map(&map_y);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    int s = 0;
    uint32_t ph = 0;
    uint32_t pending = 0, pend_ph = 0;  // stages with a copy in flight, and its phase
    bool ok = true;
    bool skip_first = inject_stall != 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const int kt = tile % n_ktiles, tt = tile / n_ktiles;
      for (int c = 0; c < n_chunks; ++c) {
        ok = mbar_wait(empty(s), ph ^ 1u, ctl, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          if (skip_first) {
            skip_first = false;  // fault-injection: this stage never fills
          } else {
            mbar_arrive_expect_tx(full_tma(s), C::TMA_BYTES);
            if constexpr (C::QUANT) {
              tma_load_2d(smem_addr(sP + s * (C::STAGE - A_STAGE - C::B_STAGE)), &map_w,
                          full_tma(s), p_window_start<WT>(kt) / 4, c * BC);
            } else {
              tma_load_2d(smem_addr(sA + s * A_STAGE), &map_w, full_tma(s), kt * BM, c * BC);
              tma_load_2d(smem_addr(sA + s * A_STAGE + A_COLBLK), &map_w, full_tma(s),
                          kt * BM + 64, c * BC);
            }
            tma_load_2d(smem_addr(sB + s * C::B_STAGE), &map_y, full_tma(s), c * BC, tt * BT);
            pending |= 1u << s;
            pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
          }
        }
        __syncwarp();
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // drain: every copy this thread started must land before the CTA exits
      WaitCtl quick{ctl.status, ctl.limit_ns};
      volatile int no_abort = 0;
      for (int st = 0; st < S; ++st)
        if (pending & (1u << st)) (void)mbar_wait(full_tma(st), (pend_ph >> st) & 1u, quick, &no_abort);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int j = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++j) {
      const int a = j & 1;
      const uint32_t aph = (static_cast<uint32_t>(j) >> 1) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(acc_empty(a), aph ^ 1u, ctl, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * BT);
      for (int c = 0; c < n_chunks; ++c) {
        bool got = mbar_wait(full_tma(s), ph, ctl, abort_flag);
        if constexpr (C::QUANT) got = got && mbar_wait(full_dec(s), ph, ctl, abort_flag);
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_base = smem_addr(sA + s * A_STAGE);
          const uint32_t b_base = smem_addr(sB + s * C::B_STAGE);
#pragma unroll
          for (int kk = 0; kk < BC / UMMA_K; ++kk) {
            // A: MN-major, k-column blocks 8 KB apart (LBO), 8-row groups of n 1 KB apart (SBO)
            const uint64_t ad = sdesc_sw128(a_base + kk * (UMMA_K * 128), A_COLBLK, 1024);
            // B: K-major, 16 values of n = 32 bytes along the swizzled row; 8-row groups 1 KB apart
            const uint64_t bd = sdesc_sw128(b_base + kk * (UMMA_K * 2), 16, 1024);
            tc_mma_f16(d_tmem, ad, bd, C::IDESC, (c | kk) != 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
        }
        __syncwarp();
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(acc_full(a));
      __syncwarp();
    }
    if (!ok && lane == 0) {
      // drain: all MMAs this thread issued complete before tensor memory is freed
      tc_commit(drain_bar);
      volatile int no_abort = 0;
      (void)mbar_wait(drain_bar, 0, ctl, &no_abort);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- decoders ----------------
    if constexpr (C::QUANT) {
      const int dtid = threadIdx.x - 128;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int kt = tile % n_ktiles;
        for (int c = 0; c < n_chunks; ++c) {
          ok = __all_sync(0xffffffffu, mbar_wait(full_tma(s), ph, ctl, abort_flag));
          if (!ok) break;
          decode_stage<WT>(sP + s * (C::STAGE - A_STAGE - C::B_STAGE), sA + s * A_STAGE, dtid, kt);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_dec(s));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp >= 8) {
    // ---------------- epilogue ----------------
    const int eq = warp & 3;  // TMEM lanes 32*eq .. 32*eq+31
    bool ok = true;
    int j = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++j) {
      const int kt = tile % n_ktiles, tt = tile / n_ktiles;
      const int a = j & 1;
      const uint32_t aph = (static_cast<uint32_t>(j) >> 1) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(acc_full(a), aph, ctl, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int k = kt * BM + 32 * eq + lane;
      const bool kin = k < K;
#pragma unroll 1
      for (int cb = 0; cb < BT / 32; ++cb) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * eq) << 16) +
                               static_cast<uint32_t>(a * BT + 32 * cb),
                           r);
        const int tb = tt * BT + 32 * cb;
        if (kin) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int t = tb + i;
            if (t < T) {
              float* o = dX + static_cast<int64_t>(t) * K + k;
              const float v = __uint_as_float(r[i]);
              *o = beta != 0.0f ? fmaf(beta, *o, v) : v;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(a));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace tc

// --- host side ------------------------------------------------------------------

int64_t tc_dy16_ld(int64_t N) { return (N + 7) / 8 * 8; }

TcPlan plan_tc(int64_t N, int64_t K, int64_t T, const DevInfo& dev) {
  TcPlan p{};
  p.n_ktiles = static_cast<int>((K + tc::BM - 1) / tc::BM);
  p.n_chunks = static_cast<int>((N + tc::BC - 1) / tc::BC);
  const int64_t tiles256 = p.n_ktiles * ((T + 255) / 256);
  p.bt = tiles256 >= dev.num_sms ? 256 : 128;
  p.n_ttiles = static_cast<int>((T + p.bt - 1) / p.bt);
  const int64_t tiles = static_cast<int64_t>(p.n_ktiles) * p.n_ttiles;
  p.grid = static_cast<int>(std::min<int64_t>(tiles, dev.num_sms));
  return p;
}

template <int WT, int BT>
static cudaError_t launch_tc_t(const CUtensorMap& mw, const CUtensorMap& my, float* dX,
                               float beta, int T, int K, const TcPlan& p, const DevInfo& dev,
                               cudaStream_t stream, int inject) {
  using C = tc::Cfg<WT, BT>;
  auto kern = tc::out_prod_tc_kernel<WT, BT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  WaitCtl ctl{dev.status, dev.wait_limit_ns};
  const int n_tiles = p.n_ktiles * p.n_ttiles;
  kern<<<p.grid, tc::NUM_THREADS, C::SMEM_BYTES, stream>>>(mw, my, dX, beta, T, K, p.n_ktiles,
                                                          n_tiles, p.n_chunks, ctl, inject);
  return cudaGetLastError();
}

template <int WT>
static cudaError_t launch_tc_w(const CUtensorMap& mw, const CUtensorMap& my, float* dX,
                               float beta, int T, int K, const TcPlan& p, const DevInfo& dev,
                               cudaStream_t stream, int inject) {
  if (p.bt == 256) return launch_tc_t<WT, 256>(mw, my, dX, beta, T, K, p, dev, stream, inject);
  return launch_tc_t<WT, 128>(mw, my, dX, beta, T, K, p, dev, stream, inject);
}

cudaError_t launch_tc(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                      int64_t ld_dy16, int64_t T, float* dX, float beta, const DevInfo& dev,
                      cudaStream_t stream, int inject_stall) {
  const TcPlan p = plan_tc(N, K, T, dev);
  CUtensorMap mw, my;
  CUresult r;
  if (is_quant(wtype)) {
    const uint64_t rb = static_cast<uint64_t>(K / block_values(wtype) * block_bytes(wtype));
    const uint32_t box_bytes = wtype == RG_Q4_0 ? 80u : 144u;
    r = encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rb / 4, static_cast<uint64_t>(N), rb,
                     box_bytes / 4, tc::BC, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    r = encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, W, static_cast<uint64_t>(K),
                     static_cast<uint64_t>(N), static_cast<uint64_t>(K) * 2, 64, tc::BC,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  r = encode_tiled(&my, CU_TENSOR_MAP_DATA_TYPE_UINT16, dy16, static_cast<uint64_t>(N),
                   static_cast<uint64_t>(T), static_cast<uint64_t>(ld_dy16) * 2, tc::BC,
                   static_cast<uint32_t>(p.bt), CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int t = static_cast<int>(T), k = static_cast<int>(K);
  switch (wtype) {
    case RG_F16: return launch_tc_w<RG_F16>(mw, my, dX, beta, t, k, p, dev, stream, inject_stall);
    case RG_BF16: return launch_tc_w<RG_BF16>(mw, my, dX, beta, t, k, p, dev, stream, inject_stall);
    case RG_Q8_0: return launch_tc_w<RG_Q8_0>(mw, my, dX, beta, t, k, p, dev, stream, inject_stall);
    case RG_Q4_0: return launch_tc_w<RG_Q4_0>(mw, my, dX, beta, t, k, p, dev, stream, inject_stall);
    case RG_Q4_K: return launch_tc_w<RG_Q4_K>(mw, my, dX, beta, t, k, p, dev, stream, inject_stall);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rg
