// rg_tc_kernel.cuh - the fused decode + tcgen05 GEMM kernel and its launch
// templates, shared by rg_tc.cu (no adapter) and rg_tc_ad.cu (an adapter
// rides along as extra contraction chunks): two translation units, so the
// two builds of every instance compile in parallel.
//
// The kernel computes
//   dX[t, k] = beta * dX[t, k] + sum_n dY[t, n] * deq(W)[n, k].
//
// The llama.cpp fork's PR "cuda: out_prod accepts a quantized src0" (section
// "What") reaches this product by writing deq(W) to a dense F32 pool copy and
// running cuBLAS SGEMM on it, and names a fused dequant-GEMM as the follow-on.
// This kernel is that fused GEMM, built for sm_103a.
//
//  * Orientation: the tensor core computes D[k, t] = sum_n deq(W)[n, k] *
//    dY[t, n], i.e. A = deq(W)^T (M along k, MN-major: k is contiguous in a
//    stored row) and B = dY^T (N along t, K-major: n is contiguous in a row
//    of dY).  The contraction runs over the rows n of W, so every block scale
//    belongs to one contraction row and is folded into the operand while
//    decoding; it could not be applied in the epilogue.
//  * CG = 2 (the main configuration): a cluster of two CTAs on the two SMs of
//    a pair computes a 256(k) x 256(t) tile with tcgen05.mma.cta_group::2
//    (M = 256, N = 256).  Each CTA decodes its own 128 values of k into its
//    A half and TMA-loads its own 128 rows of t into its B half; the even CTA
//    issues the MMAs and commits to both CTAs' barriers.  Per SM this halves
//    the dY operand traffic of a one-CTA 128 x 256 tile.
//    CG = 1: one CTA, M = 128, N = 128, for shapes with few tiles.
//  * Persistent, warp-specialised, 512 threads per CTA:
//      warp 0      TMA producer (packed W window or F16/BF16 operand tile, and
//                  the 16-bit dY tile, per stage of 64 contraction rows);
//      warp 1      tensor-memory owner and (even CTA) MMA issuer;
//      warps 2-11  decoders, two per stage slot: packed blocks -> fp16
//                  operand tile, 128-byte swizzled, MN-major; a follower's
//                  warps arrive on the issuing CTA's barrier (idle for F16/BF16);
//      warps 12-15 epilogue: tcgen05.ld -> beta*dX + acc -> global.
//  * F32 accumulators in tensor memory, two per CTA (2 x BT columns): the
//    epilogue of one tile overlaps the main loop of the next.
//  * Every wait is bounded; a wait that gives up raises the CTA's abort flag
//    and records RG_ERR_TIMEOUT, and the CTA drains its in-flight copies and
//    MMAs before freeing tensor memory and returning.
#pragma once

#include <algorithm>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {
namespace tc {

constexpr int BM = 128;           // values of k per CTA (A rows of M per CTA)
constexpr int BC = 64;            // contraction rows (n) per pipeline stage
constexpr int UMMA_K = 16;        // contraction rows per tcgen05.mma (16-bit inputs)
constexpr int B_ROWS = 128;       // rows of t per CTA in a B stage
constexpr int NUM_THREADS = 512;  // 16 warps
constexpr int DEC_WARP0 = 2, DEC_WARPS = 10, EPI_WARP0 = 12;
constexpr int A_STAGE = BC * BM * 2;      // 16 KB: 64 rows of n x 128 fp16 values of k
constexpr int A_COLBLK = BC * 128;        // 8 KB: one 64-value column block of k
constexpr int B_STAGE = B_ROWS * 128;     // 16 KB: 128 rows of t x 64 16-bit values of n
constexpr int SMEM_BUDGET = 224 * 1024;

// Bytes of one packed W row that a 128-value tile loads (16-byte multiples):
// Q8_0 4 blocks = 136 B inside a 144 B window, Q4_0 72 B inside 80 B, Q4_1
// exactly 80 B, Q5_0 88 B and Q5_1 96 B inside 112 B (the wider row stride
// puts eight consecutive rows in distinct shared-memory bank groups), Q4_K
// and Q5_K the whole super-block (its header holds every sub-block's scale),
// Q6_K the whole 210-byte super-block inside a 240-byte window that starts at
// the 16-byte grain before it (0..14 bytes in; 15 chunks keep eight rows in
// distinct bank groups), MXFP4 four 17-byte blocks (68 B, 0, 4, 8 or 12
// bytes into the grain) inside 112 B (7 chunks: distinct bank groups), NVFP4
// two 36-byte blocks (72 B, 0 or 8 bytes in) inside 80 B (as Q4_0).
template <int WT>
__host__ __device__ constexpr int p_row_bytes() {
  return WT == RG_Q8_0   ? 144
         : WT == RG_Q4_0 ? 80
         : WT == RG_Q4_K ? 144
         : WT == RG_Q4_1 ? 80
         : WT == RG_Q5_0 ? 112
         : WT == RG_Q5_1 ? 112
         : WT == RG_Q5_K ? 176
         : WT == RG_Q6_K ? 240
         : WT == RG_Q3_K ? 128
         : WT == RG_Q2_K ? 96
         : WT == RG_MXFP4 ? 112
         : WT == RG_NVFP4 ? 80
                         : 0;
}

// Bytes of one packed W row that the forward's 64-value stage copies: Q4_K
// the 16-byte header and the chunk's 32 nibble bytes (two copies into two
// regions of the stage); Q8_0 its two 34-byte blocks inside an 80-byte
// window (0, 4, 8 or 12 bytes in); Q6_K three windows that each start at
// the same offset (0..14) into their first 16-byte grain: the half's 64
// bytes of low bits (80), its 32 bytes of high bits (48), and the 16
// scales and d (32); Q3_K and Q2_K their 128-value window, widened to an odd
// number of 16-byte grains (144, 112: the forward decoders' 32-bit loads of
// one row a lane then fall in 8 bank groups, not 1 or 4); the other types
// their whole 128-value window.
template <int WT>
__host__ __device__ constexpr int p_fwd_row_bytes() {
  return WT == RG_Q4_K ? 48 : WT == RG_Q8_0 ? 80 : WT == RG_Q6_K ? 80 + 48 + 32
         : WT == RG_Q3_K ? 144 : WT == RG_Q2_K ? 112 : p_row_bytes<WT>();
}
// The forward's Q6_K windows, bytes a row: low bits, high bits, scales and d.
constexpr int Q6F_A = 80, Q6F_H = 48, Q6F_S = 32;

template <int WT, int CG, int BT, bool FWD = false>
struct Cfg {
  static constexpr bool QUANT = is_quant(WT);
  static constexpr bool BF = WT == RG_BF16;
  // rows of W in a packed-window stage: the OUT_PROD's 64 contraction rows,
  // or the forward's 128 output rows (FWD: the contraction runs along the rows)
  static constexpr int P_ROWS = FWD ? 2 * BC : BC;
  static constexpr int P_ROW = FWD ? p_fwd_row_bytes<WT>() : p_row_bytes<WT>();
  static constexpr int P_STAGE = QUANT ? ((P_ROWS * P_ROW + 1023) / 1024) * 1024 : 0;
  static constexpr int STAGE = A_STAGE + B_STAGE + P_STAGE;
  // quantized: five slots (Q6_K four; fewer when they do not fit), each
  // decoded by two warps; F16/BF16: as deep as fits
  static constexpr int S_MAX = QUANT ? (WT == RG_Q6_K && !FWD ? 4 : 5) : 8;
  // the epilogue's staging for its bulk stores: per epilogue warp two boxes
  // of EPI_ROWS rows of t by 32 values of k, F32 (16 KB for 16 rows); in the
  // forward, boxes of 8 rows where the 8 KB they save buys one more stage
  // slot (Q8_0's forward 4 -> 5 slots: 14 % faster; the OUT_PROD's Q5_K
  // measured 9 % slower with the same trade, so it keeps 16 rows)
  static constexpr int slots_with(int epi_bytes) { return std::min(S_MAX, (SMEM_BUDGET - epi_bytes) / STAGE); }
  static constexpr int EPI_ROWS =
      FWD && slots_with(4 * 2 * 8 * 32 * 4) > slots_with(4 * 2 * 16 * 32 * 4) ? 8 : 16;
  static constexpr int EPI_BYTES = 4 * 2 * EPI_ROWS * 32 * 4;
  static constexpr int S = slots_with(EPI_BYTES);
  static constexpr int WARPS_PER_SLOT = QUANT ? 2 : 0;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + S * A_STAGE;
  static constexpr int OFF_P = OFF_B + S * B_STAGE;
  static constexpr int OFF_EPI = OFF_P + S * P_STAGE;
  static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
  // barriers: full_p, full_ab, full_dec, empty (S each), acc_full[2],
  // acc_empty[2], drain
  static constexpr int NUM_BARS = 4 * S + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024 B alignment
  static constexpr uint32_t P_BYTES = QUANT ? P_ROWS * P_ROW : 0;
  // operand bytes of one stage over the whole pair (B halves, and A for F16/BF16)
  static constexpr uint32_t AB_BYTES_PAIR = CG * (B_STAGE + (QUANT ? 0 : A_STAGE));
  static constexpr uint32_t TMEM_COLS = 2 * BT;
  static constexpr int MMA_M = BM * CG;
  // A: the OUT_PROD's deq(W)^T is MN-major (k along a stored row is M); the
  // forward's deq(W) is K-major (the row is the contraction)
  static constexpr uint32_t IDESC = idesc_f16(BF, MMA_M, BT, /*A MN-major*/ !FWD, /*B*/ false);
  // the slot's decoder warps of every CTA of the pair
  static constexpr uint32_t FULL_DEC_COUNT = (QUANT ? WARPS_PER_SLOT : 1) * CG;
  static constexpr uint32_t ACC_EMPTY_COUNT = 4 * CG;
  static_assert(BT / CG == B_ROWS, "each CTA holds 128 rows of t in a B stage");
  static_assert(S >= 3, "pipeline depth");
  static_assert(!QUANT || S * WARPS_PER_SLOT <= DEC_WARPS, "decoder warps cover the slots");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// --- operand packing helpers ------------------------------------------------

__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
  return *reinterpret_cast<const __half2*>(&u);
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Bytes of `b` are small unsigned integers u (< 256).  Returns the two fp16
// values 1024 + u of the bytes `sel` picks, packed as a half2: 0x64 is the
// high byte of 1024.0 in binary16, whose unit in the last place is 1, so the
// byte lands in the mantissa exactly.
__device__ __forceinline__ __half2 bytes_plus1024(uint32_t b, uint32_t sel) {
  return u32_as_h2(__byte_perm(b, 0x64646464u, sel));
}
constexpr uint32_t SEL_B01 = 0x5140;  // bytes 0,1 -> (lo half, hi half)
constexpr uint32_t SEL_B23 = 0x7362;  // bytes 2,3

// Four bytes x = 4 values each (q + bias already unsigned) -> two half2 of
// (1024 + u - off) * d.
__device__ __forceinline__ void four_scaled(uint32_t u, __half2 off, __half2 d, uint32_t& o0,
                                            uint32_t& o1) {
  o0 = h2_as_u32(__hmul2(__hsub2(bytes_plus1024(u, SEL_B01), off), d));
  o1 = h2_as_u32(__hmul2(__hsub2(bytes_plus1024(u, SEL_B23), off), d));
}
// Four nibble values in bytes -> two half2 of q * ds + nm (Q4_K).
__device__ __forceinline__ void four_affine(uint32_t u, __half2 magic, __half2 ds, __half2 nm,
                                            uint32_t& o0, uint32_t& o1) {
  o0 = h2_as_u32(__hfma2(__hsub2(bytes_plus1024(u, SEL_B01), magic), ds, nm));
  o1 = h2_as_u32(__hfma2(__hsub2(bytes_plus1024(u, SEL_B23), magic), ds, nm));
}

// Store a 16-byte chunk (8 fp16 values of k = 8*cidx .. 8*cidx+7 of the tile)
// of contraction row n into the A stage: MN-major, 128-byte swizzle (chunk c
// of a 128-byte row r sits at position c ^ (r mod 8)); column blocks of 64
// values of k are A_COLBLK apart.  Lanes that store the same cidx for eight
// consecutive rows hit eight distinct 16-byte bank groups.
__device__ __forceinline__ void st_a_chunk(uint8_t* a, int n, int cidx, uint32_t x, uint32_t y,
                                           uint32_t z, uint32_t w) {
  const int jb = cidx >> 3, cc = cidx & 7;
  *reinterpret_cast<uint4*>(a + jb * A_COLBLK + n * 128 + ((cc ^ (n & 7)) << 4)) =
      make_uint4(x, y, z, w);
}

// Words of a packed row held in registers: chunks of 16 bytes from C0 on.
// word_at(x) = the 4 bytes at byte offset x from the first loaded chunk.
template <int NW>
struct RowWords {
  uint32_t w[NW];
  __device__ __forceinline__ uint32_t word_at(int x) const {
    const int i = x >> 2, sh = x & 3;
    return sh == 0 ? w[i] : __funnelshift_r(w[i], w[i + 1], 8 * sh);
  }
};
template <int C0, int C1>
__device__ __forceinline__ RowWords<4 * (C1 - C0 + 1)> load_chunks(const uint8_t* row) {
  RowWords<4 * (C1 - C0 + 1)> r;
#pragma unroll
  for (int c = 0; c <= C1 - C0; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * (C0 + c));
    r.w[4 * c] = v.x;
    r.w[4 * c + 1] = v.y;
    r.w[4 * c + 2] = v.z;
    r.w[4 * c + 3] = v.w;
  }
  return r;
}

// Q8_0 block starting at byte S of a row window: fp16 d, 32 int8 q.
// Writes its 32 values as chunks 4b .. 4b+3 of row n.
template <int S>
__device__ __forceinline__ void dec_q8_block(const uint8_t* row, uint8_t* A, int n, int b) {
  constexpr int C0 = S / 16;
  constexpr int C1 = (S + ((S & 3) == 0 ? 35 : 33)) / 16;
  const auto r = load_chunks<C0, C1>(row);
  constexpr int X = S - 16 * C0;
  const __half2 d2 = __half2half2(__ushort_as_half(static_cast<uint16_t>(r.word_at(X) & 0xFFFFu)));
  const __half2 off = __float2half2_rn(1152.0f);  // 1024 + 128 (int8 sign bias)
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t o[4];
    four_scaled(r.word_at(X + 2 + 8 * q) ^ 0x80808080u, off, d2, o[0], o[1]);
    four_scaled(r.word_at(X + 6 + 8 * q) ^ 0x80808080u, off, d2, o[2], o[3]);
    st_a_chunk(A, n, 4 * b + q, o[0], o[1], o[2], o[3]);
  }
}

// Q4_0 block starting at byte S: fp16 d, 16 bytes of nibbles (low = value j,
// high = value j + 16).  Writes chunks 4b .. 4b+3 of row n.
template <int S>
__device__ __forceinline__ void dec_q4_0_block(const uint8_t* row, uint8_t* A, int n, int b) {
  constexpr int C0 = S / 16;
  constexpr int C1 = (S + ((S & 3) == 0 ? 19 : 17)) / 16;
  const auto r = load_chunks<C0, C1>(row);
  constexpr int X = S - 16 * C0;
  const __half2 d2 = __half2half2(__ushort_as_half(static_cast<uint16_t>(r.word_at(X) & 0xFFFFu)));
  const __half2 off = __float2half2_rn(1032.0f);  // 1024 + 8 (the Q4_0 zero point)
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = r.word_at(X + 2 + 4 * j);
    four_scaled(w & 0x0F0F0F0Fu, off, d2, lo[2 * j], lo[2 * j + 1]);
    four_scaled((w >> 4) & 0x0F0F0F0Fu, off, d2, hi[2 * j], hi[2 * j + 1]);
  }
  st_a_chunk(A, n, 4 * b, lo[0], lo[1], lo[2], lo[3]);
  st_a_chunk(A, n, 4 * b + 1, lo[4], lo[5], lo[6], lo[7]);
  st_a_chunk(A, n, 4 * b + 2, hi[0], hi[1], hi[2], hi[3]);
  st_a_chunk(A, n, 4 * b + 3, hi[4], hi[5], hi[6], hi[7]);
}

// Four E2M1 codes in the low nibbles of the bytes of x (high nibbles zero)
// -> two half2 (the codes of bytes 0, 1 and 2, 3), exact: a byte lookup
// gives each magnitude's fp16 high byte (every low byte is zero), the code's
// sign bit becomes that byte's top bit.
__device__ __forceinline__ void e2m1x4_f16(uint32_t x, uint32_t& o01, uint32_t& o23) {
  const uint32_t t = x & 0x07070707u;
  const uint32_t u = t | (t >> 4);
  const uint32_t sel = (u & 0xFFu) | ((u >> 8) & 0xFF00u);  // nibble k: magnitude of byte k
  // fp16 high bytes of 0, 0.5, 1, 1.5 | 2, 3, 4, 6
  const uint32_t hb = __byte_perm(0x3E3C3800u, 0x46444240u, sel) | ((x & 0x08080808u) << 4);
  o01 = __byte_perm(hb, 0u, 0x1404);
  o23 = __byte_perm(hb, 0u, 0x3424);
}

// MXFP4 block B of a 128-value tile whose blocks start o = 0, 4, 8 or 12
// bytes into the row window (a run-time value: one code path for every
// offset, so the decoders' instructions stay few).  Block B begins at byte
// o + 17B: its 16-byte chunk and the next are loaded, the five words from
// the block's own word on are selected by (o + 17B) mod 16 / 4 (the shift
// inside a word, B mod 4, is fixed).  Writes its 32 values,
// E2M1(q) * 2^(e - 127) rounded once to fp16, as chunks 4B .. 4B+3 of row n.
template <int B>
__device__ __forceinline__ void dec_mxfp4_block(const uint8_t* row, uint8_t* A, int n, int o) {
  constexpr int SH = B & 3;  // (o + 17B) mod 4
  const int S = o + 17 * B;
  const uint4 c0 = *reinterpret_cast<const uint4*>(row + (S & ~15));
  const uint4 c1 = *reinterpret_cast<const uint4*>(row + (S & ~15) + 16);
  const uint32_t q[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const int j0 = (S & 15) >> 2;  // 0..3: the block's first word in q
  uint32_t w[5];
#pragma unroll
  for (int k = 0; k < 5; ++k)
    w[k] = j0 == 0 ? q[k] : j0 == 1 ? q[k + 1] : j0 == 2 ? q[k + 2] : q[k + 3];
  const uint32_t e = (w[0] >> (8 * SH)) & 0xFFu;
  const __half2 sc = __float2half2_rn(e8m0_f32(e));
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // qs word j: bytes SH + 1 + 4j .. + 3 of w
    constexpr int X = SH + 1;
    const uint32_t v = (X & 3) == 0 ? w[(X >> 2) + j]
                                    : __funnelshift_r(w[(X >> 2) + j], w[(X >> 2) + j + 1], 8 * (X & 3));
    uint32_t a0, a1, b0, b1;
    e2m1x4_f16(v & 0x0F0F0F0Fu, a0, a1);
    e2m1x4_f16((v >> 4) & 0x0F0F0F0Fu, b0, b1);
    lo[2 * j] = h2_as_u32(__hmul2(u32_as_h2(a0), sc));
    lo[2 * j + 1] = h2_as_u32(__hmul2(u32_as_h2(a1), sc));
    hi[2 * j] = h2_as_u32(__hmul2(u32_as_h2(b0), sc));
    hi[2 * j + 1] = h2_as_u32(__hmul2(u32_as_h2(b1), sc));
  }
  st_a_chunk(A, n, 4 * B, lo[0], lo[1], lo[2], lo[3]);
  st_a_chunk(A, n, 4 * B + 1, lo[4], lo[5], lo[6], lo[7]);
  st_a_chunk(A, n, 4 * B + 2, hi[0], hi[1], hi[2], hi[3]);
  st_a_chunk(A, n, 4 * B + 3, hi[4], hi[5], hi[6], hi[7]);
}

// Two E4M3 bytes (bits 0-7 and 8-15 of w) -> their fp16 pair, exactly: the
// seven magnitude bits shifted into an fp16's exponent and mantissa fields
// give 2^(e-15) (1 + m/8), or for e = 0 the fp16 subnormal m/8 2^-14, so one
// multiply by 2^8 (exact) rebiases both to E4M3's 2^(e-7) (1 + m/8) and
// m 2^-9; then the sign, and NaN for the magnitude code 0x7f.
__device__ __forceinline__ __half2 e4m3x2_f16(uint32_t w) {
  const uint32_t mag = ((w & 0x7Fu) << 7) | ((w & 0x7F00u) << 15);
  uint32_t r = h2_as_u32(__hmul2(u32_as_h2(mag), __float2half2_rn(256.0f))) |
               ((w & 0x80u) << 8) | ((w & 0x8000u) << 16);
  if ((w & 0x7Fu) == 0x7Fu) r = (r & 0xFFFF0000u) | 0x7E00u;
  if ((w & 0x7F00u) == 0x7F00u) r = (r & 0x0000FFFFu) | 0x7E000000u;
  return u32_as_h2(r);
}

// NVFP4 item B of a 128-value tile (values 32B .. 32B+31): micro-blocks
// s0 = 2(B & 1) and s0 + 1 of the 36-byte block B >> 1, which starts
// o + 36 (B >> 1) bytes into the row window (o = 0 or 8, a run-time value:
// one code path for both offsets, so the decoders' instructions stay few).
// The block's bytes lie from chunk 2 (B >> 1) on, word (B >> 1) + o / 4 of
// them first: its scales (bytes s0, s0 + 1), then the item's 16 code bytes
// at 4 + 8 s0; micro-block s gives 8 values from the low nibbles of its 8
// bytes, then 8 from the high nibbles.  E2M1 codes become fp16 by the byte
// lookup and the product with the scale is exact in fp16 (six significant
// bits, magnitudes 2^-10 .. 2688).  Writes chunks 4B .. 4B+3 of row n.
template <int B>
__device__ __forceinline__ void dec_nvfp4_item(const uint8_t* row, uint8_t* A, int n, int o) {
  constexpr int C0 = 2 * (B >> 1), J0 = B >> 1, NCH = (B & 1) ? 3 : 2;
  static_assert(16 * (C0 + NCH) <= p_row_bytes<RG_NVFP4>(), "reads stay inside the row window");
  const auto r = load_chunks<C0, C0 + NCH - 1>(row);
  const bool o8 = o != 0;
  auto word = [&](int k) { return o8 ? r.w[J0 + 2 + k] : r.w[J0 + k]; };  // k-th word of the block
  const __half2 sc2 = e4m3x2_f16(word(0) >> (16 * (B & 1)));
  const __half2 sc0 = __low2half2(sc2), sc1 = __high2half2(sc2);
  uint32_t out[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // code word j: bytes 4j .. 4j+3 of the item's 16
    const uint32_t w = word(1 + 4 * (B & 1) + j);
    const __half2 sc = j < 2 ? sc0 : sc1;
    const int c = 2 * (j >> 1);  // chunk of the low nibbles: 0 (s0) or 2 (s1)
    uint32_t a0, a1, b0, b1;
    e2m1x4_f16(w & 0x0F0F0F0Fu, a0, a1);
    e2m1x4_f16((w >> 4) & 0x0F0F0F0Fu, b0, b1);
    out[c][2 * (j & 1)] = h2_as_u32(__hmul2(u32_as_h2(a0), sc));
    out[c][2 * (j & 1) + 1] = h2_as_u32(__hmul2(u32_as_h2(a1), sc));
    out[c + 1][2 * (j & 1)] = h2_as_u32(__hmul2(u32_as_h2(b0), sc));
    out[c + 1][2 * (j & 1) + 1] = h2_as_u32(__hmul2(u32_as_h2(b1), sc));
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) st_a_chunk(A, n, 4 * B + c, out[c][0], out[c][1], out[c][2], out[c][3]);
}

__device__ __forceinline__ uint32_t byte_of(uint32_t h1, uint32_t h2, uint32_t h3, int i) {
  const uint32_t w = i < 4 ? h1 : (i < 8 ? h2 : h3);
  return (w >> (8 * (i & 3))) & 0xFFu;
}

// Q4_K: 16 bytes of nibbles of chunk c (values 64c + 16hh .. +15 from the low
// nibbles, sub-block 2c; 64c + 32 + 16hh .. +15 from the high nibbles,
// sub-block 2c+1) of the super-block at `row`; chunk cl of this CTA's half.
// `q32`: the chunk's 32 nibble bytes (row + 16 + 32c in a whole super-block;
// the forward copies them apart from the 16-byte header `row`).
template <int H2, int CL, int HH>
__device__ __forceinline__ void dec_q4_k_part(const uint8_t* row, const uint8_t* q32, uint8_t* A,
                                              int n) {
  constexpr int c = 2 * H2 + CL;
  const uint4 hdr = *reinterpret_cast<const uint4*>(row);
  const uint4 qv = *reinterpret_cast<const uint4*>(q32 + 16 * HH);
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x >> 16)));
  int sc[2], m[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = 2 * c + h;
    if (j < 4) {
      sc[h] = byte_of(hdr.y, hdr.z, hdr.w, j) & 63;
      m[h] = byte_of(hdr.y, hdr.z, hdr.w, j + 4) & 63;
    } else {
      const uint32_t e = byte_of(hdr.y, hdr.z, hdr.w, j + 4);
      sc[h] = (e & 15) | ((byte_of(hdr.y, hdr.z, hdr.w, j - 4) >> 6) << 4);
      m[h] = (e >> 4) | ((byte_of(hdr.y, hdr.z, hdr.w, j) >> 6) << 4);
    }
  }
  const __half2 magic = __float2half2_rn(1024.0f);
  const __half2 ds0 = __float2half2_rn(d * static_cast<float>(sc[0]));
  const __half2 nm0 = __float2half2_rn(-(dmin * static_cast<float>(m[0])));
  const __half2 ds1 = __float2half2_rn(d * static_cast<float>(sc[1]));
  const __half2 nm1 = __float2half2_rn(-(dmin * static_cast<float>(m[1])));
  const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    four_affine(qw[j] & 0x0F0F0F0Fu, magic, ds0, nm0, lo[2 * j], lo[2 * j + 1]);
    four_affine((qw[j] >> 4) & 0x0F0F0F0Fu, magic, ds1, nm1, hi[2 * j], hi[2 * j + 1]);
  }
  constexpr int cb = 8 * CL + 2 * HH;
  st_a_chunk(A, n, cb, lo[0], lo[1], lo[2], lo[3]);
  st_a_chunk(A, n, cb + 1, lo[4], lo[5], lo[6], lo[7]);
  st_a_chunk(A, n, cb + 4, hi[0], hi[1], hi[2], hi[3]);
  st_a_chunk(A, n, cb + 5, hi[4], hi[5], hi[6], hi[7]);
}

// Q4_1 / Q5_0 / Q5_1 block at byte S of a row window: fp16 d (then fp16 m
// for Q4_1 and Q5_1), the fifth bits qh (Q5), 16 bytes of nibbles.  Writes
// its 32 values as chunks 4b .. 4b+3 of row n: d*(q-16) (Q5_0) rounded once,
// or fma(q, d, m) rounded once (Q4_1, Q5_1; d and m are exact fp16 fields).
template <int WT, int S>
__device__ __forceinline__ void dec_q41_q5_block(const uint8_t* row, uint8_t* A, int n, int b) {
  constexpr int QH = WT == RG_Q5_0 ? 2 : WT == RG_Q5_1 ? 4 : -1;
  constexpr int QS = WT == RG_Q4_1 ? 4 : WT == RG_Q5_0 ? 6 : 8;
  constexpr int C0 = S / 16;
  constexpr int XQ = S - 16 * C0 + QS + 12;  // the last quant word, relative to chunk C0
  constexpr int LAST = (XQ & 3) == 0 ? XQ + 3 : (XQ & ~3) + 7;  // last byte word_at reads
  constexpr int C1 = C0 + LAST / 16;
  static_assert(16 * C1 + 16 <= p_row_bytes<WT>(), "reads stay inside the row window");
  const auto r = load_chunks<C0, C1>(row);
  constexpr int X = S - 16 * C0;
  const uint32_t dm = r.word_at(X);
  const __half2 d2 = __half2half2(__ushort_as_half(static_cast<uint16_t>(dm & 0xFFFFu)));
  const __half2 m2 = __half2half2(__ushort_as_half(static_cast<uint16_t>(dm >> 16)));
  uint32_t qh = 0;
  if constexpr (QH >= 0) qh = r.word_at(X + QH);
  const __half2 off = __float2half2_rn(WT == RG_Q5_0 ? 1040.0f : 1024.0f);  // 1024 (+16)
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = r.word_at(X + QS + 4 * j);
    uint32_t xl = w & 0x0F0F0F0Fu, xh = (w >> 4) & 0x0F0F0F0Fu;
    if constexpr (QH >= 0) {
      xl |= fifth_bits4(qh >> (4 * j));
      xh |= fifth_bits4(qh >> (16 + 4 * j));
    }
    if constexpr (WT == RG_Q5_0) {
      four_scaled(xl, off, d2, lo[2 * j], lo[2 * j + 1]);
      four_scaled(xh, off, d2, hi[2 * j], hi[2 * j + 1]);
    } else {
      four_affine(xl, off, d2, m2, lo[2 * j], lo[2 * j + 1]);
      four_affine(xh, off, d2, m2, hi[2 * j], hi[2 * j + 1]);
    }
  }
  st_a_chunk(A, n, 4 * b, lo[0], lo[1], lo[2], lo[3]);
  st_a_chunk(A, n, 4 * b + 1, lo[4], lo[5], lo[6], lo[7]);
  st_a_chunk(A, n, 4 * b + 2, hi[0], hi[1], hi[2], hi[3]);
  st_a_chunk(A, n, 4 * b + 3, hi[4], hi[5], hi[6], hi[7]);
}

// Q5_K: as dec_q4_k_part, with the fifth bit of each value from qh: bit 2c
// (low nibbles) or 2c+1 (high nibbles) of qh[l]; this part covers l = 16HH ..
// 16HH+15, i.e. qh bytes 16HH .. 16HH+15 at window offset 16.
template <int H2, int CL, int HH>
__device__ __forceinline__ void dec_q5_k_part(const uint8_t* row, uint8_t* A, int n) {
  constexpr int c = 2 * H2 + CL;
  const uint4 hdr = *reinterpret_cast<const uint4*>(row);
  const uint4 hv = *reinterpret_cast<const uint4*>(row + 16 + 16 * HH);
  const uint4 qv = *reinterpret_cast<const uint4*>(row + 48 + 32 * c + 16 * HH);
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(hdr.x >> 16)));
  int sc[2], m[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = 2 * c + h;
    if (j < 4) {
      sc[h] = byte_of(hdr.y, hdr.z, hdr.w, j) & 63;
      m[h] = byte_of(hdr.y, hdr.z, hdr.w, j + 4) & 63;
    } else {
      const uint32_t e = byte_of(hdr.y, hdr.z, hdr.w, j + 4);
      sc[h] = (e & 15) | ((byte_of(hdr.y, hdr.z, hdr.w, j - 4) >> 6) << 4);
      m[h] = (e >> 4) | ((byte_of(hdr.y, hdr.z, hdr.w, j) >> 6) << 4);
    }
  }
  const __half2 magic = __float2half2_rn(1024.0f);
  const __half2 ds0 = __float2half2_rn(d * static_cast<float>(sc[0]));
  const __half2 nm0 = __float2half2_rn(-(dmin * static_cast<float>(m[0])));
  const __half2 ds1 = __float2half2_rn(d * static_cast<float>(sc[1]));
  const __half2 nm1 = __float2half2_rn(-(dmin * static_cast<float>(m[1])));
  const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
  const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t xl = (qw[j] & 0x0F0F0F0Fu) | (((hw[j] >> (2 * c)) & 0x01010101u) << 4);
    const uint32_t xh = ((qw[j] >> 4) & 0x0F0F0F0Fu) | (((hw[j] >> (2 * c + 1)) & 0x01010101u) << 4);
    four_affine(xl, magic, ds0, nm0, lo[2 * j], lo[2 * j + 1]);
    four_affine(xh, magic, ds1, nm1, hi[2 * j], hi[2 * j + 1]);
  }
  constexpr int cb = 8 * CL + 2 * HH;
  st_a_chunk(A, n, cb, lo[0], lo[1], lo[2], lo[3]);
  st_a_chunk(A, n, cb + 1, lo[4], lo[5], lo[6], lo[7]);
  st_a_chunk(A, n, cb + 4, hi[0], hi[1], hi[2], hi[3]);
  st_a_chunk(A, n, cb + 5, hi[4], hi[5], hi[6], hi[7]);
}

// Q6_K: a whole row's half (128 values, H = the half) from a window whose
// super-block starts O bytes in.  Value 128H + 32i + l: nibble of
// ql[64H + 32(i%2) + l] (high for i >= 2) and bits 2i..2i+1 of qh[32H + l]
// give q; the operand is fp16(d * sc[8H + 2i + l/16]) * (q - 32).  G >= 0:
// only the 64 values 64G .. 64G+63 of the half (chunks 8G .. 8G+7).
template <int O, int H, int G = -1>
__device__ __forceinline__ void dec_q6_k_row(const uint8_t* row, uint8_t* A, int n) {
  constexpr int QA = O + 64 * H, QHB = O + 128 + 32 * H, QS = O + 192 + 8 * H, QD = O + 208;
  // the last byte a word_at at offset x (relative to chunk C) reads
  constexpr auto last = [](int x) { return (x & 3) == 0 ? x + 3 : (x & ~3) + 7; };
  constexpr int CA = QA / 16, CA1 = CA + last(QA - 16 * CA + 60) / 16;
  constexpr int CH = QHB / 16, CH1 = CH + last(QHB - 16 * CH + 28) / 16;
  // (d's word_at covers the scales' too: QS + 7 < QD)
  constexpr int CS = QS / 16, CS1 = CS + last(QD - 16 * CS) / 16;
  static_assert(16 * CA1 + 16 <= p_row_bytes<RG_Q6_K>() && 16 * CH1 + 16 <= p_row_bytes<RG_Q6_K>() &&
                    16 * CS1 + 16 <= p_row_bytes<RG_Q6_K>() && QS + 7 < QD,
                "reads stay inside the row window");
  const auto ra = load_chunks<CA, CA1>(row);
  const auto rh = load_chunks<CH, CH1>(row);
  const auto rs = load_chunks<CS, CS1>(row);
  constexpr int XA = QA - 16 * CA, XH = QHB - 16 * CH, XS = QS - 16 * CS, XD = QD - 16 * CS;
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(rs.word_at(XD) & 0xFFFFu)));
  __half2 ds[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int is = 0; is < 2; ++is) {
      const int sc = static_cast<int8_t>(rs.word_at(XS + 2 * i + is) & 0xFFu);
      ds[i][is] = __float2half2_rn(d * static_cast<float>(sc));  // exact product, one rounding
    }
  const __half2 off = __float2half2_rn(1056.0f);  // 1024 + 32
#pragma unroll
  for (int cq = 0; cq < 4; ++cq) {  // l = 8cq .. 8cq+7
    uint32_t o[4][4];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = 2 * cq + jj;  // l = 4j .. 4j+3
      const uint32_t a = ra.word_at(XA + 4 * j), b = ra.word_at(XA + 32 + 4 * j);
      const uint32_t hq = rh.word_at(XH + 4 * j);
      const uint32_t x[4] = {(a & 0x0F0F0F0Fu) | ((hq & 0x03030303u) << 4),
                             (b & 0x0F0F0F0Fu) | (((hq >> 2) & 0x03030303u) << 4),
                             ((a >> 4) & 0x0F0F0F0Fu) | (((hq >> 4) & 0x03030303u) << 4),
                             ((b >> 4) & 0x0F0F0F0Fu) | (((hq >> 6) & 0x03030303u) << 4)};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (G < 0 || (i >> 1) == G) four_scaled(x[i], off, ds[i][cq >> 1], o[i][2 * jj], o[i][2 * jj + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (G < 0 || (i >> 1) == G) st_a_chunk(A, n, 4 * i + cq, o[i][0], o[i][1], o[i][2], o[i][3]);
  }
}

// The forward's Q6_K chunk, values 64G .. 64G+63 of half H of a super-block,
// from its three split windows (the half's low bits at pa, high bits at ph,
// the scales and d at ps), each starting O bytes in; O (even) and H are run
// time values, so one instance serves every super-block (instances per
// offset made the forward instruction-fetch bound).  Words at O + 4j: an
// aligned 32-bit load, or (U: O % 4 == 2) the two aligned words around it and
// one 16-bit funnel shift; the scales and d by 16-bit loads.
template <bool U, int G>
__device__ __forceinline__ void dec_q6_k_fwd(const uint8_t* pa, const uint8_t* ph, const uint8_t* ps, int O,
                                             int H, uint8_t* A, int n) {
  auto word = [&](const uint8_t* base, int j) -> uint32_t {
    if constexpr (!U) {
      return *reinterpret_cast<const uint32_t*>(base + O + 4 * j);
    } else {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(base + O - 2);
      return __funnelshift_r(w[j], w[j + 1], 16);
    }
  };
  const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(ps + O + 16)));
  // scales 8H + 4G .. 8H + 4G + 3: quarters i = 2G, 2G + 1, values l < 16 and l >= 16
  const uint8_t* psc = ps + O + 8 * H + 4 * G;
  const uint32_t s01 = *reinterpret_cast<const uint16_t*>(psc), s23 = *reinterpret_cast<const uint16_t*>(psc + 2);
  __half2 ds[2][2];
  ds[0][0] = __float2half2_rn(d * static_cast<float>(static_cast<int8_t>(s01 & 0xFFu)));
  ds[0][1] = __float2half2_rn(d * static_cast<float>(static_cast<int8_t>(s01 >> 8)));
  ds[1][0] = __float2half2_rn(d * static_cast<float>(static_cast<int8_t>(s23 & 0xFFu)));
  ds[1][1] = __float2half2_rn(d * static_cast<float>(static_cast<int8_t>(s23 >> 8)));
  const __half2 off = __float2half2_rn(1056.0f);  // 1024 + 32
#pragma unroll
  for (int cq = 0; cq < 4; ++cq) {  // l = 8cq .. 8cq+7
    uint32_t o[2][4];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = 2 * cq + jj;  // l = 4j .. 4j+3
      const uint32_t a = word(pa, j), b = word(pa, j + 8), hq = word(ph, j);
      // quarter i = 2G + e: the low (G = 0) or high (G = 1) nibbles of a (e = 0)
      // or b (e = 1), bits 2i..2i+1 of hq above them
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t q = e ? b : a;
        const uint32_t x = ((q >> (4 * G)) & 0x0F0F0F0Fu) | (((hq >> (2 * (2 * G + e))) & 0x03030303u) << 4);
        four_scaled(x, off, ds[e][cq >> 1], o[e][2 * jj], o[e][2 * jj + 1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) st_a_chunk(A, n, 4 * (2 * G + e) + cq, o[e][0], o[e][1], o[e][2], o[e][3]);
  }
}

// Q2_K: a whole row's half (128 values, H = the half) from a window whose
// super-block starts O bytes in (O = 0, 4, 8, 12).  Value 128H + 32j + 16s
// + l: bits 2j..2j+1 of qs[32H + 16s + l]; its scales byte 8H + 2j + s gives
// sc (low nibble) and m; the operand is fp16(q * fp16(d*sc) - fp16(dmin*m)).
// G >= 0: only the 64 values 64G .. 64G+63 of the half.
template <int O, int H, int G = -1>
__device__ __forceinline__ void dec_q2_k_row(const uint8_t* row, uint8_t* A, int n) {
  constexpr int QSB = O + 8 * H, QQ = O + 16 + 32 * H, QD = O + 80;
  static_assert(O % 4 == 0 && QD + 4 <= p_row_bytes<RG_Q2_K>(), "aligned words inside the window");
  constexpr int CS = QSB / 16, CS1 = (QSB + 7) / 16;
  constexpr int CQ = QQ / 16, CQ1 = (QQ + 31) / 16;
  constexpr int CD = QD / 16;
  const auto rs = load_chunks<CS, CS1>(row);
  const auto rq = load_chunks<CQ, CQ1>(row);
  const auto rd = load_chunks<CD, CD>(row);
  const uint32_t dw = rd.word_at(QD - 16 * CD);
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(dw & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(dw >> 16)));
  const uint32_t sw[2] = {rs.word_at(QSB - 16 * CS), rs.word_at(QSB - 16 * CS + 4)};
  const __half2 magic = __float2half2_rn(1024.0f);
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      if (G >= 0 && (j >> 1) != G) continue;
      const uint32_t b = (sw[j >> 1] >> (8 * (2 * (j & 1) + sb))) & 0xFFu;  // byte 2j + sb
      const __half2 ds = __float2half2_rn(d * static_cast<float>(b & 15u));       // exact product
      const __half2 nm = __float2half2_rn(-(dmin * static_cast<float>(b >> 4)));  // exact product
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // l = 8c .. 8c+7
        const int x = QQ - 16 * CQ + 16 * sb + 8 * c;
        uint32_t o[4];
        four_affine((rq.word_at(x) >> (2 * j)) & 0x03030303u, magic, ds, nm, o[0], o[1]);
        four_affine((rq.word_at(x + 4) >> (2 * j)) & 0x03030303u, magic, ds, nm, o[2], o[3]);
        st_a_chunk(A, n, 4 * j + 2 * sb + c, o[0], o[1], o[2], o[3]);
      }
    }
}

// Q3_K: a whole row's half from a window whose super-block starts O bytes in
// (O even).  Value 128H + 32j + 16s + l: q + 4 = (bits 2j..2j+1 of
// qs[32H + 16s + l]) | (bit 4H + j of hmask[16s + l]) << 2; the sub-block's
// 6-bit scale i = 8H + 2j + s; the operand is fp16(d * (sc - 32)) * q.
// G >= 0: only the 64 values 64G .. 64G+63 of the half.
template <int O, int H, int G = -1>
__device__ __forceinline__ void dec_q3_k_row(const uint8_t* row, uint8_t* A, int n) {
  constexpr int QH = O, QQ = O + 32 + 32 * H, QS = O + 96, QD = O + 108;
  constexpr auto last = [](int x) { return (x & 3) == 0 ? x + 3 : (x & ~3) + 7; };
  constexpr int CH = QH / 16, CH1 = CH + last(QH - 16 * CH + 28) / 16;
  constexpr int CQ = QQ / 16, CQ1 = CQ + last(QQ - 16 * CQ + 28) / 16;
  constexpr int CS = QS / 16, CS1 = CS + last(QD - 16 * CS) / 16;
  static_assert(O % 2 == 0 && 16 * CH1 + 16 <= p_row_bytes<RG_Q3_K>() &&
                    16 * CQ1 + 16 <= p_row_bytes<RG_Q3_K>() && 16 * CS1 + 16 <= p_row_bytes<RG_Q3_K>(),
                "reads stay inside the row window");
  const auto rh = load_chunks<CH, CH1>(row);
  const auto rq = load_chunks<CQ, CQ1>(row);
  const auto rs = load_chunks<CS, CS1>(row);
  constexpr int XH = QH - 16 * CH, XQ = QQ - 16 * CQ, XS = QS - 16 * CS, XD = QD - 16 * CS;
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(rs.word_at(XD) & 0xFFFFu)));
  // the scales' low nibbles of this half: bytes 0..7 (H = 0: low nibbles;
  // H = 1: high nibbles), their high bits: bytes 8..11, bits 2(i / 4)..
  const uint32_t s_lo[2] = {rs.word_at(XS), rs.word_at(XS + 4)};
  const uint32_t s_hi = rs.word_at(XS + 8);
  const __half2 off = __float2half2_rn(1028.0f);  // 1024 + 4
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      if (G >= 0 && (j >> 1) != G) continue;
      const int i = 8 * H + 2 * j + sb;
      const uint32_t lo = (s_lo[(i & 7) >> 2] >> (8 * (i & 3) + 4 * H)) & 15u;
      const uint32_t hi = (s_hi >> (8 * (i & 3) + 2 * (i >> 2))) & 3u;
      const int sc = static_cast<int>(lo | (hi << 4)) - 32;
      const __half2 ds = __float2half2_rn(d * static_cast<float>(sc));  // exact product, one rounding
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // l = 8c .. 8c+7
        uint32_t o[4];
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t q = (rq.word_at(XQ + 16 * sb + 8 * c + 4 * w) >> (2 * j)) & 0x03030303u;
          const uint32_t hb = (rh.word_at(XH + 16 * sb + 8 * c + 4 * w) >> (4 * H + j)) & 0x01010101u;
          four_scaled(q | (hb << 2), off, ds, o[2 * w], o[2 * w + 1]);
        }
        st_a_chunk(A, n, 4 * j + 2 * sb + c, o[0], o[1], o[2], o[3]);
      }
    }
}

// The forward's Q2_K chunk (values 64G .. 64G+63 of half H) from a row
// window whose super-block starts O bytes in; O (0, 4, 8, 12) and H at run
// time (one instance for every super-block), every word an aligned 32-bit
// load.  Values as dec_q2_k_row.
template <int G>
__device__ __forceinline__ void dec_q2_k_fwd(const uint8_t* row, int O, int H, uint8_t* A, int n) {
  const uint8_t* b = row + O;
  const uint32_t dw = *reinterpret_cast<const uint32_t*>(b + 80);
  const float d = __half2float(__ushort_as_half(static_cast<uint16_t>(dw & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<uint16_t>(dw >> 16)));
  const uint32_t sw = *reinterpret_cast<const uint32_t*>(b + 8 * H + 4 * G);  // scale bytes 8H + 4G ..
  const uint8_t* qb = b + 16 + 32 * H;
  const __half2 magic = __float2half2_rn(1024.0f);
#pragma unroll
  for (int jj = 0; jj < 2; ++jj)
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      const int j = 2 * G + jj;
      const uint32_t sc = (sw >> (8 * (2 * jj + sb))) & 0xFFu;  // scales byte 8H + 2j + sb
      const __half2 ds = __float2half2_rn(d * static_cast<float>(sc & 15u));       // exact product
      const __half2 nm = __float2half2_rn(-(dmin * static_cast<float>(sc >> 4)));  // exact product
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // l = 8c .. 8c+7
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(qb + 16 * sb + 8 * c);
        uint32_t o[4];
        four_affine((qw[0] >> (2 * j)) & 0x03030303u, magic, ds, nm, o[0], o[1]);
        four_affine((qw[1] >> (2 * j)) & 0x03030303u, magic, ds, nm, o[2], o[3]);
        st_a_chunk(A, n, 4 * j + 2 * sb + c, o[0], o[1], o[2], o[3]);
      }
    }
}

// The forward's Q3_K chunk (values 64G .. 64G+63 of half H) from a row
// window whose super-block starts O bytes in; O (even) and H at run time,
// words at O + x by an aligned 32-bit load or (U: O % 4 == 2) the two
// aligned words around them and one 16-bit funnel shift.  Values as
// dec_q3_k_row.
template <bool U, int G>
__device__ __forceinline__ void dec_q3_k_fwd(const uint8_t* row, int O, int H, uint8_t* A, int n) {
  auto word = [&](int x) -> uint32_t {
    if constexpr (!U) {
      return *reinterpret_cast<const uint32_t*>(row + O + x);
    } else {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(row + O - 2 + x);
      return __funnelshift_r(w[0], w[1], 16);
    }
  };
  const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(row + O + 108)));
  const uint32_t s_lo[2] = {word(96), word(100)};
  const uint32_t s_hi = word(104);
  const __half2 off = __float2half2_rn(1028.0f);  // 1024 + 4
#pragma unroll
  for (int jj = 0; jj < 2; ++jj)
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      const int j = 2 * G + jj, il = 2 * j + sb;  // the sub-block 8H + il
      const uint32_t lo = (s_lo[il >> 2] >> (8 * (il & 3) + 4 * H)) & 15u;
      const uint32_t hi = (s_hi >> (8 * (il & 3) + 2 * (2 * H + (il >> 2)))) & 3u;
      const int sc = static_cast<int>(lo | (hi << 4)) - 32;
      const __half2 ds = __float2half2_rn(d * static_cast<float>(sc));  // exact product, one rounding
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // l = 8c .. 8c+7
        uint32_t o[4];
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const int x = 16 * sb + 8 * c + 4 * w;
          const uint32_t q = (word(32 + 32 * H + x) >> (2 * j)) & 0x03030303u;
          const uint32_t hb = (word(x) >> (4 * H + j)) & 0x01010101u;
          four_scaled(q | (hb << 2), off, ds, o[2 * w], o[2 * w + 1]);
        }
        st_a_chunk(A, n, 4 * j + 2 * sb + c, o[0], o[1], o[2], o[3]);
      }
    }
}

// Block b (32-value types) or part b (Q4_K, Q5_K: chunk b >> 1 of the
// half, 16 bytes b & 1) of row n of a stage.
template <int WT, int ODD, int B>
__device__ __forceinline__ void dec_item(const uint8_t* row, uint8_t* A, int n, int o) {
  if constexpr (WT == RG_MXFP4) dec_mxfp4_block<B>(row, A, n, o);
  else if constexpr (WT == RG_NVFP4) dec_nvfp4_item<B>(row, A, n, o);
  else if constexpr (WT == RG_Q8_0) dec_q8_block<8 * ODD + 34 * B>(row, A, n, B);
  else if constexpr (WT == RG_Q4_0) dec_q4_0_block<8 * ODD + 18 * B>(row, A, n, B);
  else if constexpr (WT == RG_Q4_1) dec_q41_q5_block<WT, 20 * B>(row, A, n, B);
  else if constexpr (WT == RG_Q5_0) dec_q41_q5_block<WT, 8 * ODD + 22 * B>(row, A, n, B);
  else if constexpr (WT == RG_Q5_1) dec_q41_q5_block<WT, 24 * B>(row, A, n, B);
  else if constexpr (WT == RG_Q4_K) dec_q4_k_part<ODD, B / 2, B % 2>(row, row + 16 + 32 * (2 * ODD + B / 2), A, n);
  else dec_q5_k_part<ODD, B / 2, B % 2>(row, A, n);
}

// One warp decodes a whole stage: P holds BC packed rows (row stride
// p_row_bytes) of this CTA's 128-value tile, A receives the fp16 operand.
// Item i of lane l is row n = l + 32*(i & 1) and block (or Q4_K part) i >> 1:
// eight independent blocks per lane, and the lanes of a load or store sit on
// consecutive rows, i.e. in distinct bank groups.  ODD = the tile's k index is
// odd (window offset 8 for Q8_0 / Q4_0, second half of a Q4_K super-block).
// o: the MXFP4 and NVFP4 run-time window offset (0, 4, 8 or 12; 0 or 8); O: the super-block
// offset of the row-half decoders.
template <int WT, int ODD, int NPART, int O = 0>
__device__ __forceinline__ void decode_stage_warp(const uint8_t* __restrict__ P,
                                                  uint8_t* __restrict__ A, int lane, int part,
                                                  int o = 0) {
  constexpr int PR = p_row_bytes<WT>();
  if constexpr (WT == RG_Q6_K || WT == RG_Q3_K || WT == RG_Q2_K) {
    static_assert(NPART == 2, "a lane decodes one row's half");
    const int n = lane + 32 * part;
    if constexpr (WT == RG_Q6_K) dec_q6_k_row<O, ODD>(P + n * PR, A, n);
    else if constexpr (WT == RG_Q3_K) dec_q3_k_row<O, ODD>(P + n * PR, A, n);
    else dec_q2_k_row<O, ODD>(P + n * PR, A, n);
    return;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if ((i & (NPART - 1)) != part) continue;  // this warp's share of the items
    const int n = lane + 32 * (i & 1);
    const uint8_t* row = P + n * PR;
    switch (i >> 1) {
      case 0: dec_item<WT, ODD, 0>(row, A, n, o); break;
      case 1: dec_item<WT, ODD, 1>(row, A, n, o); break;
      case 2: dec_item<WT, ODD, 2>(row, A, n, o); break;
      default: dec_item<WT, ODD, 3>(row, A, n, o); break;
    }
  }
}

// The forward's stage (FWD kernels): 128 rows of W by the 64 values HV of a
// 128-value tile (HV = 0: values 0..63, 1: 64..127), decoded into a K-major
// operand tile (row n: 128 bytes, chunk c at c ^ (n mod 8), rows 8 apart by
// 1024 bytes): the OUT_PROD decoders' own layout once the half's column
// block is taken as the tile (A - HV column blocks), with 128 rows instead
// of 64.  Warp `part` of the slot's two takes rows lane + 32 (2 part + r),
// r = 0, 1, and of each row the items (blocks, Q4_K parts) of half HV.
template <int WT, int ODD, int HV, int O = 0>
__device__ __forceinline__ void decode_stage_fwd(const uint8_t* __restrict__ P, uint8_t* __restrict__ A,
                                                 int lane, int part, int o = 0) {
  constexpr int PR = p_row_bytes<WT>();
  uint8_t* Ah = A - HV * A_COLBLK;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int n = lane + 32 * (2 * part + r);
    const uint8_t* row = P + n * PR;
    if constexpr (WT == RG_Q4_K) {
      // the 16-byte headers of the stage's 128 rows, then their 32 nibble bytes
      const uint8_t* hdr = P + n * 16;
      const uint8_t* q32 = P + 128 * 16 + n * 32;
      dec_q4_k_part<ODD, HV, 0>(hdr, q32, Ah, n);
      dec_q4_k_part<ODD, HV, 1>(hdr, q32, Ah, n);
    } else {
      static_assert(WT != RG_Q6_K && WT != RG_Q3_K && WT != RG_Q2_K,
                    "the forward's K-quant stages are decode_stage_fwd_q6 and decode_stage_fwd_k");
      dec_item<WT, ODD, 2 * HV>(row, Ah, n, o);
      dec_item<WT, ODD, 2 * HV + 1>(row, Ah, n, o);
    }
  }
}

// The forward's Q3_K and Q2_K stages: 128 rows of the chunk from their
// whole windows, the super-block O bytes in, half H, quarter HV.
template <int WT, bool U, int HV>
__device__ __forceinline__ void decode_stage_fwd_k(const uint8_t* __restrict__ P, uint8_t* __restrict__ A,
                                                   int lane, int part, int O, int H) {
  uint8_t* Ah = A - HV * A_COLBLK;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int n = lane + 32 * (2 * part + r);
    if constexpr (WT == RG_Q3_K) dec_q3_k_fwd<U, HV>(P + n * p_fwd_row_bytes<WT>(), O, H, Ah, n);
    else dec_q2_k_fwd<HV>(P + n * p_fwd_row_bytes<WT>(), O, H, Ah, n);
  }
}

// The forward's Q6_K stage: 128 rows of the chunk, the super-block O bytes
// into its windows, half H, quarter G (of the half) HV.
template <bool U, int HV>
__device__ __forceinline__ void decode_stage_fwd_q6(const uint8_t* __restrict__ P, uint8_t* __restrict__ A,
                                                    int lane, int part, int O, int H) {
  uint8_t* Ah = A - HV * A_COLBLK;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int n = lane + 32 * (2 * part + r);
    dec_q6_k_fwd<U, HV>(P + n * Q6F_A, P + 128 * Q6F_A + n * Q6F_H, P + 128 * (Q6F_A + Q6F_H) + n * Q6F_S, O, H,
                        Ah, n);
  }
}

// The forward's Q8_0 stage: 128 rows' two blocks of the 64-value chunk,
// starting O bytes into each row's 80-byte window, as chunks 0..7.
template <int O>
__device__ __forceinline__ void decode_stage_fwd_q8(const uint8_t* __restrict__ P, uint8_t* __restrict__ A,
                                                    int lane, int part) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int n = lane + 32 * (2 * part + r);
    const uint8_t* row = P + n * p_fwd_row_bytes<RG_Q8_0>();
    dec_q8_block<O>(row, A, n, 0);
    dec_q8_block<O + 34>(row, A, n, 1);
  }
}

// decode_stage_fwd for the run-time tile kw of the row (its parity, and the
// block offset of the row-half and MXFP4 decoders) and half hv.
template <int WT>
__device__ __forceinline__ void decode_fwd_stage(const uint8_t* __restrict__ P, uint8_t* __restrict__ A,
                                                 int lane, int part, int kw, int hv) {
  if constexpr (WT == RG_Q6_K) {
    // the super-block's offset into its grain, at run time (four instances)
    const int o = ((kw >> 1) * block_bytes(WT)) & 15;
    if (o & 2) {
      if (hv) decode_stage_fwd_q6<true, 1>(P, A, lane, part, o, kw & 1);
      else decode_stage_fwd_q6<true, 0>(P, A, lane, part, o, kw & 1);
    } else {
      if (hv) decode_stage_fwd_q6<false, 1>(P, A, lane, part, o, kw & 1);
      else decode_stage_fwd_q6<false, 0>(P, A, lane, part, o, kw & 1);
    }
  } else if constexpr (WT == RG_Q3_K || WT == RG_Q2_K) {
    // the super-block's offset into its grain (even; Q2_K a multiple of 4) at
    // run time: two instances (Q2_K) or four (Q3_K)
    const int o = ((kw >> 1) * block_bytes(WT)) & 15;
    bool shifted = false;
    if constexpr (WT == RG_Q3_K) shifted = (o & 2) != 0;
    if constexpr (WT == RG_Q3_K) {
      if (shifted) {
        if (hv) decode_stage_fwd_k<WT, true, 1>(P, A, lane, part, o, kw & 1);
        else decode_stage_fwd_k<WT, true, 0>(P, A, lane, part, o, kw & 1);
        return;
      }
    }
    if (hv) decode_stage_fwd_k<WT, false, 1>(P, A, lane, part, o, kw & 1);
    else decode_stage_fwd_k<WT, false, 0>(P, A, lane, part, o, kw & 1);
  } else if constexpr (WT == RG_Q8_0) {
    // the 64-value chunk's two blocks start (68 gf) mod 16 bytes into its window
    switch ((((2 * kw + hv) * 68) & 15) >> 2) {
      case 0: decode_stage_fwd_q8<0>(P, A, lane, part); break;
      case 1: decode_stage_fwd_q8<4>(P, A, lane, part); break;
      case 2: decode_stage_fwd_q8<8>(P, A, lane, part); break;
      default: decode_stage_fwd_q8<12>(P, A, lane, part); break;
    }
  } else if constexpr (WT == RG_MXFP4 || WT == RG_NVFP4) {
    // the tile's blocks start 0, 4, 8 or 12 (MXFP4) or 0 or 8 (NVFP4) bytes into the window
    const int o = WT == RG_MXFP4 ? (kw * 68) & 12 : (kw & 1) * 8;
    if (hv) decode_stage_fwd<WT, 0, 1>(P, A, lane, part, o);
    else decode_stage_fwd<WT, 0, 0>(P, A, lane, part, o);
  } else if (kw & 1) {
    if (hv) decode_stage_fwd<WT, 1, 1>(P, A, lane, part);
    else decode_stage_fwd<WT, 1, 0>(P, A, lane, part);
  } else {
    if (hv) decode_stage_fwd<WT, 0, 1>(P, A, lane, part);
    else decode_stage_fwd<WT, 0, 0>(P, A, lane, part);
  }
}

// Byte offset (16-byte multiple) of the window a 128-value tile kt loads from a packed row.
template <int WT>
__device__ __forceinline__ int p_window_start(int kt) {
  if constexpr (WT == RG_Q8_0) return (kt * 136) & ~15;
  if constexpr (WT == RG_Q4_0) return (kt * 72) & ~15;
  if constexpr (WT == RG_Q4_1) return kt * 80;
  if constexpr (WT == RG_Q5_0) return (kt * 88) & ~15;
  if constexpr (WT == RG_Q5_1) return kt * 96;
  if constexpr (WT == RG_Q5_K) return (kt >> 1) * 176;
  if constexpr (WT == RG_Q6_K) return ((kt >> 1) * 210) & ~15;
  if constexpr (WT == RG_Q3_K) return ((kt >> 1) * 110) & ~15;
  if constexpr (WT == RG_Q2_K) return ((kt >> 1) * 84) & ~15;
  if constexpr (WT == RG_MXFP4) return (kt * 68) & ~15;
  if constexpr (WT == RG_NVFP4) return (kt * 72) & ~15;
  return (kt >> 1) * 144;  // Q4_K: the whole super-block
}

// --- the work of one persistent unit -------------------------------------------
//
// A unit (a CTA pair, or one CTA) works through segments (item, c0, c1):
// contraction chunks [c0, c1) of work item `item` (a tile, or a tile and a
// contraction split).  First the data-parallel items u, u + U, ... below
// n_dp, each whole.  Then, with stream-K, its even share of the remaining
// n_items - n_dp tiles (fewer than U), whose chunks follow one another tile
// by tile: chunks [g0(u), g0(u + 1)) of that run, g0(u) = floor(u * Rn / U),
// Rn = remaining tiles x n_chunks.  A share is shorter than one tile, so it
// touches at most two tiles: the tail of one and the head of the next, and
// (Rn >= U, else no sharing) is never empty.  (The planner takes stream-K
// only while Rn * U < 2^31: 32-bit arithmetic.)
template <bool SK>
struct Segs {
  int item, U, n_dp, nck;
  uint32_t g, g1;
  __device__ __forceinline__ Segs(int u, int n_units, int n_items, int n_chunks)
      : item(u), U(n_units), nck(n_chunks), g(0), g1(0) {
    n_dp = n_items;
    if constexpr (!SK) return;
    n_dp = (n_items / n_units) * n_units;
    // fewer chunks left than units (a residency cap can make it so): whole
    // items only, so that every unit's share is non-empty when shared
    if (static_cast<uint32_t>(n_items - n_dp) * static_cast<uint32_t>(n_chunks) <
        static_cast<uint32_t>(n_units))
      n_dp = n_items;
    const uint32_t rn = static_cast<uint32_t>(n_items - n_dp) * static_cast<uint32_t>(n_chunks);
    g = static_cast<uint32_t>(u) * rn / static_cast<uint32_t>(n_units);
    g1 = static_cast<uint32_t>(u + 1) * rn / static_cast<uint32_t>(n_units);
  }
  __device__ __forceinline__ bool next(int& it, int& c0, int& c1) {
    if (item < n_dp) {
      it = item;
      c0 = 0;
      c1 = nck;
      item += U;
      return true;
    }
    if constexpr (!SK) return false;
    if (g >= g1) return false;
    const int x = static_cast<int>(g / static_cast<uint32_t>(nck));
    it = n_dp + x;
    c0 = static_cast<int>(g) - x * nck;
    c1 = min(nck, c0 + static_cast<int>(g1 - g));
    g += static_cast<uint32_t>(c1 - c0);
    return true;
  }
};

// Stream-K bookkeeping of a shared tile (remainder index x): its chunk run
// [a, a + nck), a = x * nck, is shared by units sk_unit_of(a) ..
// sk_unit_of(a + nck - 1), in chunk order.  The first of them ends its share
// with the tile's head (chunk 0 on); every later one starts its share inside
// the tile, and since a share is shorter than a tile that is the only piece
// of a tile it does not begin: its partial sums go to slab u.
__device__ __forceinline__ int sk_unit_of(uint32_t g, uint32_t rn, int U) {
  return static_cast<int>(((g + 1) * static_cast<uint32_t>(U) - 1) / rn);
}

// --- the kernel -----------------------------------------------------------------
//
// Barriers (8 bytes each, per stage s unless noted):
//   full_p[s]    packed W window landed in this CTA (quantized types; local TMA)
//   full_ab[s]   operand tiles of the whole pair landed: on the MMA-issuing
//                CTA, armed once by its producer with the pair's byte count;
//                both CTAs' TMA loads complete on it
//   full_dec[s]  this stage's A is decoded in every CTA: every decoder warp
//                of the slot, in either CTA, arrives on the issuing CTA's copy
//   empty[s]     the MMAs that read stage s completed (multicast commit)
//   acc_full[2], acc_empty[2]   the two tensor-memory accumulators
//   drain        local: the MMAs issued so far completed (abort path)

template <int WT, int CG, int BT, bool AD, bool SK, bool FWD = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    out_prod_tc_kernel(const __grid_constant__ CUtensorMap map_w,
                       const __grid_constant__ CUtensorMap map_y,
                       const __grid_constant__ CUtensorMap map_l,
                       const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_p,
                       const __grid_constant__ CUtensorMap map_q, int n_main,
                       float* __restrict__ dX, int64_t ldx, float beta, int T, int K,
                       int n_kunits, int n_ttiles, int band, int n_chunks, int n_splits,
                       float* __restrict__ part, WaitCtl ctl) {
  using C = Cfg<WT, CG, BT, FWD>;
  static_assert(!FWD || (!AD && !SK), "the forward runs without an adapter or stream-K");
  constexpr int S = C::S;
  extern __shared__ uint8_t smem_raw[];
  // align inside the shared window (pointer arithmetic keeps the shared space)
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sP = smem + C::OFF_P;
  const uint32_t bar0 = smem_addr(smem + C::OFF_BAR);
  auto full_p = [&](int s) { return bar0 + 8u * s; };
  auto full_ab = [&](int s) { return bar0 + 8u * (S + s); };
  auto full_dec = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto empty = [&](int s) { return bar0 + 8u * (3 * S + s); };
  auto acc_full = [&](int a) { return bar0 + 8u * (4 * S + a); };
  auto acc_empty = [&](int a) { return bar0 + 8u * (4 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (4 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  // the split reduction or stream-K's second pass may be scheduled as this
  // kernel's CTAs leave the SMs (it waits for this kernel before reading)
  pdl_launch_dependents();
  const int unit = blockIdx.x / CG, n_units = gridDim.x / CG;
  // work items: (tile, split); a split covers chunks [split * n_chunks, +n_chunks)
  // of the contraction (chunks past N are zero-filled by TMA and add nothing).
  // AD (a low-rank adapter rides along): chunks from n_main on are the
  // adapter's: their A rows are its dense 16-bit rows (map_l) and their B
  // columns its projected dY, which sit after dY's own columns in the same
  // 16-bit copy.  Without one (AD false) map_l and n_main are not read.
  const int n_tiles = n_kunits * n_ttiles * n_splits;
  const int n_tiles1 = n_kunits * n_ttiles;

  auto wait_any = [&](uint32_t bar, uint32_t parity) {
    if constexpr (CG == 2)
      return mbar_wait_cluster(bar, parity, ctl, abort_flag);
    else
      return mbar_wait(bar, parity, ctl, abort_flag);
  };

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_p(s), 1);
      mbar_init(full_ab(s), 1);
      mbar_init(full_dec(s), C::FULL_DEC_COUNT);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), C::ACC_EMPTY_COUNT);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&map_w);
    tma_prefetch_map(&map_y);
    if constexpr (AD || (FWD && (WT == RG_Q4_K || WT == RG_Q6_K))) tma_prefetch_map(&map_l);
    if constexpr (FWD && WT == RG_Q6_K) tma_prefetch_map(&map_q);
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc2(smem_addr(tmem_slot), C::TMEM_COLS);
      tmem_relinquish2();
    } else {
      tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (CG == 2)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // tile -> (k unit, t tile): bands of `band` k units; inside a band the t
  // tiles run outer, so the band's slice of W stays in L2 while every t tile
  // of dY passes by once per band
  auto coords = [&](int item, int& ku, int& tt) {
    const int tile = item % n_tiles1;
    const int per_band = band * n_ttiles;
    const int b = tile / per_band, r = tile - b * per_band;
    const int gk = min(band, n_kunits - b * band);
    tt = r / gk;
    ku = b * band + (r - tt * gk);
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // this kernel may start before the kernel that wrote its operands (dY's
    // 16-bit copy, a converted W) has finished: every operand copy comes
    // after this wait (the other roles read nothing an earlier kernel of the
    // call writes)
    pdl_wait();
    const uint32_t ab_bar_leader = CG == 2 ? mapa_shared(full_ab(0), 0) : full_ab(0);
    int s = 0;
    uint32_t ph = 0;
    uint32_t pend_p = 0, pend_ab = 0, pend_ph = 0;  // stages with copies in flight
    bool ok = true;
    Segs<SK> sg(unit, n_units, n_tiles, n_chunks);
    int tile = 0, c0 = 0, c1 = 0;
    while (ok && sg.next(tile, c0, c1)) {
      int ku, tt;
      coords(tile, ku, tt);
      const int cbase = (tile / n_tiles1) * n_chunks;  // first contraction chunk of the split
      const int kt = ku * CG + static_cast<int>(rank);
      const int ty = tt * BT + static_cast<int>(rank) * B_ROWS;
      for (int c = c0; c < c1; ++c) {
        ok = __all_sync(0xffffffffu, mbar_wait(empty(s), ph ^ 1u, ctl, abort_flag));
        if (!ok) break;
        if (lane == 0) {
          const uint32_t abar = ab_bar_leader + 8u * s;
          const int gc = cbase + c;  // the contraction chunk
          if constexpr (!AD) {
            if (leader) {
              mbar_arrive_expect_tx(full_ab(s), C::AB_BYTES_PAIR);
              pend_ab |= 1u << s;
            }
            if constexpr (C::QUANT) {
              mbar_arrive_expect_tx(full_p(s), C::P_BYTES);
              if constexpr (FWD && WT == RG_Q4_K) {
                // the super-block headers, then the chunk's nibbles (map_l), 128 rows each
                const int sb = (gc >> 2) * 144;
                tma_load_2d(smem_addr(sP + s * C::P_STAGE), &map_w, full_p(s), sb / 4, kt * BM);
                tma_load_2d(smem_addr(sP + s * C::P_STAGE) + 128 * 16, &map_l, full_p(s),
                            (sb + 16 + 32 * (gc & 3)) / 4, kt * BM);
              } else if constexpr (FWD && WT == RG_Q6_K) {
                // the half's low bits, its high bits, the scales and d (three
                // windows, 128 rows each, one region of the stage apiece)
                const int sb = (gc >> 2) * 210, h = (gc >> 1) & 1;
                const uint32_t dst = smem_addr(sP + s * C::P_STAGE);
                tma_load_2d(dst, &map_w, full_p(s), ((sb + 64 * h) & ~15) / 4, kt * BM);
                tma_load_2d(dst + 128 * Q6F_A, &map_l, full_p(s), ((sb + 128 + 32 * h) & ~15) / 4, kt * BM);
                tma_load_2d(dst + 128 * (Q6F_A + Q6F_H), &map_q, full_p(s), ((sb + 192) & ~15) / 4, kt * BM);
              } else if constexpr (FWD && WT == RG_Q8_0) {  // the chunk's two blocks
                tma_load_2d(smem_addr(sP + s * C::P_STAGE), &map_w, full_p(s), ((gc * 68) & ~15) / 4,
                            kt * BM);
              } else if constexpr (FWD) {  // the window of the 128-value tile holding chunk gc
                tma_load_2d(smem_addr(sP + s * C::P_STAGE), &map_w, full_p(s),
                            p_window_start<WT>(gc >> 1) / 4, kt * BM);
              } else
                tma_load_2d(smem_addr(sP + s * C::P_STAGE), &map_w, full_p(s),
                            p_window_start<WT>(kt) / 4, gc * BC);
              pend_p |= 1u << s;
            } else {
              const uint32_t a_dst = smem_addr(sA + s * A_STAGE);
              if constexpr (FWD) {
                // 64 values of 128 rows: the K-major, 128-byte swizzled operand itself
                if constexpr (CG == 2)
                  tma_load_2d_pair(a_dst, &map_w, abar, gc * BC, kt * BM);
                else
                  tma_load_2d(a_dst, &map_w, abar, gc * BC, kt * BM);
              } else if constexpr (CG == 2) {
                tma_load_2d_pair(a_dst, &map_w, abar, kt * BM, gc * BC);
                tma_load_2d_pair(a_dst + A_COLBLK, &map_w, abar, kt * BM + 64, gc * BC);
              } else {
                tma_load_2d(a_dst, &map_w, abar, kt * BM, gc * BC);
                tma_load_2d(a_dst + A_COLBLK, &map_w, abar, kt * BM + 64, gc * BC);
              }
            }
          } else {
            const bool adapter = gc >= n_main;
            const bool dense_a = !C::QUANT || adapter;  // A straight from TMA
            if (leader) {
              mbar_arrive_expect_tx(full_ab(s), C::QUANT && adapter
                                                    ? C::AB_BYTES_PAIR + CG * A_STAGE
                                                    : C::AB_BYTES_PAIR);
              pend_ab |= 1u << s;
            }
            if constexpr (C::QUANT) {
              if (adapter) {
                mbar_arrive(full_p(s));  // no packed window: the decoders pass
              } else {
                mbar_arrive_expect_tx(full_p(s), C::P_BYTES);
                tma_load_2d(smem_addr(sP + s * C::P_STAGE), &map_w, full_p(s),
                            p_window_start<WT>(kt) / 4, gc * BC);
                pend_p |= 1u << s;
              }
            }
            if (dense_a) {
              const CUtensorMap* ma = adapter ? &map_l : &map_w;
              const int row = (adapter ? gc - n_main : gc) * BC;
              const uint32_t a_dst = smem_addr(sA + s * A_STAGE);
              if constexpr (CG == 2) {
                tma_load_2d_pair(a_dst, ma, abar, kt * BM, row);
                tma_load_2d_pair(a_dst + A_COLBLK, ma, abar, kt * BM + 64, row);
              } else {
                tma_load_2d(a_dst, ma, abar, kt * BM, row);
                tma_load_2d(a_dst + A_COLBLK, ma, abar, kt * BM + 64, row);
              }
            }
          }
          if constexpr (CG == 2)
            tma_load_2d_pair(smem_addr(sB + s * B_STAGE), &map_y, abar, (cbase + c) * BC, ty);
          else
            tma_load_2d(smem_addr(sB + s * B_STAGE), &map_y, abar, (cbase + c) * BC, ty);
          pend_ph = (pend_ph & ~(1u << s)) | (ph << s);
        }
        __syncwarp();
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // drain: the copies this CTA started land before it leaves.  Local
      // barriers are waited on; a follower's operand halves complete on the
      // issuing CTA's barrier, which that CTA drains, and the follower waits
      // out a copy's latency many times over.
      volatile int no_abort = 0;
      for (int st = 0; st < S; ++st) {
        const uint32_t p = (pend_ph >> st) & 1u;
        if (pend_p & (1u << st)) (void)mbar_wait(full_p(st), p, ctl, &no_abort);
        if (pend_ab & (1u << st)) (void)mbar_wait(full_ab(st), p, ctl, &no_abort);
      }
      if (!leader) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the even CTA of a pair) ----------------
    if (leader) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      Segs<SK> sg(unit, n_units, n_tiles, n_chunks);
      int tile = 0, c0 = 0, c1 = 0;
      for (int j = 0; ok && sg.next(tile, c0, c1); ++j) {
        const int a = j & 1;
        const uint32_t aph = (static_cast<uint32_t>(j) >> 1) & 1u;
        ok = __all_sync(0xffffffffu, wait_any(acc_empty(a), aph ^ 1u));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * BT);
        for (int c = c0; c < c1; ++c) {
          bool got = wait_any(full_ab(s), ph);
          if constexpr (C::QUANT) got = got && wait_any(full_dec(s), ph);
          ok = __all_sync(0xffffffffu, got);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_base = smem_addr(sA + s * A_STAGE);
            const uint32_t b_base = smem_addr(sB + s * B_STAGE);
#pragma unroll
            for (int kk = 0; kk < BC / UMMA_K; ++kk) {
              // A: MN-major, k-column blocks 8 KB apart (LBO), 8-row groups of n 1 KB apart
              // (SBO); the forward's K-major A as B below (16 values = 32 bytes along a row)
              const uint64_t ad = FWD ? sdesc_sw128(a_base + kk * (UMMA_K * 2), 16, 1024)
                                      : sdesc_sw128(a_base + kk * (UMMA_K * 128), A_COLBLK, 1024);
              // B: K-major, 16 values of n = 32 bytes along the swizzled row; 8-row groups 1 KB apart
              const uint64_t bd = sdesc_sw128(b_base + kk * (UMMA_K * 2), 16, 1024);
              const uint32_t acc = ((c - c0) | kk) != 0 ? 1u : 0u;
              if constexpr (CG == 2)
                tc_mma_f16_pair(d_tmem, ad, bd, C::IDESC, acc);
              else
                tc_mma_f16(d_tmem, ad, bd, C::IDESC, acc);
            }
            if constexpr (CG == 2)
              tc_commit_pair(empty(s), 0x3);
            else
              tc_commit(empty(s));
          }
          __syncwarp();
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) {
          if constexpr (CG == 2)
            tc_commit_pair(acc_full(a), 0x3);
          else
            tc_commit(acc_full(a));
        }
        __syncwarp();
      }
      if (!ok && lane == 0) {
        // drain: every MMA this thread issued completes before tensor memory is freed
        if constexpr (CG == 2)
          tc_commit_pair(drain_bar, 0x1);
        else
          tc_commit(drain_bar);
        volatile int no_abort = 0;
        (void)mbar_wait(drain_bar, 0, ctl, &no_abort);
      }
    }
  } else if (warp >= DEC_WARP0 && warp < DEC_WARP0 + DEC_WARPS) {
    // ---------------- decoders: warps own stage slots ----------------
    // (the warps of a slot take its phases in order, so a parity wait can
    // never be satisfied by the slot's previous phase)
    if constexpr (C::QUANT) {
      constexpr int WPS = C::WARPS_PER_SLOT;
      const int s = (warp - DEC_WARP0) / WPS;
      const int part = (warp - DEC_WARP0) % WPS;
      if (s < S) {  // (Q6_K's four slots leave two decoder warps idle)
        // a follower's warps arrive on the issuing CTA's barrier directly
        const uint32_t done_bar = CG == 2 ? mapa_shared(full_dec(s), 0) : full_dec(s);
        // walk this warp's stages s, s + S, ... of the unit's segments
        // without per-stage divisions (c: the next one, counted from the
        // current segment's first stage)
        Segs<SK> sg(unit, n_units, n_tiles, n_chunks);
        int tile = 0, c0 = 0, c1 = 0;
        int c = s;
        uint32_t ph = 0;
        bool run = true;
        while (run && sg.next(tile, c0, c1)) {
          const int len = c1 - c0;
          if (c >= len) {
            c -= len;
            continue;
          }
          int ku, tt;
          coords(tile, ku, tt);
          const int kt = ku * CG + static_cast<int>(rank);
          // chunks of this item from c_ad on are the adapter's (TMA fills A)
          int c_ad = 0;
          if constexpr (AD) c_ad = n_main - (tile / n_tiles1) * n_chunks;
          for (; c < len; c += S, ph ^= 1u) {
            const int cc = c0 + c;  // the chunk of the item
            if (!__all_sync(0xffffffffu, mbar_wait(full_p(s), ph, ctl, abort_flag))) {
              run = false;
              break;
            }
            if constexpr (FWD) {
              // chunk gf: values 64 gf .. 64 gf + 63 of this CTA's 128 rows of W
              const int gf = (tile / n_tiles1) * n_chunks + cc;
              decode_fwd_stage<WT>(sP + s * C::P_STAGE, sA + s * A_STAGE, lane, part, gf >> 1, gf & 1);
            } else if (AD && cc >= c_ad) {
              // nothing to decode
            } else if constexpr (WT == RG_Q6_K || WT == RG_Q3_K || WT == RG_Q2_K) {
              // the super-block starts o bytes into its window: one decoder per
              // o (Q6_K, Q3_K: any even o; Q2_K: a multiple of 4)
              const int o = ((kt >> 1) * block_bytes(WT)) & 15;
              const uint8_t* P = sP + s * C::P_STAGE;
              uint8_t* Ad = sA + s * A_STAGE;
#define RG_WIN_CASE(OO)                                                          \
  case OO / 2:                                                                   \
    if constexpr (WT != RG_Q2_K || OO % 4 == 0) {                                \
      if (kt & 1) decode_stage_warp<WT, 1, WPS, OO>(P, Ad, lane, part);          \
      else decode_stage_warp<WT, 0, WPS, OO>(P, Ad, lane, part);                 \
    }                                                                            \
    break;
              switch (o >> 1) {
                RG_WIN_CASE(0) RG_WIN_CASE(2) RG_WIN_CASE(4) RG_WIN_CASE(6)
                RG_WIN_CASE(8) RG_WIN_CASE(10) RG_WIN_CASE(12) RG_WIN_CASE(14)
                default: break;
              }
#undef RG_WIN_CASE
            } else if constexpr (WT == RG_MXFP4 || WT == RG_NVFP4) {
              // the tile's blocks start (kt * 68) mod 16 = 0, 4, 8 or 12 (MXFP4)
              // or (kt * 72) mod 16 = 0 or 8 (NVFP4) bytes into the window
              decode_stage_warp<WT, 0, WPS>(sP + s * C::P_STAGE, sA + s * A_STAGE, lane, part,
                                            WT == RG_MXFP4 ? (kt * 68) & 12 : (kt & 1) * 8);
          } else if (kt & 1) {
              decode_stage_warp<WT, 1, WPS>(sP + s * C::P_STAGE, sA + s * A_STAGE, lane, part);
            } else {
              decode_stage_warp<WT, 0, WPS>(sP + s * C::P_STAGE, sA + s * A_STAGE, lane, part);
            }
            if (!AD || cc < c_ad) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if constexpr (CG == 2)
                mbar_arrive_cluster(done_bar);
              else
                mbar_arrive(done_bar);
            }
          }
          c -= len;
        }
      }
    }
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue ----------------
    const int eq = warp & 3;  // TMEM lanes 32*eq .. 32*eq+31
    const uint32_t empty_leader = CG == 2 ? mapa_shared(acc_empty(0), 0) : acc_empty(0);
    // split contraction: raw partial sums to part[split] (beta in the reduce);
    // stream-K plans never split (part holds their slabs)
    float* split_part = SK ? nullptr : part;
    // stream-K: one partial slab per unit ([unit][CTA of the pair]
    // [epilogue warp][t of the tile][lane]), one warp's piece SLAB_W floats
    constexpr int SLAB_W = BT * 32;
    constexpr int ER = C::EPI_ROWS;  // rows of t in a staged box
    float* stg = reinterpret_cast<float*>(smem + C::OFF_EPI) + eq * (2 * ER * 32);
    bool ok = true;
    Segs<SK> sg(unit, n_units, n_tiles, n_chunks);
    int tile = 0, c0 = 0, c1 = 0;
    for (int j = 0; ok && sg.next(tile, c0, c1); ++j) {
      int ku, tt;
      coords(tile, ku, tt);
      const int kt = ku * CG + static_cast<int>(rank);
      const int a = j & 1;
      const uint32_t aph = (static_cast<uint32_t>(j) >> 1) & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(acc_full(a), aph, ctl, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int k = kt * BM + 32 * eq + lane;
      const bool kin = k < K;
      if (!SK || c0 == 0) {
        // a whole item, or the first piece of a shared tile (the second
        // kernel adds the others to it): straight to dX (or to its split's slab)
        float* out = split_part ? split_part + static_cast<int64_t>(tile / n_tiles1) * T * K : dX;
        const float b = split_part ? 0.0f : beta;
        const int64_t ldo = split_part ? static_cast<int64_t>(K) : ldx;  // row stride of `out`
        // dX with beta 0 or 1, or a split's partial sums: 16 x 32 boxes staged
        // in shared memory and written by bulk tensor stores (beta 1: bulk
        // adds into dX; a split's slab: a 3-D map, the split the third
        // coordinate), so the warp issues 16 shared stores a box instead of
        // 16 global ones a row of lanes; other beta are stored element by
        // element
        const bool bulk = b == 0.0f || b == 1.0f;
        const int split = tile / n_tiles1;
#pragma unroll 1
        for (int cb = 0; cb < BT / 32; ++cb) {
          const int tb = tt * BT + 32 * cb;
          float old[32];
          if (!bulk && b != 0.0f && kin) {
            // all loads of the column block first: one round trip, not 32
#pragma unroll
            for (int i = 0; i < 32; ++i)
              old[i] = (tb + i < T) ? out[static_cast<int64_t>(tb + i) * ldo + k] : 0.0f;
          }
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * eq) << 16) +
                                 static_cast<uint32_t>(a * BT + 32 * cb),
                             r);
          if (bulk) {
#pragma unroll
            for (int h = 0; h < 32 / ER; ++h) {
              float* half = stg + (h & 1) * (ER * 32);
              // the store issued from this box two boxes ago has read it
              if (lane == 0) bulk_wait_read_1();
              __syncwarp();
#pragma unroll
              for (int i = 0; i < ER; ++i) half[i * 32 + lane] = __uint_as_float(r[ER * h + i]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                const int x = kt * BM + 32 * eq, y = tb + ER * h;
                if (x < K && y < T) {
                  if (split_part)
                    tma_store_3d(&map_p, smem_addr(half), x, y, split);
                  else if (b == 0.0f)
                    tma_store_2d(&map_x, smem_addr(half), x, y);
                  else
                    tma_add_2d(&map_x, smem_addr(half), x, y);
                }
                bulk_commit();
              }
            }
          } else if (kin) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (tb + i < T) {
                const float v = __uint_as_float(r[i]);
                out[static_cast<int64_t>(tb + i) * ldo + k] = b != 0.0f ? fmaf(b, old[i], v) : v;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 2)
            mbar_arrive_cluster(empty_leader + 8u * a);
          else
            mbar_arrive(acc_empty(a));
        }
      } else if constexpr (SK) {
        // a later piece of a tile shared by several units: raw partial sums
        // to its slab; a second kernel adds them, in chunk order, to dX
        float* mine = part + (static_cast<int64_t>(unit) * CG * 4 + static_cast<int64_t>(rank) * 4 + eq) *
                                 SLAB_W;
#pragma unroll 1
        for (int cb = 0; cb < BT / 32; ++cb) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * eq) << 16) +
                                 static_cast<uint32_t>(a * BT + 32 * cb),
                             r);
          // rows 32cb .. 32cb+31 of the piece are 4 KB of the slab: staged
          // boxes of ER rows, each one bulk copy
#pragma unroll
          for (int h = 0; h < 32 / ER; ++h) {
            float* half = stg + (h & 1) * (ER * 32);
            if (lane == 0) bulk_wait_read_1();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < ER; ++i) half[i * 32 + lane] = __uint_as_float(r[ER * h + i]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              bulk_store(mine + (32 * cb + ER * h) * 32, smem_addr(half), ER * 32 * 4);
              bulk_commit();
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 2)
            mbar_arrive_cluster(empty_leader + 8u * a);
          else
            mbar_arrive(acc_empty(a));
        }
      }
    }
    // the bulk stores have completed (their staging is freed with the CTA)
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (CG == 2)
    cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2)
      tmem_dealloc2(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace tc

// --- launch templates ---------------------------------------------------------

template <int WT, int CG, int BT, bool AD, bool SK, bool FWD>
static cudaError_t launch_tc_t(const CUtensorMap& mw, const CUtensorMap& my,
                               const CUtensorMap& ml, const CUtensorMap& mx, const CUtensorMap& mp,
                               const CUtensorMap& mq, int n_main, float* dX, int64_t ldx,
                               float beta, int T, int K, const TcPlan& p, float* part,
                               const DevInfo& dev, cudaStream_t stream) {
  using C = tc::Cfg<WT, CG, BT, FWD>;
  auto kern = tc::out_prod_tc_kernel<WT, CG, BT, AD, SK, FWD>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  WaitCtl ctl{dev.status, dev.wait_limit_ns};
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(tc::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // its prologue (barriers, tensor memory, tensor-map prefetch) overlaps the
  // end of the conversion kernel before it; the producer waits for that
  // kernel before its first copy
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // persistent grid: no more clusters than can be resident at once
  // (per device; threads that race on the first call store the same value)
  static std::atomic<int> max_clusters[64];
  std::atomic<int>& mc_slot = max_clusters[dev.device & 63];
  int mc = mc_slot.load(std::memory_order_relaxed);
  if (mc == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(CG * (dev.num_sms / CG)), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0)
      n = dev.num_sms / CG;
    mc_slot.store(n, std::memory_order_relaxed);
    mc = n;
  }
  const int units = std::min(p.grid / CG, mc);
  cfg.gridDim = dim3(static_cast<unsigned>(units * CG), 1, 1);
  if (SK && part == nullptr) return cudaErrorInvalidValue;
  e = counted(cudaLaunchKernelEx(&cfg, kern, mw, my, ml, mx, mp, mq, n_main, dX, ldx, beta, T, K, p.n_kunits,
                                 p.n_ttiles, p.band, p.n_chunks, p.n_splits, part, ctl));
  if (e != cudaSuccess || !SK) return e;
  // stream-K: the shared tiles' pieces, added in chunk order (the same unit
  // count as the launch: the pieces' slabs follow from it)
  return launch_sk_fixup(part, units, CG, BT, p, T, K, dX, ldx, dev, stream);
}

template <int WT, bool AD, bool SK, bool FWD>
static cudaError_t launch_tc_w(const CUtensorMap& mw, const CUtensorMap& my,
                               const CUtensorMap& ml, const CUtensorMap& mx, const CUtensorMap& mp,
                               const CUtensorMap& mq, int n_main, float* dX, int64_t ldx, float beta,
                               int T, int K, const TcPlan& p, float* part, const DevInfo& dev,
                               cudaStream_t stream) {
  if (p.cg == 2)
    return launch_tc_t<WT, 2, 256, AD, SK, FWD>(mw, my, ml, mx, mp, mq, n_main, dX, ldx, beta, T, K, p,
                                                part, dev, stream);
  return launch_tc_t<WT, 1, 128, AD, SK, FWD>(mw, my, ml, mx, mp, mq, n_main, dX, ldx, beta, T, K, p,
                                              part, dev, stream);
}

// The body of launch_tc: AD = an adapter rides along (rank > 0).  W is N
// rows of K values either way; FWD (the forward mul_mat) contracts over the
// K values of each row into an output N wide, the OUT_PROD over the N rows
// into an output K wide.  dy16 (dY's or X's 16-bit copy) has one row of the
// contraction's length per row of the output's T.
// zeroed: dX was set to zero before this launch (by the dY conversion) and
// the plan splits the contraction in two: both halves are added into dX by
// the epilogue's bulk adds (two adds onto an exact zero give the same bits
// in either order), no partial sums and no reduction kernel.
template <bool AD, bool SK, bool FWD = false>
static cudaError_t launch_tc_impl(int wtype, const void* W, int64_t N, int64_t K,
                                  const uint16_t* dy16, int64_t ld_dy16, int64_t T, float* dX,
                                  int64_t dx_t, float beta, float* part, const DevInfo& dev,
                                  cudaStream_t stream, int cg_force, const uint16_t* a16,
                                  int64_t rank, bool zeroed = false) {
  // with an adapter the contraction runs over tc_adapter_cols(N, r) columns
  // of dy16: dY's N, zeros to the chunk boundary, then the adapter's rank
  const int64_t n_ext = FWD ? K : rank > 0 ? tc_adapter_cols(N, rank) : N;
  const int64_t k_out = FWD ? N : K;  // the output's width
  const int n_main = rank > 0 ? static_cast<int>((N + tc::BC - 1) / tc::BC) : (1 << 30);
  TcPlan p = plan_tc(n_ext, k_out, T, dev, cg_force);
  if (p.sk != SK) return cudaErrorInvalidValue;  // the dispatcher chose the other build
  if (zeroed && (p.n_splits != 2 || p.sk)) return cudaErrorInvalidValue;
  if ((p.n_splits > 1 || p.sk) && part == nullptr && !zeroed) return cudaErrorInvalidValue;
  float* partial = (p.n_splits > 1 || p.sk) && !zeroed ? part : nullptr;
  if (zeroed) beta = 1.0f;  // each half adds itself to dX
  p.band = tc_band(wtype, n_ext, p);
  CUtensorMap mw, my, mq, m3;
  CUresult r;
  if (is_quant(wtype)) {
    const uint64_t rb = static_cast<uint64_t>(K / block_values(wtype) * block_bytes(wtype));
    const uint32_t box_bytes = static_cast<uint32_t>(with_wtype(wtype, 0, [](auto wt) {
      return FWD ? tc::p_fwd_row_bytes<decltype(wt)::value>() : tc::p_row_bytes<decltype(wt)::value>();
    }));
    // a stage's packed windows: 64 contraction rows, or the forward's 128 output rows
    // (the forward's Q4_K: the 16-byte headers here, the 32 nibble bytes in map_l)
    const bool split = FWD && wtype == RG_Q4_K;
    const bool split6 = FWD && wtype == RG_Q6_K;  // three windows: low bits, high bits, scales
    const uint32_t box_words = split ? 4 : (FWD && wtype == RG_Q8_0) ? 20 : split6 ? tc::Q6F_A / 4
                                                                              : box_bytes / 4;
    r = encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rb / 4, static_cast<uint64_t>(N), rb,
                     box_words, FWD ? 2 * tc::BC : tc::BC, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r == CUDA_SUCCESS && (split || split6))
      r = encode_tiled(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rb / 4, static_cast<uint64_t>(N), rb,
                       split ? 8 : tc::Q6F_H / 4, 2 * tc::BC, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r == CUDA_SUCCESS && split6)
      r = encode_tiled(&m3, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rb / 4, static_cast<uint64_t>(N), rb,
                       tc::Q6F_S / 4, 2 * tc::BC, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    r = encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, W, static_cast<uint64_t>(K),
                     static_cast<uint64_t>(N), static_cast<uint64_t>(K) * 2, 64,
                     FWD ? 2 * tc::BC : tc::BC, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  r = encode_tiled(&my, CU_TENSOR_MAP_DATA_TYPE_UINT16, dy16, static_cast<uint64_t>(n_ext),
                   static_cast<uint64_t>(T), static_cast<uint64_t>(ld_dy16) * 2, tc::BC,
                   tc::B_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // the adapter's rows [rank, K] (16-bit, same kind as the decoded W), or the
  // forward's Q4_K nibble copies; else a copy that no stage reads
  CUtensorMap ml = (FWD && (wtype == RG_Q4_K || wtype == RG_Q6_K)) ? mq : mw;
  // the forward Q6_K's scales window; else a copy that no stage reads
  if (!(FWD && wtype == RG_Q6_K)) m3 = mw;
  if (rank > 0) {
    r = encode_tiled(&ml, CU_TENSOR_MAP_DATA_TYPE_UINT16, a16, static_cast<uint64_t>(K),
                     static_cast<uint64_t>(rank), static_cast<uint64_t>(K) * 2, 64, tc::BC,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // the output for the epilogue's bulk stores: F32 [T, k_out], rows dx_t
  // apart, boxes of 32 values by the kernel's staged rows
  const uint32_t er = static_cast<uint32_t>(with_wtype(wtype, 16, [&](auto wt) {
    constexpr int W_ = decltype(wt)::value;
    return p.cg == 2 ? tc::Cfg<W_, 2, 256, FWD>::EPI_ROWS : tc::Cfg<W_, 1, 128, FWD>::EPI_ROWS;
  }));
  CUtensorMap mx;
  r = encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dX, static_cast<uint64_t>(k_out),
                   static_cast<uint64_t>(T), static_cast<uint64_t>(dx_t) * 4, 32, er,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // a split contraction's partial sums [n_splits][T][k_out], the split the third dimension
  CUtensorMap mp = mx;
  if (p.n_splits > 1 && partial != nullptr) {
    r = encode_tiled(&mp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, partial, static_cast<uint64_t>(k_out),
                     static_cast<uint64_t>(T), static_cast<uint64_t>(k_out) * 4, 32, er,
                     CU_TENSOR_MAP_SWIZZLE_NONE, static_cast<uint64_t>(p.n_splits),
                     static_cast<uint64_t>(T) * static_cast<uint64_t>(k_out) * 4);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const int t = static_cast<int>(T), k = static_cast<int>(k_out);
  const cudaError_t e = with_wtype(wtype, cudaErrorInvalidValue, [&](auto wt) {
    return launch_tc_w<decltype(wt)::value, AD, SK, FWD>(mw, my, ml, mx, mp, m3, n_main, dX, dx_t, beta,
                                                        t, k, p, partial, dev, stream);
  });
  if (e != cudaSuccess || p.n_splits == 1 || zeroed) return e;
  return launch_reduce_partials(partial, p.n_splits, T, k_out, dX, dx_t, beta, dev, stream);
}

// launch_tc with an adapter (rg_tc_ad.cu; its plans never take stream-K) and
// the stream-K plans (rg_tc_sk.cu)
cudaError_t launch_tc_adapter(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                              int64_t ld_dy16, int64_t T, float* dX, int64_t dx_t, float beta,
                              float* part, const DevInfo& dev, cudaStream_t stream, int cg_force,
                              const uint16_t* a16, int64_t rank);
cudaError_t launch_tc_stream_k(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                               int64_t ld_dy16, int64_t T, float* dX, int64_t dx_t, float beta,
                               float* part, const DevInfo& dev, cudaStream_t stream, int cg_force);

}  // namespace rg
