// rg_internal.cuh - device helpers shared by the librg kernels (sm_103a).
//
// Inline PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), the 5th
// generation tensor core (tcgen05: tensor-memory alloc, mma, commit, ld), the
// bounded waits every kernel uses, and the exact F32 block decoders used by
// the dequant, SIMT and small-T kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rg.h"

namespace rg {

// ---------------------------------------------------------------------------
// storage formats: values per block, bytes per block

__host__ __device__ constexpr bool valid_wtype(int wt) { return wt >= RG_F16 && wt <= RG_NVFP4; }
__host__ __device__ constexpr bool is_quant(int wt) {
  return valid_wtype(wt) && wt != RG_F16 && wt != RG_BF16 && wt != RG_F32;
}
__host__ __device__ constexpr int block_values(int wt) {
  return (wt == RG_Q4_K || wt == RG_Q5_K || wt == RG_Q6_K || wt == RG_Q2_K || wt == RG_Q3_K) ? 256
         : wt == RG_NVFP4                                                                 ? 64
         : is_quant(wt)                                                                   ? 32
                                                                                          : 1;
}
__host__ __device__ constexpr int block_bytes(int wt) {
  return wt == RG_Q4_K   ? 144
         : wt == RG_Q5_K ? 176
         : wt == RG_Q6_K ? 210
         : wt == RG_Q2_K ? 84
         : wt == RG_Q3_K ? 110
         : wt == RG_Q8_0 ? 34
         : wt == RG_Q4_0 ? 18
         : wt == RG_Q4_1 ? 20
         : wt == RG_Q5_0 ? 22
         : wt == RG_Q5_1 ? 24
         : wt == RG_MXFP4 ? 17
         : wt == RG_NVFP4 ? 36
         : wt == RG_F32  ? 4
                         : 2;
}

// Everything a kernel needs to report a wait that gave up.
struct WaitCtl {
  int* status;                   // per-device status word (global memory)
  unsigned long long limit_ns;   // give up after this long
};

// ---------------------------------------------------------------------------
// small device utilities

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void report_timeout(int* status) {
  atomicCAS(status, 0, (int)RG_ERR_TIMEOUT);
}
__device__ __forceinline__ void report_range(int* status) {
  atomicCAS(status, 0, (int)RG_ERR_RANGE);
}

// Whether the finite F32 value v became +-inf when rounded to the 16-bit
// operand kind (bits16: fp16, or bf16 when BF16): a value beyond the kind's
// range (fp16: |v| >= 65520), which the tensor cores would carry as inf.
template <bool BF16>
__device__ __forceinline__ bool overflowed16(float v, uint32_t bits16) {
  constexpr uint32_t INF = BF16 ? 0x7F80u : 0x7C00u;
  return (bits16 & 0x7FFFu) == INF && fabsf(v) <= 3.40282347e38f;  // false for NaN and inf
}

// fp16 bits -> F32 (exact: every binary16 value is a float32).
__device__ __forceinline__ float f16_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}
// bf16 bits -> F32 (the bits are the top half of the float32 word).
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Byte B of x (an unsigned integer u < 256) as the F32 value u - bias, exactly
// and without the integer-conversion unit: the word 0x4B0000uu is the float
// 2^23 + u (u sits in the low mantissa bits), and subtracting 2^23 + bias is
// exact for these small integers.
template <int B>
__device__ __forceinline__ float byte_minus(uint32_t x, float two23_plus_bias) {
  return __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u | B)) - two23_plus_bias;
}
constexpr float kTwo23 = 8388608.0f;  // 2^23

// Bit i (i = 0..3) of v -> bit 4 of byte i: the fifth bits of four
// consecutive Q5 values, ready to OR onto their nibbles.  The multiply by
// 1 + 2^7 + 2^14 + 2^21 places copies of v at bits 0, 7, 14, 21 (no carries
// between them), so bit 8i of the product is bit i of v.
__device__ __forceinline__ uint32_t fifth_bits4(uint32_t v) {
  return (((v & 15u) * 0x00204081u) & 0x01010101u) << 4;
}

// ---------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with this parity has completed.  Gives up when the
// CTA's abort flag is raised or after ctl.limit_ns; a thread that gives up on
// its own raises the abort flag and records RG_ERR_TIMEOUT.  Returns false on
// giving up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl,
                                          volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > ctl.limit_ns) {
        *abort_flag = 1;
        report_timeout(ctl.status);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// TMA

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled load of one box at element coordinates (x inner, y outer) into
// shared memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// The same load issued by either CTA of a pair, counted on a barrier that may
// live in the peer CTA (`bar_cluster`: a shared::cluster address, e.g. from
// mapa): both CTAs' operand halves then complete on the MMA-issuing CTA's
// barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

// Bulk tensor store of a box from shared memory to global memory (its
// elements outside the tensor are not written), or element-wise add of the
// box into global memory (F32 add, as one rounding each); both join this
// thread's current bulk group.  x (innermost) must be 16-byte aligned.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from shared to global memory, in this thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until at most one of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the kernel before it on the stream still
// runs; pdl_wait() returns once that kernel has completed and its writes are
// visible, and pdl_launch_dependents() (in the earlier kernel) lets the
// dependent kernel be scheduled before this one ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (one CTA per MMA: cta_group::1)

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// D(tmem) (+)= A(smem desc) x B(smem desc), fp16/bf16 inputs, F32 accumulate.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// --- pairs of CTAs (cta_group::2): one MMA spans the tensor cores of two SMs
// of a cluster; the even-ranked CTA issues it, each CTA supplies half of A
// (rows of M) and half of B (columns of N) from its own shared memory at the
// same offsets, and each CTA's tensor memory holds its half of D.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Address in the shared::cluster window of the variable at `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its shared::cluster address (possibly in the
// peer CTA), with the default release semantics: the pipeline handshake of a
// pair.  The data it publishes lives in the arriving CTA's own shared memory
// and is read there by that CTA's tensor core, after a proxy fence.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for barriers that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const WaitCtl& ctl,
                                                  volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > ctl.limit_ns) {
        *abort_flag = 1;
        report_timeout(ctl.status);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at this shared offset in every CTA of `mask`
// when the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes (lane i of the
// warp reads TMEM lane base+i), waited for before returning.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor of the tcgen05 MMA: start address, leading
// and stride byte offsets (all >> 4), descriptor version 1 (bits 46-47),
// 128-byte swizzle (layout code 2 in bits 61-63).  Tiles are 1024-byte
// aligned, so the base-offset field stays 0.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: F32 accumulator (bit 4),
// A and B both F16 (0) or both BF16 (1) in bits 7-9 / 10-12, A MN-major
// (bit 15), B K-major (bit 16 clear), N >> 3 in bits 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N, bool a_mn_major,
                                                 bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// exact F32 decode of 8 consecutive values of a stored row
//
// row: the row's first byte (global or shared memory, at least 2-byte
// aligned); k0: first value, a multiple of 8.  out[i] = deq(W)[row][k0 + i],
// bit for bit: Q8_0 d*q and Q4_0 d*(q-8) are exact products (signed zero
// kept, since a product is taken rather than a select); Q4_K's
// (d*sc)*q - dmin*m has exact products and one rounding, so fused or
// unfused evaluation gives the same word.

__device__ __forceinline__ uint16_t ld_u16(const uint8_t* p) {
  return *reinterpret_cast<const uint16_t*>(p);
}

__device__ __forceinline__ void q4k_scale_min(const uint8_t* S, int j, int& sc, int& m) {
  if (j < 4) {
    sc = S[j] & 63;
    m = S[j + 4] & 63;
  } else {
    sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4);
    m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4);
  }
}

// OCP microscaling fields (MXFP4).  E8M0 scale: 2^(e - 127), the float32
// with biased exponent e; e = 0 is the subnormal 2^-127, e = 255 NaN.
__device__ __forceinline__ float e8m0_f32(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u)
                : (e == 255 ? __uint_as_float(0x7FC00000u) : __uint_as_float(e << 23));
}
// E2M1 element (4-bit code): bit 3 sign, bits 2-1 exponent (bias 1), bit 0
// mantissa: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives (code 8: -0.0).
__device__ __forceinline__ float e2m1_f32(uint32_t c) {
  const uint32_t m = c & 7u;
  const uint32_t mag = m >= 2u ? (((m >> 1) + 126u) << 23) | ((m & 1u) << 22) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((c & 8u) << 28));
}

// FP8 E4M3 (NVFP4's micro-block scale): bit 7 sign, 4 exponent bits (bias
// 7), 3 mantissa bits; exponent 0 is m/8 * 2^-6, 0x7f / 0xff NaN, no
// infinities.  Exact in F32 (and in fp16: 2^-9 .. 448, four significant bits).
__device__ __forceinline__ float e4m3_f32(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float mag;
  if (e == 0)
    mag = static_cast<float>(m) * 0.001953125f;  // m * 2^-9, exact
  else
    mag = __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) * 2^(e - 7)
  if (e == 15 && m == 7) mag = __uint_as_float(0x7FC00000u);
  return (c & 0x80u) ? -mag : mag;
}

template <int WT>
__device__ __forceinline__ void decode8_f32(const uint8_t* row, int k0, float (&out)[8]) {
  if constexpr (WT == RG_NVFP4) {
    // E2M1(code) * E4M3(d[s]): an exact product (two and four significant
    // bits); values 8h .. 8h+7 of micro-block s are the low (h = 0) or high
    // (h = 1) nibbles of its eight bytes
    const uint8_t* blk = row + (k0 >> 6) * 36;
    const int v0 = k0 & 63, s = v0 >> 4, shift = (v0 & 8) ? 4 : 0;
    const float sc = e4m3_f32(blk[s]);
    const uint8_t* qs = blk + 4 + 8 * s;
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = e2m1_f32((qs[i] >> shift) & 15u) * sc;
  } else if constexpr (WT == RG_MXFP4) {
    // E2M1(code) * 2^(e - 127): an exact product (a power of two times a
    // two-bit significand; subnormal and overflowing results as IEEE gives)
    const uint8_t* blk = row + (k0 >> 5) * 17;
    const float sc = e8m0_f32(blk[0]);
    const int j = k0 & 31;  // 0, 8, 16 or 24
    const uint8_t* qs = blk + 1 + (j & 15);
    const int shift = j >= 16 ? 4 : 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = e2m1_f32((qs[i] >> shift) & 15u) * sc;
  } else if constexpr (WT == RG_F32) {
    const float4 a = *reinterpret_cast<const float4*>(row + 4 * k0);
    const float4 b = *reinterpret_cast<const float4*>(row + 4 * k0 + 16);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
  } else if constexpr (WT == RG_F16 || WT == RG_BF16) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + 2 * k0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = static_cast<uint16_t>(w[i] & 0xFFFFu);
      const uint16_t hi = static_cast<uint16_t>(w[i] >> 16);
      out[2 * i] = WT == RG_F16 ? f16_to_f32(lo) : bf16_to_f32(lo);
      out[2 * i + 1] = WT == RG_F16 ? f16_to_f32(hi) : bf16_to_f32(hi);
    }
  } else if constexpr (WT == RG_Q8_0) {
    const uint8_t* blk = row + (k0 >> 5) * 34;
    const float d = f16_to_f32(ld_u16(blk));
    const int8_t* qs = reinterpret_cast<const int8_t*>(blk + 2 + (k0 & 31));
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = d * static_cast<float>(qs[i]);
  } else if constexpr (WT == RG_Q4_0) {
    const uint8_t* blk = row + (k0 >> 5) * 18;
    const float d = f16_to_f32(ld_u16(blk));
    const int j = k0 & 31;  // 0, 8, 16 or 24
    const uint8_t* qs = blk + 2 + (j & 15);
    const int shift = j >= 16 ? 4 : 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      out[i] = d * static_cast<float>(static_cast<int>((qs[i] >> shift) & 15) - 8);
  } else if constexpr (WT == RG_Q4_K) {
    const uint8_t* blk = row + (k0 >> 8) * 144;
    const float d = f16_to_f32(ld_u16(blk));
    const float dmin = f16_to_f32(ld_u16(blk + 2));
    const int e = k0 & 255;
    const int c = e >> 6, half = (e >> 5) & 1, l0 = e & 31;
    int sc, m;
    q4k_scale_min(blk + 4, 2 * c + half, sc, m);
    const float ds = d * static_cast<float>(sc);
    const float dm = dmin * static_cast<float>(m);
    const uint8_t* qs = blk + 16 + 32 * c + l0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = half ? (qs[i] >> 4) : (qs[i] & 15);
      out[i] = ds * static_cast<float>(q) - dm;
    }
  } else if constexpr (WT == RG_Q4_1 || WT == RG_Q5_0 || WT == RG_Q5_1) {
    // 32-value blocks: d (and m), the fifth bits (Q5), 16 bytes of nibbles
    constexpr int BB = block_bytes(WT);
    constexpr int QS = WT == RG_Q4_1 ? 4 : WT == RG_Q5_0 ? 6 : 8;
    const uint8_t* blk = row + (k0 >> 5) * BB;
    const float d = f16_to_f32(ld_u16(blk));
    const int j = k0 & 31;  // 0, 8, 16 or 24
    const uint8_t* qs = blk + QS + (j & 15);
    const int shift = j >= 16 ? 4 : 0;
    uint32_t qh = 0;
    if constexpr (WT != RG_Q4_1) {
      constexpr int QH = WT == RG_Q5_0 ? 2 : 4;
      qh = static_cast<uint32_t>(ld_u16(blk + QH)) | (static_cast<uint32_t>(ld_u16(blk + QH + 2)) << 16);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = ((qs[i] >> shift) & 15) | (static_cast<int>((qh >> (j + i)) & 1u) << 4);
      if constexpr (WT == RG_Q5_0) {
        out[i] = d * static_cast<float>(q - 16);  // exact
      } else {
        // exact product, one rounding of the sum
        out[i] = fmaf(d, static_cast<float>(q), f16_to_f32(ld_u16(blk + 2)));
      }
    }
  } else if constexpr (WT == RG_Q6_K) {
    // value v = 128h + 32i + l: nibble of ql[64h + 32(i%2) + l] (high for
    // i >= 2), bits 2i..2i+1 of qh[32h + l]; (d * sc) * (q - 32) is exact
    const uint8_t* blk = row + (k0 >> 8) * 210;
    const int v0 = k0 & 255;
    const int h = v0 >> 7, i = (v0 >> 5) & 3, l0 = v0 & 31;
    const uint8_t* ql = blk + 64 * h + 32 * (i & 1) + l0;
    const uint8_t* qh = blk + 128 + 32 * h + l0;
    const float ds = f16_to_f32(ld_u16(blk + 208)) *
                     static_cast<float>(static_cast<int8_t>(blk[192 + (v0 >> 4)]));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = ((i >= 2 ? (ql[j] >> 4) : ql[j]) & 15) | (((qh[j] >> (2 * i)) & 3) << 4);
      out[j] = ds * static_cast<float>(q - 32);
    }
  } else if constexpr (WT == RG_Q2_K) {
    // value v = 128h + 32j + 16s + l: bits 2j.. of qs[32h + 16s + l], scales
    // byte 8h + 2j + s; (d * sc) * q exact, minus dmin * m rounded once
    const uint8_t* blk = row + (k0 >> 8) * 84;
    const int v0 = k0 & 255;
    const int h = v0 >> 7, j = (v0 >> 5) & 3, sb = (v0 >> 4) & 1, l0 = v0 & 15;
    const int b = blk[8 * h + 2 * j + sb];
    const float ds = f16_to_f32(ld_u16(blk + 80)) * static_cast<float>(b & 15);
    const float dm = f16_to_f32(ld_u16(blk + 82)) * static_cast<float>(b >> 4);
    const uint8_t* qs = blk + 16 + 32 * h + 16 * sb + l0;
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = fmaf(ds, static_cast<float>((qs[i] >> (2 * j)) & 3), -dm);
  } else if constexpr (WT == RG_Q3_K) {
    // value v = 128h + 32j + 16s + l: bits 2j.. of qs[32h + 16s + l], minus 4
    // unless bit 4h + j of hmask[16s + l]; (d * (sc - 32)) * q, all exact
    const uint8_t* blk = row + (k0 >> 8) * 110;
    const int v0 = k0 & 255;
    const int h = v0 >> 7, j = (v0 >> 5) & 3, sb = (v0 >> 4) & 1, l0 = v0 & 15;
    const int si = 8 * h + 2 * j + sb;
    const uint8_t* S = blk + 96;
    const int lo4 = si < 8 ? (S[si] & 15) : (S[si - 8] >> 4);
    const int hi2 = (S[8 + (si & 3)] >> (2 * (si >> 2))) & 3;
    const float ds = f16_to_f32(ld_u16(blk + 108)) * static_cast<float>((lo4 | (hi2 << 4)) - 32);
    const uint8_t* qs = blk + 32 + 32 * h + 16 * sb + l0;
    const uint8_t* hm = blk + 16 * sb + l0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = ((qs[i] >> (2 * j)) & 3) - (((hm[i] >> (4 * h + j)) & 1) ? 0 : 4);
      out[i] = ds * static_cast<float>(q);
    }
  } else if constexpr (WT == RG_Q5_K) {
    const uint8_t* blk = row + (k0 >> 8) * 176;
    const float d = f16_to_f32(ld_u16(blk));
    const float dmin = f16_to_f32(ld_u16(blk + 2));
    const int e = k0 & 255;
    const int c = e >> 6, half = (e >> 5) & 1, l0 = e & 31;
    int sc, m;
    q4k_scale_min(blk + 4, 2 * c + half, sc, m);
    const float ds = d * static_cast<float>(sc);
    const float dm = dmin * static_cast<float>(m);
    const uint8_t* qh = blk + 16 + l0;
    const uint8_t* qs = blk + 48 + 32 * c + l0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = (half ? (qs[i] >> 4) : (qs[i] & 15)) + 16 * ((qh[i] >> (2 * c + half)) & 1);
      out[i] = ds * static_cast<float>(q) - dm;
    }
  }
}

}  // namespace rg
