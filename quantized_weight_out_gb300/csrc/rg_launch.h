// rg_launch.h - host-side launchers shared between the librg translation
// units (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <utility>

#include "../../include/rg.h"

namespace rg {

struct WaitCtl;

// Per-device facts the launchers need.
struct DevInfo {
  int device;
  int num_sms;
  int max_smem_optin;   // bytes of dynamic shared memory a block may opt into
  int* status;          // device address of this device's status word
  unsigned long long wait_limit_ns;
};

// Kernels launched by this library (rg_launch_count); every launcher passes
// its launch status through counted().
extern std::atomic<unsigned long long> g_launch_count;
inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// f(std::integral_constant<int, WT>{}) for the run-time weight type wtype;
// `fallback` for a type the library does not know (callers validate first).
template <class R, class F>
R with_wtype(int wtype, R fallback, F&& f) {
  switch (wtype) {
    case RG_F16: return f(std::integral_constant<int, RG_F16>{});
    case RG_BF16: return f(std::integral_constant<int, RG_BF16>{});
    case RG_Q8_0: return f(std::integral_constant<int, RG_Q8_0>{});
    case RG_Q4_0: return f(std::integral_constant<int, RG_Q4_0>{});
    case RG_Q4_K: return f(std::integral_constant<int, RG_Q4_K>{});
    case RG_Q4_1: return f(std::integral_constant<int, RG_Q4_1>{});
    case RG_Q5_0: return f(std::integral_constant<int, RG_Q5_0>{});
    case RG_Q5_1: return f(std::integral_constant<int, RG_Q5_1>{});
    case RG_Q5_K: return f(std::integral_constant<int, RG_Q5_K>{});
    case RG_Q6_K: return f(std::integral_constant<int, RG_Q6_K>{});
    case RG_Q2_K: return f(std::integral_constant<int, RG_Q2_K>{});
    case RG_Q3_K: return f(std::integral_constant<int, RG_Q3_K>{});
    case RG_MXFP4: return f(std::integral_constant<int, RG_MXFP4>{});
    case RG_NVFP4: return f(std::integral_constant<int, RG_NVFP4>{});
    case RG_F32: return f(std::integral_constant<int, RG_F32>{});
    default: return fallback;
  }
}

// All launchers enqueue on `stream` and return cudaSuccess or the launch
// error; arguments are already validated by the entry points.
cudaError_t launch_dequant(int wtype, const void* W, int64_t N, int64_t K, float* out,
                           const DevInfo& dev, cudaStream_t stream);

// Element strides of the caller's activations: dY[t, n] at
// dY[t * dy_t + n * dy_n], dX[t, k] at dX[t * dx_t + k].
struct Layout {
  int64_t dy_t, dy_n, dx_t;
};

// deq(W)^T as fp16 (bf16 when `bf16`) [K, N], rows ldo values apart.
cudaError_t launch_dequant_t16(int wtype, const void* W, int64_t N, int64_t K, bool bf16,
                               uint16_t* out, int64_t ldo, const DevInfo& dev, cudaStream_t stream);

// Launch `kern` (a plain kernel: no cluster) so that it may be scheduled
// while the kernel before it on the stream finishes (programmatic stream
// serialization); the kernel must call pdl_wait() before it reads anything
// that kernel writes.  A kernel before it that never triggers its
// dependents (every kernel outside this library) is waited for as usual.
template <class... P, class... A>
cudaError_t launch_after_prev(void (*kern)(P...), dim3 grid, dim3 block, cudaStream_t stream,
                              A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

// Blocks of a grid-stride kernel over work_items (one per thread): enough
// for the items, at most eight per SM.
inline int grid_for(int64_t work_items, int threads, const DevInfo& dev) {
  const int64_t blocks = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
  return static_cast<int>(std::max<int64_t>(1, std::min(blocks, cap)));
}

// dY [T, N] (strided) F32 -> out [T, ld] fp16 (bf16 when `bf16`), rows padded to ld.
// mul != 1 (contiguous rows only) converts mul * dY.
// zero (optional, row-contiguous dY only): T rows of zk floats, zld apart,
// set to zero by the same kernel (zk, zld multiples of 4)
cudaError_t launch_convert_dy(const float* dY, int64_t T, int64_t N, int64_t dy_t, int64_t dy_n,
                              int64_t ld, bool bf16, uint16_t* out, const DevInfo& dev,
                              cudaStream_t stream, float mul = 1.0f, float* zero = nullptr,
                              int64_t zk = 0, int64_t zld = 0);

// --- the low-rank adapter (rg_adapter.cu) ---
// U [T, rank] (rows ldu floats apart) into columns [roundup8(N),
// tc_adapter_cols(N, rank)) of the 16-bit dY copy: zeros up to the chunk
// boundary after N, then U, then zeros.
cudaError_t launch_adapter_pack(const float* U, int64_t ldu, int64_t T, int64_t rank, int64_t N,
                                int64_t ld, bool bf16, uint16_t* out, const DevInfo& dev,
                                cudaStream_t stream);
// Ranks up to kAdapterFusedRank take the fused route: launch_convert_dy_adapter
// writes dY's 16-bit copy and U = dY . B (16-bit operands, F32 accumulation)
// after it in one pass over dY; bt is B^T [rank, ldb] 16-bit (ldb % 8 == 0),
// and the copy's columns are as launch_adapter_pack leaves them.  (A rank-64
// build of it cost more than the separate tensor-core product of U: its warp
// MMAs and B^T's re-reads from L2 grow with the rank.)
constexpr int64_t kAdapterFusedRank = 32;
cudaError_t launch_convert_dy_adapter(const float* dY, int64_t T, int64_t N, const uint16_t* bt,
                                      int64_t ldb, int64_t rank, int64_t ld, bool bf16,
                                      uint16_t* out, cudaStream_t stream);
// Ranges of n the F32 route splits dY . B into (its workspace holds
// parts * T * rank floats).
int adapter_down_parts(int64_t N, int64_t T, int64_t rank, const DevInfo& dev);
// dX [T, K] (rows dx_t apart) += scale * (dY . B) . A, all F32, dY and A
// row-contiguous and 16-byte aligned.
cudaError_t launch_adapter_f32(const float* dY, int64_t N, int64_t T, const float* A,
                               const float* B, int64_t rank, int64_t K, float scale, float* dX,
                               int64_t dx_t, float* part, int n_parts, const DevInfo& dev,
                               cudaStream_t stream);

// dX = beta * dX (beta == 0: dX = 0) over T rows of K, the N == 0 case.
cudaError_t launch_scale(float* dX, int64_t T, int64_t K, int64_t dx_t, float beta,
                         const DevInfo& dev, cudaStream_t stream);

cudaError_t launch_simt32(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, const Layout& lay, const DevInfo& dev,
                          cudaStream_t stream);

// Small-T path: rows of W split over n_splits CTAs per 256-value tile and
// dY chunk of tb rows; partial sums go to a workspace of `workspace` bytes
// ([n_splits][T][K] F32), then a second kernel adds them with beta * dX.
struct SmalltPlan {
  int tb;              // dY rows per pass: 1, 2, 4 or 8
  int n_ktiles;        // ceil(K / 256)
  int n_tchunks;       // ceil(T / tb)
  int n_splits;        // CTAs along N per tile (1: the kernel writes dX itself)
  int rows_per_split;  // rows of W per CTA (multiple of 8)
  size_t workspace;    // bytes of partial sums (0 for one slice)
};
// Sized so that the grid fills the GPU once at the kernel's residency.
SmalltPlan plan_smallt(int wtype, int64_t N, int64_t K, int64_t T, const DevInfo& dev);
// inject_stall (debug): the producer skips its first stage, whose wait then
// runs out (the bounded-wait path, tested without a fault)
cudaError_t launch_smallt(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                          int64_t T, float* dX, float beta, const Layout& lay, float* part,
                          const SmalltPlan& p, const DevInfo& dev, cudaStream_t stream,
                          int inject_stall = 0);
// The forward Y = beta * Y + X . deq(W)^T streaming W once per four rows of
// X (rg_mul_mat's route for one or two rows): one launch, no workspace.  X [T, K] and Y [T, N] row-major; W's rows
// must be 16-byte aligned (aligned_rows).
cudaError_t launch_smallt_fwd(int wtype, const void* W, int64_t N, int64_t K, const float* X, int64_t T,
                              float* Y, float beta, const DevInfo& dev, cudaStream_t stream);

// Tensor-core path.  dy16 is the converted dY with row stride ld_dy16 values.
struct TcPlan {
  int cg;        // CTAs per MMA: 2 (cta_group::2, 256 x 256 tiles) or 1 (128 x 128)
  int bt;        // t-columns per tile (MMA N): 256 (cg 2) or 128 (cg 1)
  int n_kunits;  // tiles along k: ceil(K / (128 * cg))
  int n_ttiles;  // tiles along t: ceil(T / bt)
  int n_chunks;  // ceil(N / 64) contraction stages per tile
  int grid;      // persistent CTAs (a multiple of cg), before the occupancy cap
  int band;      // k units per rasterization band (tile order), set at launch
  int n_splits;  // contraction split into this many ranges of n_chunks stages
  bool sk;       // stream-K: whole waves of tiles, then the last tiles' chunks
                 // shared evenly over the units (n_splits is 1)
};
// While one of these lives, tensor-core plans made on its thread leave
// stream-K out: the no-alloc entry point's fixed scratch has no room for the
// partial slabs (a whole tile per unit), and the adapter's kernels are built
// without stream-K.
struct NoStreamK {
  NoStreamK();
  ~NoStreamK();
  NoStreamK(const NoStreamK&) = delete;
  NoStreamK& operator=(const NoStreamK&) = delete;
};

// cg_force: 0 = choose from the shape, 1 or 2 = that tile configuration.
TcPlan plan_tc(int64_t N, int64_t K, int64_t T, const DevInfo& dev, int cg_force);
int64_t tc_dy16_ld(int64_t N);
// part: [n_splits][T][K] F32 partial sums when the plan splits the
// contraction (tc_partial_splits > 0), else unused.
// With a low-rank adapter (rank > 0): a16 holds its rows [rank, K] in the
// 16-bit kind of the product, and dy16 has tc_adapter_cols(N, rank) columns:
// dY's N values, zeros up to the next multiple of 64, then the rank values
// of the adapter's projected dY and zeros to the next multiple of 64.
// zeroed: dX was zeroed by the dY conversion and the plan splits the
// contraction in two (tc_adds_halves): both halves are bulk-added into dX,
// no partial sums, no reduction kernel.
cudaError_t launch_tc(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                      int64_t ld_dy16, int64_t T, float* dX, int64_t dx_t, float beta, float* part,
                      const DevInfo& dev, cudaStream_t stream, int cg_force,
                      const uint16_t* a16 = nullptr, int64_t rank = 0, bool zeroed = false);
// Whether an OUT_PROD with this beta runs its two contraction halves as adds
// into a dX the conversion zeroed: beta 0, row-contiguous dY, a plan split in
// exactly two (two adds onto an exact zero are order-independent; with more
// halves, or beta * dX under them, the order would show in the bits).
bool tc_adds_halves(int64_t N, int64_t K, int64_t T, float beta, bool dy_rows, const DevInfo& dev,
                    int cg_force);
// k units per rasterization band of a plan (see launch_tc).
int tc_band(int wtype, int64_t n_contr, const TcPlan& p);
int64_t tc_adapter_cols(int64_t N, int64_t rank);
// The forward mul_mat (rg_mm.cu): Y [T, N] (rows ldy apart) = beta * Y +
// X . deq(W)^T for W of N rows of K values (decoded inside the tensor-core
// kernel, contracted over each row's K values), x16 X's 16-bit copy [T, K]
// (rows ld_x16 apart); part: [n_splits][T][N] partial sums when the plan of
// (contraction K, output N, T) splits the contraction.  Stream-K is never
// taken (call it under NoStreamK).
// zeroed: as launch_tc's (Y zeroed by X's conversion, a plan split in two).
cudaError_t launch_mm(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* x16,
                      int64_t ld_x16, int64_t T, float* Y, int64_t ldy, float beta, float* part,
                      const DevInfo& dev, cudaStream_t stream, int cg_force, bool zeroed = false);
// Number of partial-sum slabs the tensor-core plan needs (0 when unsplit).
int64_t tc_partial_splits(int64_t N, int64_t K, int64_t T, const DevInfo& dev, int cg_force);
// Bytes of the `part` workspace the tensor-core plan needs: the splits'
// [n_splits][T][K] partial sums, or stream-K's partial slabs (a whole tile
// per unit), or 0.
size_t tc_partial_bytes(int64_t N, int64_t K, int64_t T, const DevInfo& dev, int cg_force);
// Stream-K's second pass: every tile the units shared (the plan's last
// tiles) already holds beta * dX + its first piece in dX; the later pieces'
// partial sums are added to it in chunk order from the slabs in `part` that
// `units` units of cg CTAs wrote.
cudaError_t launch_sk_fixup(const float* part, int units, int cg, int bt, const TcPlan& p, int T,
                            int K, float* dX, int64_t ldx, const DevInfo& dev,
                            cudaStream_t stream);

// dX = beta * dX + sum of n_splits slabs of [T, K] floats, in a fixed
// order; dX rows dx_t floats apart (a multiple of 4).
cudaError_t launch_reduce_partials(const float* part, int n_splits, int64_t T, int64_t K,
                                   float* dX, int64_t dx_t, float beta, const DevInfo& dev,
                                   cudaStream_t stream);

// A kernel whose one wait can never complete; it must give up after
// `limit_ns`, record RG_ERR_TIMEOUT and return.
cudaError_t launch_wait_probe(const DevInfo& dev, unsigned long long limit_ns,
                              cudaStream_t stream);

// cuTensorMapEncodeTiled (resolved from the driver at first use), through a
// small cache of recently encoded maps keyed by address, shape and device.
// dim2 > 1: a third dimension (rows of planes stride2_bytes apart), box 1 deep.
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                      uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                      uint32_t box1, CUtensorMapSwizzle swizzle, uint64_t dim2 = 1,
                      uint64_t stride2_bytes = 0);
CUresult encode_tiled_uncached(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                               uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                               uint32_t box1, CUtensorMapSwizzle swizzle, uint64_t dim2 = 1,
                               uint64_t stride2_bytes = 0);

// Raise `func`'s dynamic shared memory limit to `bytes` on the current device,
// once per (kernel, device).
cudaError_t ensure_smem_attr(const void* func, int bytes);

}  // namespace rg
