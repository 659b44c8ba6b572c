// rg_api.cu - the C ABI of librg: argument validation, the T/N/K shape
// dispatcher, per-device state (status word, SM count), workspaces and the
// tensor-map encoder.  Every compute step runs in the kernels of the other
// translation units; nothing here touches the data.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "rg_internal.cuh"
#include "rg_launch.h"

namespace rg {

std::atomic<unsigned long long> g_launch_count{0};

// The per-device status word: a kernel that gives up a bounded wait records
// RG_ERR_TIMEOUT here; rg_check reads and clears it.
__device__ int g_status_word;

// Scratch of rg_out_prod_noalloc: the tensor-core path's 16-bit copy of dY
// lives in this fixed array instead of in memory allocated per call.  It is
// part of the library's device image, so every GPU that loads the library
// holds it (RG_NOALLOC_SCRATCH_BYTES) until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RG_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 2147483647;

std::mutex g_mu;
bool g_dev_ready[kMaxDevices];
DevInfo g_dev[kMaxDevices];

struct Env {
  int variant = RG_VARIANT_AUTO;
  unsigned long long wait_limit_ns = 2000ull * 1000 * 1000;
  int inject_stall = 0;
};

const Env& env() {
  static const Env e = [] {
    Env r;
    if (const char* v = std::getenv("RG_VARIANT")) {
      if (!std::strcmp(v, "tc")) r.variant = RG_VARIANT_TC;
      else if (!std::strcmp(v, "tc1")) r.variant = RG_VARIANT_TC_SINGLE;
      else if (!std::strcmp(v, "tc2")) r.variant = RG_VARIANT_TC_PAIR;
      else if (!std::strcmp(v, "smallt")) r.variant = RG_VARIANT_SMALLT;
      else if (!std::strcmp(v, "simt32")) r.variant = RG_VARIANT_SIMT32;
    }
    if (const char* v = std::getenv("RG_WAIT_TIMEOUT_MS")) {
      const long long ms = std::atoll(v);
      if (ms > 0) r.wait_limit_ns = static_cast<unsigned long long>(ms) * 1000000ull;
    }
    if (const char* v = std::getenv("RG_DEBUG_INJECT_STALL")) r.inject_stall = std::atoi(v) != 0;
    return r;
  }();
  return e;
}

// Facts about the current device, queried once per device.
int current_dev(DevInfo** out) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return RG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev_ready[d]) {
    DevInfo info{};
    info.device = d;
    if (cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
      return RG_ERR_CUDA;
    if (cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               d) != cudaSuccess)
      return RG_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return RG_ERR_CUDA;
    info.status = static_cast<int*>(p);
    info.wait_limit_ns = env().wait_limit_ns;
    g_dev[d] = info;
    g_dev_ready[d] = true;
  }
  *out = &g_dev[d];
  return RG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t row_bytes_i(int wtype, int64_t K) {
  if (!valid_wtype(wtype) || K < 0) return 0;
  const int bv = block_values(wtype);
  if (K % bv) return 0;
  return K / bv * block_bytes(wtype);
}

bool contiguous_dy(const Layout& lay, int64_t N) { return lay.dy_n == 1 && lay.dy_t == N; }

// Shared validation of the OUT_PROD arguments.  Returns RG_OK and sets
// *empty when there is nothing to launch.  Strided dY needs 4-byte
// alignment, row-contiguous dY 16-byte (vector loads); dX rows must be
// 16-byte aligned (dx_t a multiple of 4, at least K).
int validate(int wtype, const void* W, int64_t N, int64_t K, const float* dY, int64_t T,
             const float* dX, const Layout& lay, bool* empty) {
  *empty = false;
  if (!valid_wtype(wtype)) return RG_ERR_TYPE;
  if (N < 0 || K < 0 || T < 0 || N > kMaxDim || K > kMaxDim || T > kMaxDim) return RG_ERR_ARG;
  const int64_t kmul = is_quant(wtype) ? 256 : 8;
  if (K % kmul) return RG_ERR_SHAPE;
  if (T == 0 || K == 0) {
    *empty = true;
    return RG_OK;
  }
  if (lay.dx_t < K) return RG_ERR_ARG;
  if (lay.dx_t % 4) return RG_ERR_ALIGN;
  if (!dX) return RG_ERR_ARG;
  if (!aligned16(dX)) return RG_ERR_ALIGN;
  if (N > 0) {
    if (lay.dy_t < 1 || lay.dy_n < 1) return RG_ERR_ARG;
    if (!W || !dY) return RG_ERR_ARG;
    if (!aligned16(W)) return RG_ERR_ALIGN;
    if (contiguous_dy(lay, N) ? !aligned16(dY) : (reinterpret_cast<uintptr_t>(dY) & 3u) != 0)
      return RG_ERR_ALIGN;
  }
  return RG_OK;
}

// Q6_K and Q3_K rows (210 and 110 bytes per 256 values) are 16-byte aligned,
// as the tensor-core and small-T kernels' copies need, only when K is a
// multiple of 2048; Q2_K rows (84 bytes per 256) when K is a multiple of 1024;
// MXFP4 rows (17 bytes per 32) when K is a multiple of 512.
bool aligned_rows(int wtype, int64_t K) {
  if (wtype == RG_Q6_K || wtype == RG_Q3_K) return K % 2048 == 0;
  if (wtype == RG_Q2_K) return K % 1024 == 0;
  if (wtype == RG_MXFP4) return K % 512 == 0;
  return true;
}

int select_variant(int wtype, int64_t N, int64_t K, int64_t T) {
  if (!aligned_rows(wtype, K)) return RG_VARIANT_SIMT32;
  // a few rows of dY, or a problem too small to fill a tensor-core pipeline:
  // the weight-streaming kernel (for Q4_K and Q8_0, whose warp-level MMA
  // consumer costs little more at four rows than at one, up to four rows at
  // any size); else the tensor cores (which split the contraction over idle
  // SMs when the output is small)
  const double flops = 2.0 * static_cast<double>(T) * static_cast<double>(N) * static_cast<double>(K);
  if (T <= 2 || ((wtype == RG_Q4_K || wtype == RG_Q8_0) && T <= 4) || (T <= 32 && flops <= 268435456.0))
    return RG_VARIANT_SMALLT;
  return RG_VARIANT_TC;
}

size_t tc_workspace(int64_t N, int64_t T) {
  const size_t b = static_cast<size_t>(T) * static_cast<size_t>(tc_dy16_ld(N)) * 2;
  return (b + 255) / 256 * 256;
}

bool is_tc(int variant) {
  return variant == RG_VARIANT_TC || variant == RG_VARIANT_TC_SINGLE ||
         variant == RG_VARIANT_TC_PAIR;
}

int cg_force_of(int variant) {
  return variant == RG_VARIANT_TC_SINGLE ? 1 : variant == RG_VARIANT_TC_PAIR ? 2 : 0;
}

// Tensor-core workspace: the 16-bit dY copy; for F32 W its bf16 copy
// [N, K]; then (split contraction) the partial-sum slabs; each 256-byte
// aligned.
size_t tc_w16_bytes(int wtype, int64_t N, int64_t K) {
  if (wtype != RG_F32) return 0;
  return (static_cast<size_t>(N) * static_cast<size_t>(K) * 2 + 255) / 256 * 256;
}
size_t tc_partial_offset(int wtype, int64_t N, int64_t K, int64_t T) {
  return tc_workspace(N, T) + tc_w16_bytes(wtype, N, K);
}
size_t tc_workspace_total(int variant, int wtype, int64_t N, int64_t K, int64_t T,
                          const DevInfo& dev) {
  return tc_partial_offset(wtype, N, K, T) + tc_partial_bytes(N, K, T, dev, cg_force_of(variant));
}

// Workspace bytes of a resolved (non-auto) variant; N, K, T > 0.
size_t workspace_for(int variant, int wtype, int64_t N, int64_t K, int64_t T, const DevInfo& dev) {
  if (is_tc(variant)) return tc_workspace_total(variant, wtype, N, K, T, dev);
  if (variant == RG_VARIANT_SMALLT)
    return (plan_smallt(wtype, N, K, T, dev).workspace + 255) / 256 * 256;
  return 0;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? RG_OK : RG_ERR_CUDA; }

// rg_profile_next_gemm: events for the next tensor-core launch of this thread
thread_local cudaEvent_t t_prof_before = nullptr;
thread_local cudaEvent_t t_prof_after = nullptr;

// One stream-ordered memory pool per device for rg_out_prod's own workspace:
// allocations are cached by the pool (release threshold: never), so a steady
// state of calls does not reach the driver, and stream capture records them as
// graph memory nodes.
cudaMemPool_t g_pool[kMaxDevices];
bool g_pool_ready[kMaxDevices];

int pool_for(int d, cudaMemPool_t* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_pool_ready[d]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = d;
    if (cudaMemPoolCreate(&g_pool[d], &props) != cudaSuccess) return RG_ERR_CUDA;
    uint64_t keep = ~0ull;
    if (cudaMemPoolSetAttribute(g_pool[d], cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
      return RG_ERR_CUDA;
    g_pool_ready[d] = true;
  }
  *out = g_pool[d];
  return RG_OK;
}

// Device address of g_noalloc_scratch on device d (which must be current),
// looked up once per device.  Host code must not use the symbol itself: on
// the host it names a stand-in, not device memory.
void* g_noalloc_ptr[kMaxDevices];
bool g_noalloc_ready[kMaxDevices];

int noalloc_scratch(int d, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ready[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return RG_ERR_CUDA;
    g_noalloc_ptr[d] = p;
    g_noalloc_ready[d] = true;
  }
  *out = g_noalloc_ptr[d];
  return RG_OK;
}

int run(int variant, int wtype, const void* W, int64_t N, int64_t K, const float* dY, int64_t T,
        float* dX, float beta, void* ws, size_t ws_bytes, bool own_ws, cudaStream_t stream,
        const Layout& lay) {
  bool empty = false;
  int st = validate(wtype, W, N, K, dY, T, dX, lay, &empty);
  if (st != RG_OK || empty) return st;
  if (variant < RG_VARIANT_AUTO || variant > RG_VARIANT_TC_PAIR) return RG_ERR_TYPE;
  DevInfo* dev = nullptr;
  if ((st = current_dev(&dev)) != RG_OK) return st;
  if (N == 0) return from_cuda(launch_scale(dX, T, K, lay.dx_t, beta, *dev, stream));
  if (variant == RG_VARIANT_AUTO) variant = select_variant(wtype, N, K, T);
  if (variant != RG_VARIANT_SIMT32 && !aligned_rows(wtype, K)) return RG_ERR_SHAPE;

  if (variant == RG_VARIANT_SIMT32)
    return from_cuda(launch_simt32(wtype, W, N, K, dY, T, dX, beta, lay, *dev, stream));
  // the small-T and tensor-core paths take a workspace: partial sums, or the
  // 16-bit copy of dY
  const size_t need = workspace_for(variant, wtype, N, K, T, *dev);
  void* buf = ws;
  cudaMemPool_t pool{};
  if (own_ws) {
    if ((st = pool_for(dev->device, &pool)) != RG_OK) return st;
    if (cudaMallocFromPoolAsync(&buf, need, pool, stream) != cudaSuccess) return RG_ERR_CUDA;
  } else {
    if (!ws || ws_bytes < need) return RG_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return RG_ERR_ALIGN;
  }
  cudaError_t e = cudaSuccess;
  if (variant == RG_VARIANT_SMALLT) {
    e = launch_smallt(wtype, W, N, K, dY, T, dX, beta, lay, static_cast<float*>(buf),
                      plan_smallt(wtype, N, K, T, *dev), *dev, stream, env().inject_stall);
    if (own_ws) {
      const cudaError_t f = cudaFreeAsync(buf, stream);
      if (e == cudaSuccess) e = f;
    }
    return from_cuda(e);
  }
  // F32 W: both operands in bf16 (the F32 range); W's copy is [N, K]
  const bool bf16 = wtype == RG_BF16 || wtype == RG_F32;
  const int64_t ld = tc_dy16_ld(N);
  uint16_t* dy16 = static_cast<uint16_t*>(buf);
  // a contraction split in two with beta 0: the conversion zeroes dX and the
  // two halves add themselves into it (no partial sums, no reduction kernel)
  const bool halves = tc_adds_halves(N, K, T, beta, lay.dy_n == 1 && lay.dy_t == N, *dev,
                                     cg_force_of(variant));
  e = launch_convert_dy(dY, T, N, lay.dy_t, lay.dy_n, ld, bf16, dy16, *dev, stream, 1.0f,
                        halves ? dX : nullptr, K, lay.dx_t);
  const void* Wtc = W;
  int wtc = wtype;
  if (wtype == RG_F32) {
    uint16_t* w16 = reinterpret_cast<uint16_t*>(static_cast<char*>(buf) + tc_workspace(N, T));
    if (e == cudaSuccess)
      e = launch_convert_dy(static_cast<const float*>(W), N, K, K, 1, K, true, w16, *dev, stream);
    Wtc = w16;
    wtc = RG_BF16;
  }
  cudaEvent_t ev0 = t_prof_before, ev1 = t_prof_after;
  t_prof_before = t_prof_after = nullptr;
  if (e == cudaSuccess && ev0) e = cudaEventRecord(ev0, stream);
  if (e == cudaSuccess)
    e = launch_tc(wtc, Wtc, N, K, dy16, ld, T, dX, lay.dx_t, beta,
                  reinterpret_cast<float*>(static_cast<char*>(buf) +
                                           tc_partial_offset(wtype, N, K, T)),
                  *dev, stream, cg_force_of(variant), nullptr, 0, halves);
  if (e == cudaSuccess && ev1) e = cudaEventRecord(ev1, stream);
  if (own_ws) {
    const cudaError_t f = cudaFreeAsync(buf, stream);
    if (e == cudaSuccess) e = f;
  }
  return from_cuda(e);
}

}  // namespace

namespace {

// Recently encoded tensor maps: encoding is a driver call of a few
// microseconds, and a training step calls with the same tensors every time.
struct MapKey {
  const void* base;
  uint64_t dim0, dim1, stride1, dim2, stride2;
  uint32_t box0, box1;
  int dtype, swizzle, device;
  bool operator==(const MapKey& o) const {
    return base == o.base && dim0 == o.dim0 && dim1 == o.dim1 && stride1 == o.stride1 &&
           dim2 == o.dim2 && stride2 == o.stride2 && box0 == o.box0 && box1 == o.box1 &&
           dtype == o.dtype && swizzle == o.swizzle && device == o.device;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  uint64_t stamp;
  bool used;
};
constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
uint64_t g_map_clock = 0;

// (kernel, device) pairs whose dynamic shared memory limit is already set
struct AttrEntry {
  const void* func;
  int device, bytes;
};
constexpr int kAttrCache = 256;
std::mutex g_attr_mu;
AttrEntry g_attrs[kAttrCache];
int g_n_attrs = 0;

}  // namespace

cudaError_t ensure_smem_attr(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  for (int i = 0; i < g_n_attrs; ++i)
    if (g_attrs[i].func == func && g_attrs[i].device == dev && g_attrs[i].bytes >= bytes)
      return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_n_attrs < kAttrCache) g_attrs[g_n_attrs++] = AttrEntry{func, dev, bytes};
  return e;
}

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                      uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                      uint32_t box1, CUtensorMapSwizzle swizzle, uint64_t dim2,
                      uint64_t stride2_bytes) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return CUDA_ERROR_INVALID_CONTEXT;
  const MapKey key{base, dim0, dim1, stride1_bytes, dim2, stride2_bytes, box0, box1,
                   static_cast<int>(dtype), static_cast<int>(swizzle), device};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (MapEntry& m : g_maps)
      if (m.used && m.key == key) {
        m.stamp = ++g_map_clock;
        *map = m.map;
        return CUDA_SUCCESS;
      }
  }
  const CUresult r = encode_tiled_uncached(map, dtype, base, dim0, dim1, stride1_bytes, box0, box1,
                                           swizzle, dim2, stride2_bytes);
  if (r != CUDA_SUCCESS) return r;
  std::lock_guard<std::mutex> lk(g_map_mu);
  MapEntry* slot = &g_maps[0];
  for (MapEntry& m : g_maps) {
    if (!m.used) { slot = &m; break; }
    if (m.stamp < slot->stamp) slot = &m;
  }
  *slot = MapEntry{key, *map, ++g_map_clock, true};
  return CUDA_SUCCESS;
}

CUresult encode_tiled_uncached(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                               uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0,
                               uint32_t box1, CUtensorMapSwizzle swizzle, uint64_t dim2,
                               uint64_t stride2_bytes) {
  using Fn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                          const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                          CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                          CUtensorMapFloatOOBfill);
  static Fn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<Fn>(p);
  }();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, dim2 > 1 ? 3 : 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace rg

using namespace rg;

extern "C" {

int rg_out_prod(int wtype, const void* W, int64_t N, int64_t K, const float* dY, int64_t T,
                float* dX, float beta, void* stream) {
  return run(env().variant, wtype, W, N, K, dY, T, dX, beta, nullptr, 0, true,
             static_cast<cudaStream_t>(stream), Layout{N, 1, K});
}

int rg_out_prod_variant(int variant, int wtype, const void* W, int64_t N, int64_t K,
                        const float* dY, int64_t T, float* dX, float beta, void* stream) {
  return run(variant, wtype, W, N, K, dY, T, dX, beta, nullptr, 0, true,
             static_cast<cudaStream_t>(stream), Layout{N, 1, K});
}

int rg_out_prod_batched(int variant, int wtype, const void* W, int64_t N, int64_t K, int64_t w_n2,
                        int64_t w_n3, int64_t w_s2, int64_t w_s3, const float* dY, int64_t T,
                        int64_t dy_t, int64_t dy_n, int64_t dy_s2, int64_t dy_s3, float* dX,
                        int64_t dx_t, int64_t dx_s2, int64_t dx_s3, int64_t n2, int64_t n3,
                        float beta, void* stream) {
  if (n2 < 0 || n3 < 0 || w_n2 < 1 || w_n3 < 1 || w_s2 < 0 || w_s3 < 0 || dy_s2 < 0 ||
      dy_s3 < 0 || dx_s2 < 0 || dx_s3 < 0)
    return RG_ERR_ARG;
  if (n2 == 0 || n3 == 0) return RG_OK;
  if (n2 % w_n2 || n3 % w_n3) return RG_ERR_SHAPE;
  if (w_s2 % 16 || w_s3 % 16 || dx_s2 % 4 || dx_s3 % 4) return RG_ERR_ALIGN;
  if (n2 > kMaxDim / n3) return RG_ERR_ARG;
  const Layout lay{dy_t, dy_n, dx_t};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // batch (i2, i3) reads weight (i2 / r2, i3 / r3): each weight serves r2 x r3 batches
  const int64_t r2 = n2 / w_n2, r3 = n3 / w_n3, total = n2 * n3;
  auto w_of = [&](int64_t i) {
    return static_cast<const uint8_t*>(W) + (i % n2) / r2 * w_s2 + (i / n2) / r3 * w_s3;
  };
  auto dy_off = [&](int64_t i) { return (i % n2) * dy_s2 + (i / n2) * dy_s3; };
  auto dx_off = [&](int64_t i) { return (i % n2) * dx_s2 + (i / n2) * dx_s3; };
  // every batch's pointers before the first launch
  for (int64_t i = 0; i < total; ++i) {
    bool empty = false;
    const int st = validate(wtype, w_of(i), N, K, dY + dy_off(i), T, dX + dx_off(i), lay, &empty);
    if (st != RG_OK) return st;
  }
  // consecutive batches (i2 fastest) that read the same weight and whose dY
  // and dX rows continue one another's (batch i + c starts c * T rows on)
  // are one call with that many times T rows
  for (int64_t i = 0; i < total;) {
    int64_t c = 1;
    while (i + c < total && w_of(i + c) == w_of(i) && dy_off(i + c) == dy_off(i) + c * T * dy_t &&
           dx_off(i + c) == dx_off(i) + c * T * dx_t && T * (c + 1) <= kMaxDim)
      ++c;
    const int st = run(variant, wtype, w_of(i), N, K, dY + dy_off(i), T * c, dX + dx_off(i), beta,
                       nullptr, 0, true, s, lay);
    if (st != RG_OK) return st;
    i += c;
  }
  return RG_OK;
}

int rg_out_prod_ex(int variant, int wtype, const void* W, int64_t N, int64_t K,
                   int64_t w_batch_bytes, const float* dY, int64_t T, int64_t dy_t, int64_t dy_n,
                   int64_t dy_batch, float* dX, int64_t dx_t, int64_t dx_batch, int64_t batch,
                   float beta, void* stream) {
  if (batch < 0 || w_batch_bytes < 0) return RG_ERR_ARG;
  if (batch == 0) return RG_OK;
  // one batch dimension: a weight per batch, or one shared by all of them
  return rg_out_prod_batched(variant, wtype, W, N, K, w_batch_bytes ? batch : 1, 1, w_batch_bytes, 0,
                             dY, T, dy_t, dy_n, dy_batch, 0, dX, dx_t, dx_batch, 0, batch, 1, beta,
                             stream);
}

size_t rg_workspace_bytes(int variant, int wtype, int64_t N, int64_t K, int64_t T) {
  if (variant == RG_VARIANT_AUTO) variant = select_variant(wtype, N, K, T);
  if (N <= 0 || T <= 0 || K <= 0) return 0;
  if (!is_tc(variant) && variant != RG_VARIANT_SMALLT) return 0;
  DevInfo* dev = nullptr;
  if (current_dev(&dev) != RG_OK) return is_tc(variant) ? tc_workspace(N, T) : 0;
  return workspace_for(variant, wtype, N, K, T, *dev);
}

int rg_out_prod_ws(int variant, int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                   int64_t T, float* dX, float beta, void* workspace, size_t workspace_bytes,
                   void* stream) {
  return run(variant, wtype, W, N, K, dY, T, dX, beta, workspace, workspace_bytes, false,
             static_cast<cudaStream_t>(stream), Layout{N, 1, K});
}

int rg_out_prod_noalloc(int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                        int64_t T, float* dX, float beta, void* stream) {
  const NoStreamK no_stream_k;  // its partial slabs would not fit the scratch
  bool empty = false;
  int st = validate(wtype, W, N, K, dY, T, dX, Layout{N, 1, K}, &empty);
  if (st != RG_OK || empty) return st;
  int variant = env().variant;
  if (variant == RG_VARIANT_AUTO) variant = select_variant(wtype, N, K, T);
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (N > 0) {
    DevInfo* dev = nullptr;
    if ((st = current_dev(&dev)) != RG_OK) return st;
    const size_t need = workspace_for(variant, wtype, N, K, T, *dev);
    if (need > 0) {
      if (need > static_cast<size_t>(RG_NOALLOC_SCRATCH_BYTES)) return RG_ERR_ARG;
      if ((st = noalloc_scratch(dev->device, &ws)) != RG_OK) return st;
      ws_bytes = static_cast<size_t>(RG_NOALLOC_SCRATCH_BYTES);
    }
  }
  return run(variant, wtype, W, N, K, dY, T, dX, beta, ws, ws_bytes, false,
             static_cast<cudaStream_t>(stream), Layout{N, 1, K});
}

int rg_select_variant(int wtype, int64_t N, int64_t K, int64_t T) {
  return select_variant(wtype, N, K, T);
}

namespace {

// Workspace of the forward: X's 16-bit copy [T, round8(K)], F32 W's bf16
// copy [N, K] (the tensor cores take no F32), a split contraction's partial
// sums [n_splits][T][N]; each 256-byte aligned.  Plans without stream-K.
// Rows that TMA cannot read (aligned_rows false) take the transient route:
// w16 is then the dense 16-bit deq(W)^T [K, N] the OUT_PROD kernel reads.
struct MmWs {
  size_t x16, w16, parts;
  size_t total() const { return x16 + w16 + parts; }
};
MmWs mm_workspace(int wtype, int64_t N, int64_t K, int64_t T, const DevInfo& dev) {
  const NoStreamK no_stream_k;
  if (!aligned_rows(wtype, K))
    return MmWs{tc_workspace(K, T), (static_cast<size_t>(K) * static_cast<size_t>(N) * 2 + 255) / 256 * 256,
                tc_partial_bytes(K, N, T, dev, 0)};
  return MmWs{tc_workspace(K, T), tc_w16_bytes(wtype, N, K), tc_partial_bytes(K, N, T, dev, 0)};
}

}  // namespace

namespace {

// The forward's automatic choice: one or two rows of X stream W once
// (small-T); from three rows the tensor-core kernel, whose time barely
// grows with T at these sizes, is faster.
bool mm_smallt(int wtype, int64_t K, int64_t T) { return T <= 2 && aligned_rows(wtype, K); }

}  // namespace

size_t rg_mul_mat_workspace_bytes(int wtype, int64_t N, int64_t K, int64_t T) {
  if (!valid_wtype(wtype) || N <= 0 || K <= 0 || T <= 0) return 0;
  if (mm_smallt(wtype, K, T)) return 0;
  DevInfo* dev = nullptr;
  if (current_dev(&dev) != RG_OK) return 0;
  return mm_workspace(wtype, N, K, T, *dev).total();
}

int rg_mul_mat(int wtype, const void* W, int64_t N, int64_t K, const float* X, int64_t T, float* Y,
               float beta, void* stream) {
  return rg_mul_mat_variant(RG_VARIANT_AUTO, wtype, W, N, K, X, T, Y, beta, stream);
}

int rg_mul_mat_variant(int variant, int wtype, const void* W, int64_t N, int64_t K, const float* X,
                       int64_t T, float* Y, float beta, void* stream) {
  if (!valid_wtype(wtype)) return RG_ERR_TYPE;
  if (variant != RG_VARIANT_AUTO && variant != RG_VARIANT_TC && variant != RG_VARIANT_SMALLT)
    return RG_ERR_TYPE;
  if (N < 0 || K < 0 || T < 0 || N > kMaxDim || K > kMaxDim || T > kMaxDim) return RG_ERR_ARG;
  if (K % (is_quant(wtype) ? 256 : 8) || N % 8) return RG_ERR_SHAPE;
  if (T == 0 || N == 0) return RG_OK;
  if (!Y) return RG_ERR_ARG;
  if (!aligned16(Y)) return RG_ERR_ALIGN;
  if (K > 0) {
    if (!W || !X) return RG_ERR_ARG;
    if (!aligned16(W) || !aligned16(X)) return RG_ERR_ALIGN;
    // the named small-T route: 16-byte aligned rows, a grid row per four rows of X
    if (variant == RG_VARIANT_SMALLT && (!aligned_rows(wtype, K) || (T + 3) / 4 > 65535))
      return RG_ERR_SHAPE;
  }
  DevInfo* dev = nullptr;
  int st = current_dev(&dev);
  if (st != RG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(launch_scale(Y, T, N, N, beta, *dev, s));
  if (variant == RG_VARIANT_AUTO) variant = mm_smallt(wtype, K, T) ? RG_VARIANT_SMALLT : RG_VARIANT_TC;
  if (variant == RG_VARIANT_SMALLT) {
    // W streamed once per four rows of X, F32 products: one launch
    cudaEvent_t ev0 = t_prof_before, ev1 = t_prof_after;
    t_prof_before = t_prof_after = nullptr;
    cudaError_t e = ev0 ? cudaEventRecord(ev0, s) : cudaSuccess;
    if (e == cudaSuccess) e = launch_smallt_fwd(wtype, W, N, K, X, T, Y, beta, *dev, s);
    if (e == cudaSuccess && ev1) e = cudaEventRecord(ev1, s);
    return from_cuda(e);
  }
  // Y = X . deq(W)^T: the tensor-core kernel decodes W's blocks as the
  // K-major operand of a contraction over each row's K values; X is rounded
  // to the 16-bit kind once (F32 W: both W and X to bf16)
  const NoStreamK no_stream_k;
  const bool bf16 = wtype == RG_BF16 || wtype == RG_F32;
  const MmWs ws = mm_workspace(wtype, N, K, T, *dev);
  cudaMemPool_t pool{};
  if ((st = pool_for(dev->device, &pool)) != RG_OK) return st;
  void* buf = nullptr;
  if (cudaMallocFromPoolAsync(&buf, ws.total(), pool, s) != cudaSuccess) return RG_ERR_CUDA;
  char* b = static_cast<char*>(buf);
  uint16_t* xh = reinterpret_cast<uint16_t*>(b);
  uint16_t* w16 = reinterpret_cast<uint16_t*>(b + ws.x16);
  float* part = reinterpret_cast<float*>(b + ws.x16 + ws.w16);
  const int64_t ld = tc_dy16_ld(K);
  const bool fused = aligned_rows(wtype, K);
  // rows whose 16-byte windows TMA cannot address (Q6_K and Q3_K rows with
  // K % 2048 != 0, Q2_K K % 1024, MXFP4 K % 512): a transient dense 16-bit
  // deq(W)^T, contracted by the OUT_PROD kernel as a weight of K rows
  cudaError_t e = fused ? cudaSuccess : launch_dequant_t16(wtype, W, N, K, bf16, w16, N, *dev, s);
  // a contraction split in two with beta 0: X's conversion zeroes Y and the
  // two halves add themselves into it
  const TcPlan mp = plan_tc(K, N, T, *dev, 0);
  const bool halves = fused && beta == 0.0f && mp.n_splits == 2 && !mp.sk;
  if (e == cudaSuccess)
    e = launch_convert_dy(X, T, K, K, 1, ld, bf16, xh, *dev, s, 1.0f, halves ? Y : nullptr, N, N);
  const void* Wtc = W;
  int wtc = wtype;
  if (wtype == RG_F32 && fused) {
    if (e == cudaSuccess)
      e = launch_convert_dy(static_cast<const float*>(W), N, K, K, 1, K, true, w16, *dev, s);
    Wtc = w16;
    wtc = RG_BF16;
  }
  cudaEvent_t ev0 = t_prof_before, ev1 = t_prof_after;
  t_prof_before = t_prof_after = nullptr;
  if (e == cudaSuccess && ev0) e = cudaEventRecord(ev0, s);
  if (e == cudaSuccess)
    e = fused ? launch_mm(wtc, Wtc, N, K, xh, ld, T, Y, N, beta, part, *dev, s, 0, halves)
              : launch_tc(bf16 ? RG_BF16 : RG_F16, w16, K, N, xh, ld, T, Y, N, beta, part, *dev, s, 0);
  if (e == cudaSuccess && ev1) e = cudaEventRecord(ev1, s);
  const cudaError_t f = cudaFreeAsync(buf, s);
  if (e == cudaSuccess) e = f;
  return from_cuda(e);
}

int rg_out_prod_lora(int variant, int wtype, const void* W, int64_t N, int64_t K, const float* dY,
                     int64_t T, float* dX, float beta, const float* lora_a, const float* lora_b,
                     int64_t rank, float scale, void* stream) {
  const NoStreamK no_stream_k;  // the adapter's kernels are built without it
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout lay{N, 1, K};
  bool empty = false;
  int st = validate(wtype, W, N, K, dY, T, dX, lay, &empty);
  if (st != RG_OK) return st;
  if (rank < 0) return RG_ERR_ARG;
  if (rank > 1024) return RG_ERR_SHAPE;
  if (variant < RG_VARIANT_AUTO || variant > RG_VARIANT_TC_PAIR) return RG_ERR_TYPE;
  // no adapter term: the base product alone (N == 0 makes dY . B zero)
  if (empty || rank == 0 || N == 0)
    return run(variant, wtype, W, N, K, dY, T, dX, beta, nullptr, 0, true, s, lay);
  if (!lora_a || !lora_b) return RG_ERR_ARG;
  if (!aligned16(lora_a) || !aligned16(lora_b)) return RG_ERR_ALIGN;
  if (variant == RG_VARIANT_AUTO) variant = select_variant(wtype, N, K, T);
  if (variant != RG_VARIANT_SIMT32 && !aligned_rows(wtype, K)) return RG_ERR_SHAPE;
  DevInfo* dev = nullptr;
  if ((st = current_dev(&dev)) != RG_OK) return st;
  cudaMemPool_t pool{};
  if ((st = pool_for(dev->device, &pool)) != RG_OK) return st;

  if (!is_tc(variant)) {
    // the base product as the variant computes it, then the F32 adapter term
    if ((st = run(variant, wtype, W, N, K, dY, T, dX, beta, nullptr, 0, true, s, lay)) != RG_OK)
      return st;
    const int parts = adapter_down_parts(N, T, rank, *dev);
    void* buf = nullptr;
    const size_t bytes = static_cast<size_t>(parts) * static_cast<size_t>(T) * static_cast<size_t>(rank) * 4;
    if (cudaMallocFromPoolAsync(&buf, bytes, pool, s) != cudaSuccess) return RG_ERR_CUDA;
    cudaError_t e = launch_adapter_f32(dY, N, T, lora_a, lora_b, rank, K, scale, dX, K,
                                       static_cast<float*>(buf), parts, *dev, s);
    const cudaError_t f = cudaFreeAsync(buf, s);
    return from_cuda(e == cudaSuccess ? f : e);
  }

  // tensor cores: dY's 16-bit copy gets U = dY . B after its own columns,
  // scale * A joins W's rows as extra contraction chunks of the base product
  const bool bf16 = wtype == RG_BF16 || wtype == RG_F32;
  const int cg = cg_force_of(variant);
  const bool fused = rank <= kAdapterFusedRank;
  const int64_t ld = tc_adapter_cols(N, rank);
  const int64_t r8 = (rank + 7) / 8 * 8;
  const int64_t ldb = (N + 7) / 8 * 8;
  auto up256 = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t dy_bytes = up256(static_cast<size_t>(T) * static_cast<size_t>(ld) * 2);
  const size_t w_bytes = tc_w16_bytes(wtype, N, K);
  const size_t a_bytes = up256(static_cast<size_t>(rank) * static_cast<size_t>(K) * 2);
  // B as 16 bits: B^T [rank, ldb] for the fused pass, else B [N, r8]
  const size_t b_bytes = up256(fused ? static_cast<size_t>(rank) * static_cast<size_t>(ldb) * 2
                                     : static_cast<size_t>(N) * static_cast<size_t>(r8) * 2);
  const size_t u_bytes = fused ? 0 : up256(static_cast<size_t>(T) * static_cast<size_t>(r8) * 4);
  const size_t p_main = tc_partial_bytes(ld, K, T, *dev, cg);
  const size_t p_u = fused ? 0 : tc_partial_bytes(N, r8, T, *dev, 0);
  const size_t p_bytes = up256(std::max(p_main, p_u));
  void* buf = nullptr;
  if (cudaMallocFromPoolAsync(&buf, dy_bytes + w_bytes + a_bytes + b_bytes + u_bytes + p_bytes,
                              pool, s) != cudaSuccess)
    return RG_ERR_CUDA;
  char* b = static_cast<char*>(buf);
  uint16_t* dy16 = reinterpret_cast<uint16_t*>(b);
  uint16_t* w16 = reinterpret_cast<uint16_t*>(b + dy_bytes);
  uint16_t* a16 = reinterpret_cast<uint16_t*>(b + dy_bytes + w_bytes);
  uint16_t* b16 = reinterpret_cast<uint16_t*>(b + dy_bytes + w_bytes + a_bytes);
  float* u32 = reinterpret_cast<float*>(b + dy_bytes + w_bytes + a_bytes + b_bytes);
  float* part = reinterpret_cast<float*>(b + dy_bytes + w_bytes + a_bytes + b_bytes + u_bytes);
  cudaError_t e = launch_convert_dy(lora_a, rank, K, K, 1, K, bf16, a16, *dev, s, scale);
  if (fused) {
    // one pass over dY: its 16-bit copy and U behind it
    if (e == cudaSuccess) e = launch_convert_dy(lora_b, rank, N, 1, rank, ldb, bf16, b16, *dev, s);
    if (e == cudaSuccess) e = launch_convert_dy_adapter(dY, T, N, b16, ldb, rank, ld, bf16, dy16, s);
  } else {
    // U [T, r8] = dY . B as an OUT_PROD over B's 16-bit copy (ranks past
    // `rank` are zero), then packed behind dY's columns
    if (e == cudaSuccess) e = launch_convert_dy(dY, T, N, N, 1, ld, bf16, dy16, *dev, s);
    if (e == cudaSuccess) e = launch_convert_dy(lora_b, N, rank, rank, 1, r8, bf16, b16, *dev, s);
    if (e == cudaSuccess)
      e = launch_tc(bf16 ? RG_BF16 : RG_F16, b16, N, r8, dy16, ld, T, u32, r8, 0.0f, part, *dev,
                    s, 0);
    if (e == cudaSuccess) e = launch_adapter_pack(u32, r8, T, rank, N, ld, bf16, dy16, *dev, s);
  }
  const void* Wtc = W;
  int wtc = wtype;
  if (wtype == RG_F32) {
    if (e == cudaSuccess)
      e = launch_convert_dy(static_cast<const float*>(W), N, K, K, 1, K, true, w16, *dev, s);
    Wtc = w16;
    wtc = RG_BF16;
  }
  cudaEvent_t ev0 = t_prof_before, ev1 = t_prof_after;
  t_prof_before = t_prof_after = nullptr;
  if (e == cudaSuccess && ev0) e = cudaEventRecord(ev0, s);
  if (e == cudaSuccess)
    e = launch_tc(wtc, Wtc, N, K, dy16, ld, T, dX, K, beta, part, *dev, s, cg, a16, rank);
  if (e == cudaSuccess && ev1) e = cudaEventRecord(ev1, s);
  const cudaError_t f = cudaFreeAsync(buf, s);
  return from_cuda(e == cudaSuccess ? f : e);
}

int rg_plan(int variant, int wtype, int64_t N, int64_t K, int64_t T, rg_plan_info* out) {
  if (!out) return RG_ERR_ARG;
  if (!valid_wtype(wtype)) return RG_ERR_TYPE;
  if (variant < RG_VARIANT_AUTO || variant > RG_VARIANT_TC_PAIR) return RG_ERR_TYPE;
  if (N < 0 || K < 0 || T < 0 || N > kMaxDim || K > kMaxDim || T > kMaxDim) return RG_ERR_ARG;
  if (K % (is_quant(wtype) ? 256 : 8)) return RG_ERR_SHAPE;
  DevInfo* dev = nullptr;
  const int st = current_dev(&dev);
  if (st != RG_OK) return st;
  rg_plan_info r{};
  r.variant = variant == RG_VARIANT_AUTO ? select_variant(wtype, N, K, T) : variant;
  if (r.variant != RG_VARIANT_SIMT32 && !aligned_rows(wtype, K) && T > 0 && K > 0 && N > 0)
    return RG_ERR_SHAPE;
  r.n_splits = 1;
  if (T == 0 || K == 0 || N == 0) {
    r.launches = (T == 0 || K == 0) ? 0 : 1;
    *out = r;
    return RG_OK;
  }
  int64_t tile_t = 0;
  if (is_tc(r.variant)) {
    const TcPlan p = plan_tc(N, K, T, *dev, cg_force_of(r.variant));
    r.cta_group = p.cg;
    r.tile_k = 128 * p.cg;
    tile_t = p.bt;
    r.n_splits = p.n_splits;
    r.grid = p.grid;
    r.stream_k = p.sk ? 1 : 0;
    // dY conversion (and F32 W's), GEMM, split reduction or stream-K fixup
    // (a split in two adds its halves into dX, for beta 0: no third kernel)
    r.launches = (p.sk || p.n_splits > 2 ? 3 : 2) + (wtype == RG_F32 ? 1 : 0);
  } else if (r.variant == RG_VARIANT_SMALLT) {
    const SmalltPlan p = plan_smallt(wtype, N, K, T, *dev);
    r.tile_k = 256;
    tile_t = p.tb;
    r.n_splits = p.n_splits;
    r.grid = p.n_ktiles * p.n_splits * p.n_tchunks;
    r.launches = p.n_splits > 1 ? 2 : 1;  // row-split partial sums and their reduction, or dX directly
  } else {
    r.tile_k = 64;
    tile_t = 64;
    r.grid = static_cast<int32_t>(((K + 63) / 64) * ((T + 63) / 64));
    r.launches = 1;
  }
  r.tile_t = static_cast<int32_t>(tile_t);
  r.decode_ops = (T + tile_t - 1) / tile_t * N * K;
  r.workspace_bytes = static_cast<int64_t>(workspace_for(r.variant, wtype, N, K, T, *dev));
  *out = r;
  return RG_OK;
}

uint64_t rg_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

int rg_dequant_async(int wtype, const void* W, int64_t N, int64_t K, float* out, void* stream) {
  if (!valid_wtype(wtype)) return RG_ERR_TYPE;
  if (N < 0 || K < 0 || N > kMaxDim || K > kMaxDim) return RG_ERR_ARG;
  const int64_t kmul = is_quant(wtype) ? 256 : 8;
  if (K % kmul) return RG_ERR_SHAPE;
  if (N == 0 || K == 0) return RG_OK;
  if (!W || !out) return RG_ERR_ARG;
  if (!aligned16(W) || !aligned16(out)) return RG_ERR_ALIGN;
  DevInfo* dev = nullptr;
  int st = current_dev(&dev);
  if (st != RG_OK) return st;
  return from_cuda(launch_dequant(wtype, W, N, K, out, *dev, static_cast<cudaStream_t>(stream)));
}

int rg_dequant(int wtype, const void* W, int64_t N, int64_t K, float* out) {
  return rg_dequant_async(wtype, W, N, K, out, nullptr);
}

size_t rg_row_bytes(int wtype, int64_t K) {
  return static_cast<size_t>(row_bytes_i(wtype, K));
}

const char* rg_strerror(int status) {
  switch (status) {
    case RG_OK: return "ok";
    case RG_ERR_ARG: return "invalid argument (null pointer, negative or too large size, small workspace)";
    case RG_ERR_TYPE: return "unknown weight type or variant";
    case RG_ERR_SHAPE:
      return "K is not a multiple of 256 (quantized types) or 8 (F32/F16/BF16); or rows not "
             "16-byte aligned on a tensor-core or small-T variant (Q6_K, Q3_K: K % 2048 != 0; "
             "Q2_K: K % 1024 != 0; MXFP4: K % 512 != 0); or a batch or N rule of the call";
    case RG_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case RG_ERR_CUDA: return "CUDA call or kernel launch failed";
    case RG_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case RG_ERR_RANGE:
      return "a dY value lay outside the 16-bit tensor-core operand range (fp16: |dY| >= 65520)";
    default: return "unknown status";
  }
}

int rg_check(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return RG_ERR_CUDA;
  DevInfo* dev = nullptr;
  int st = current_dev(&dev);
  if (st != RG_OK) return st;
  int v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return RG_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return RG_ERR_CUDA;
  }
  return v;
}

int rg_debug_wait_probe(int timeout_ms, void* stream) {
  if (timeout_ms <= 0 || timeout_ms > 60000) return RG_ERR_ARG;
  DevInfo* dev = nullptr;
  int st = current_dev(&dev);
  if (st != RG_OK) return st;
  return from_cuda(launch_wait_probe(*dev, static_cast<unsigned long long>(timeout_ms) * 1000000ull,
                                     static_cast<cudaStream_t>(stream)));
}

int rg_version(void) { return (0 << 16) | 1; }

int rg_profile_next_gemm(void* before, void* after) {
  t_prof_before = static_cast<cudaEvent_t>(before);
  t_prof_after = static_cast<cudaEvent_t>(after);
  return RG_OK;
}

}  // extern "C"
