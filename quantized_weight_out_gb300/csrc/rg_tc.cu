// rg_tc.cu - the tensor-core OUT_PROD without an adapter: the tile planner,
// launch_tc (its dispatch), and the kernel's instances (rg_tc_kernel.cuh).
#include "rg_tc_kernel.cuh"

namespace rg {

// --- host side ------------------------------------------------------------------

int64_t tc_dy16_ld(int64_t N) { return (N + 7) / 8 * 8; }

// Tile shape and contraction split from a small cost model: a stage (64
// contraction rows of one tile) costs about the same time in either tile
// shape (the decoders bound it), pair tiles cover 4x the outputs on 2 SMs,
// items run in waves over the persistent units, and a split adds the partial
// slabs' write + read (plus one dX read for beta) at ~6 TB/s.  Stream-K
// (whole waves, then the last tiles' stages spread evenly over the units)
// removes the last wave's idle units for a few microseconds of counters,
// partial slabs (kept in L2) and the last pieces' sums.
namespace {
thread_local int t_no_stream_k = 0;
}  // namespace
NoStreamK::NoStreamK() { ++t_no_stream_k; }
NoStreamK::~NoStreamK() { --t_no_stream_k; }

TcPlan plan_tc(int64_t N, int64_t K, int64_t T, const DevInfo& dev, int cg_force) {
  const int64_t chunks = (N + tc::BC - 1) / tc::BC;
  const double stage_us = 0.45, bw_bytes_per_us = 6.0e6;
  TcPlan best{};
  double best_t = -1.0;
  for (int cg = 1; cg <= 2; ++cg) {
    if (cg_force && cg != cg_force) continue;
    const int64_t bt = cg == 2 ? 256 : 128;
    const int64_t nku = (K + 128 * cg - 1) / (128 * cg), ntt = (T + bt - 1) / bt;
    const int64_t tiles = nku * ntt, avail = dev.num_sms / cg;
    for (int64_t s = 1; s <= 16; ++s) {
      const int64_t cps = (chunks + s - 1) / s;
      if (s > 1 && cps < 8) break;  // at least 8 stages per split
      const int64_t waves = (tiles * s + avail - 1) / avail;
      double t = static_cast<double>(waves) * static_cast<double>(cps) * stage_us;
      if (s > 1) t += static_cast<double>(2 * s + 2) * static_cast<double>(T * K) * 4.0 / bw_bytes_per_us;
      if (best_t < 0 || t < best_t * 0.98) {
        best_t = t;
        best = TcPlan{};
        best.cg = cg;
        best.bt = static_cast<int>(bt);
        best.n_kunits = static_cast<int>(nku);
        best.n_ttiles = static_cast<int>(ntt);
        best.n_splits = static_cast<int>(s);
        best.n_chunks = static_cast<int>(cps);
        best.grid = static_cast<int>(std::min(tiles * s, avail) * cg);
      }
    }
    {
      // stream-K: whole waves (at least one: with fewer tiles than units a
      // split's second kernel is cheaper than the shared tiles'), then the
      // remaining R tiles' stages over all units
      const int64_t F = tiles / avail, R = tiles % avail;
      // (the kernel's 32-bit stage arithmetic needs units^2 * chunks < 2^31
      // for any unit count the residency cap may leave)
      if (t_no_stream_k == 0 && F >= 1 && R > 0 && R * chunks >= 4 * avail &&
          avail * avail * chunks < (int64_t{1} << 31)) {
        const int64_t per = F * chunks + (R * chunks + avail - 1) / avail;
        const double slab = static_cast<double>(bt) * static_cast<double>(128 * cg) * 4.0;
        const double t = static_cast<double>(per) * stage_us + 4.0 +
                         2.0 * static_cast<double>(R + avail) * slab / 15.0e6;
        if (best_t < 0 || t < best_t * 0.98) {
          best_t = t;
          best = TcPlan{};
          best.cg = cg;
          best.bt = static_cast<int>(bt);
          best.n_kunits = static_cast<int>(nku);
          best.n_ttiles = static_cast<int>(ntt);
          best.n_splits = 1;
          best.n_chunks = static_cast<int>(chunks);
          best.grid = static_cast<int>(avail * cg);
          best.sk = true;
        }
      }
    }
  }
  return best;
}

cudaError_t launch_tc(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                      int64_t ld_dy16, int64_t T, float* dX, int64_t dx_t, float beta, float* part,
                      const DevInfo& dev, cudaStream_t stream, int cg_force, const uint16_t* a16,
                      int64_t rank, bool zeroed) {
  if (zeroed && rank > 0) return cudaErrorInvalidValue;
  if (rank > 0)
    return launch_tc_adapter(wtype, W, N, K, dy16, ld_dy16, T, dX, dx_t, beta, part, dev, stream,
                             cg_force, a16, rank);
  if (plan_tc(N, K, T, dev, cg_force).sk)
    return launch_tc_stream_k(wtype, W, N, K, dy16, ld_dy16, T, dX, dx_t, beta, part, dev, stream,
                              cg_force);
  return launch_tc_impl<false, false>(wtype, W, N, K, dy16, ld_dy16, T, dX, dx_t, beta, part, dev,
                                      stream, cg_force, nullptr, 0, zeroed);
}

bool tc_adds_halves(int64_t N, int64_t K, int64_t T, float beta, bool dy_rows, const DevInfo& dev,
                    int cg_force) {
  if (beta != 0.0f || !dy_rows) return false;
  const TcPlan p = plan_tc(N, K, T, dev, cg_force);
  return p.n_splits == 2 && !p.sk;
}

int tc_band(int wtype, int64_t n_contr, const TcPlan& p) {
  // k units whose slice of W (128 cg values of every contraction row, or the
  // forward's 128 cg rows of n_contr values) fits comfortably in L2 (48 MB)
  const double w_per_value =
      is_quant(wtype) ? static_cast<double>(block_bytes(wtype)) / block_values(wtype) : 2.0;
  const double slice = static_cast<double>(n_contr) * (tc::BM * p.cg) * w_per_value;
  return static_cast<int>(std::max(1.0, std::min<double>(p.n_kunits, 48.0 * 1024 * 1024 / slice)));
}

// Warp slices of the shared tiles: slice (x, req) is tile x (item n_dp + x
// of the plan's banded order), CTA half r and epilogue warp eq (req = 4r +
// eq): 32 values of k by bt rows of t.  The piece with the tile's first
// chunk wrote dX (beta applied); a later piece's unit u holds the slice at
// ((u * cg + r) * 4 + eq) * bt * 32 of the slabs, row-major [t][lane].  One
// 4-value group per thread (blocks of 256 over a slice), every piece's load
// in flight before the adds, which go in chunk order: the result does not
// depend on timing.
constexpr int kFixupThreads = 256;
__global__ void __launch_bounds__(kFixupThreads) sk_fixup_kernel(
    const float* __restrict__ slabs, int units, int cg, int bt, int n_dp, int R, int nck,
    int n_kunits, int n_ttiles, int band, int T, int K, float* __restrict__ dX, int64_t ldx) {
  __shared__ int64_t s_off[256];
  __shared__ int s_meta[3];
  pdl_wait();  // dX's head pieces and the slabs come from the main kernel before this one
  const int per_slice = bt * 8 / kFixupThreads;  // blocks per slice (4-value groups / threads)
  const int slice = blockIdx.x / per_slice;
  const int x = slice / (cg * 4), req = slice - x * (cg * 4);
  const uint32_t rn = static_cast<uint32_t>(R) * static_cast<uint32_t>(nck);
  const uint32_t a0 = static_cast<uint32_t>(x) * static_cast<uint32_t>(nck);
  if (threadIdx.x == 0) {
    // the tile's coordinates in the banded order (as the main kernel)
    const int tile = n_dp + x;
    const int per_band = band * n_ttiles;
    const int b = tile / per_band, rr = tile - b * per_band;
    const int gk = min(band, n_kunits - b * band);
    const int tt = rr / gk, ku = b * band + (rr - tt * gk);
    s_meta[0] = (ku * cg + req / 4) * 128 + 32 * (req & 3);  // first k
    s_meta[1] = tt * bt;                                       // first t
    s_meta[2] = min(256, tc::sk_unit_of(a0 + static_cast<uint32_t>(nck) - 1u, rn, units) -
                             tc::sk_unit_of(a0, rn, units) + 1);  // pieces
  }
  __syncthreads();
  const int ufirst = tc::sk_unit_of(a0, rn, units);
  const int pieces = s_meta[2];
  for (int q = 1 + static_cast<int>(threadIdx.x); q < pieces; q += blockDim.x)
    s_off[q] = (static_cast<int64_t>(ufirst + q) * cg * 4 + req) * bt * 32;
  __syncthreads();
  const int e = 4 * ((blockIdx.x - slice * per_slice) * kFixupThreads + static_cast<int>(threadIdx.x));
  const int t = s_meta[1] + (e >> 5), k = s_meta[0] + (e & 31);
  if (t >= T || k >= K) return;  // K % 4 == 0: a group is in or out whole
  float4* o = reinterpret_cast<float4*>(dX + static_cast<int64_t>(t) * ldx + k);
  float4 v = *o;
  for (int q0 = 1; q0 < pieces; q0 += 4) {
    float4 y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (q0 + j < pieces) y[j] = __ldcg(reinterpret_cast<const float4*>(slabs + s_off[q0 + j] + e));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (q0 + j < pieces) {
        v.x += y[j].x;
        v.y += y[j].y;
        v.z += y[j].z;
        v.w += y[j].w;
      }
    }
  }
  *o = v;
}

cudaError_t launch_sk_fixup(const float* part, int units, int cg, int bt, const TcPlan& p, int T,
                            int K, float* dX, int64_t ldx, const DevInfo& dev,
                            cudaStream_t stream) {
  (void)dev;
  const int n_items = p.n_kunits * p.n_ttiles;
  int n_dp = (n_items / units) * units;
  // as the main kernel: too few chunks left to share means whole tiles only
  if (static_cast<int64_t>(n_items - n_dp) * p.n_chunks < units) n_dp = n_items;
  const int R = n_items - n_dp;
  if (R == 0) return cudaSuccess;
  const int blocks = R * cg * 4 * (bt * 8 / kFixupThreads);
  return counted(launch_after_prev(sk_fixup_kernel, dim3(blocks), dim3(kFixupThreads), stream, part,
                                   units, cg, bt, n_dp, R, static_cast<int>(p.n_chunks),
                                   static_cast<int>(p.n_kunits), static_cast<int>(p.n_ttiles),
                                   static_cast<int>(p.band), T, K, dX, ldx));
}

int64_t tc_adapter_cols(int64_t N, int64_t r) {
  return ((N + tc::BC - 1) / tc::BC + (r + tc::BC - 1) / tc::BC) * tc::BC;
}

int64_t tc_partial_splits(int64_t N, int64_t K, int64_t T, const DevInfo& dev, int cg_force) {
  const TcPlan p = plan_tc(N, K, T, dev, cg_force);
  return p.n_splits > 1 ? p.n_splits : 0;
}

size_t tc_partial_bytes(int64_t N, int64_t K, int64_t T, const DevInfo& dev, int cg_force) {
  const TcPlan p = plan_tc(N, K, T, dev, cg_force);
  size_t b = 0;
  if (p.n_splits > 1) {
    b = static_cast<size_t>(p.n_splits) * static_cast<size_t>(T) * static_cast<size_t>(K) * 4;
  } else if (p.sk) {
    // one slab per unit of a whole tile (bt x 128 cg floats)
    const int units = dev.num_sms / p.cg;
    b = static_cast<size_t>(units) * static_cast<size_t>(p.bt) * (128 * p.cg) * 4;
  }
  return (b + 255) / 256 * 256;
}

}  // namespace rg
