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
// slabs' write + read (plus one dX read for beta) at ~6 TB/s.
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
  }
  return best;
}

cudaError_t launch_tc(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                      int64_t ld_dy16, int64_t T, float* dX, int64_t dx_t, float beta, float* part,
                      const DevInfo& dev, cudaStream_t stream, int cg_force, int inject_stall,
                      const uint16_t* a16, int64_t rank) {
  if (rank > 0)
    return launch_tc_adapter(wtype, W, N, K, dy16, ld_dy16, T, dX, dx_t, beta, part, dev, stream,
                             cg_force, inject_stall, a16, rank);
  return launch_tc_impl<false>(wtype, W, N, K, dy16, ld_dy16, T, dX, dx_t, beta, part, dev,
                               stream, cg_force, inject_stall, nullptr, 0);
}

int64_t tc_adapter_cols(int64_t N, int64_t r) {
  return ((N + tc::BC - 1) / tc::BC + (r + tc::BC - 1) / tc::BC) * tc::BC;
}

int64_t tc_partial_splits(int64_t N, int64_t K, int64_t T, const DevInfo& dev, int cg_force) {
  const TcPlan p = plan_tc(N, K, T, dev, cg_force);
  return p.n_splits > 1 ? p.n_splits : 0;
}

}  // namespace rg
