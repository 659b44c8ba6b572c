// rg_tc_sk.cu - the tensor-core OUT_PROD on stream-K plans: whole waves of
// tiles, then the last tiles' contraction shared evenly over the units (the
// kernel's SK instances, rg_tc_kernel.cuh, and the second pass that adds the
// shared tiles' pieces, rg_tc.cu).  A translation unit of its own, so that
// every other plan runs kernels built without any of it.
#include "rg_tc_kernel.cuh"

namespace rg {

cudaError_t launch_tc_stream_k(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                               int64_t ld_dy16, int64_t T, float* dX, int64_t dx_t, float beta,
                               float* part, const DevInfo& dev, cudaStream_t stream, int cg_force) {
  return launch_tc_impl<false, true>(wtype, W, N, K, dy16, ld_dy16, T, dX, dx_t, beta, part, dev,
                                     stream, cg_force, nullptr, 0);
}

}  // namespace rg
