// rg_tc_ad.cu - the tensor-core OUT_PROD with a low-rank adapter riding along
// as extra contraction chunks (the kernel's AD instances, rg_tc_kernel.cuh).
#include "rg_tc_kernel.cuh"

namespace rg {

cudaError_t launch_tc_adapter(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* dy16,
                              int64_t ld_dy16, int64_t T, float* dX, int64_t dx_t, float beta,
                              float* part, const DevInfo& dev, cudaStream_t stream, int cg_force,
                              const uint16_t* a16, int64_t rank) {
  return launch_tc_impl<true, false>(wtype, W, N, K, dy16, ld_dy16, T, dX, dx_t, beta, part, dev,
                                     stream, cg_force, a16, rank);
}

}  // namespace rg
