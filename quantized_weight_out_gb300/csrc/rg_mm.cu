// rg_mm.cu - the forward mul_mat(W, x) through the resident weight: the
// tensor-core kernel's FWD instances (rg_tc_kernel.cuh), which contract over
// the K values of each stored row instead of over the rows.  A translation
// unit of its own, so that the OUT_PROD kernels are built without it.
#include "rg_tc_kernel.cuh"

namespace rg {

cudaError_t launch_mm(int wtype, const void* W, int64_t N, int64_t K, const uint16_t* x16,
                      int64_t ld_x16, int64_t T, float* Y, int64_t ldy, float beta, float* part,
                      const DevInfo& dev, cudaStream_t stream, int cg_force, bool zeroed) {
  return launch_tc_impl<false, false, true>(wtype, W, N, K, x16, ld_x16, T, Y, ldy, beta, part, dev,
                                            stream, cg_force, nullptr, 0, zeroed);
}

}  // namespace rg
