// Two-level Strassen instantiations of the persistent tcgen05 GEMM.
#include "fgemm_kernel.cuh"

namespace fgemm {

cudaError_t launch_gemm_depth2(int bn, const KernelParams& p, const StrassenTable& tab, int grid,
                               cudaStream_t stream) {
  switch (bn) {
    case 128: return launch_gemm_t<128, 2>(p, &tab, grid, stream);
    case 256: return launch_gemm_t<256, 2>(p, &tab, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fgemm
