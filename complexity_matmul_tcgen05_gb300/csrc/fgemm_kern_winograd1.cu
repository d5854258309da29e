// One-level Winograd-variant instantiations of the persistent tcgen05 GEMM:
// the Strassen kernel with up to four source blocks per formed operand.
#include "fgemm_kernel.cuh"

namespace fgemm {

cudaError_t launch_gemm_winograd1(int bn, const KernelParams& p, const StrassenTable& tab, int grid,
                                  cudaStream_t stream) {
  switch (bn) {
    case 128: return launch_gemm_t<128, 1, 4>(p, &tab, grid, stream);
    case 256: return launch_gemm_t<256, 1, 4>(p, &tab, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fgemm
