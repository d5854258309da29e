// Classical instantiations on CTA pairs (256-row tiles, tcgen05 cta_group::2).
#include <algorithm>

#include "fgemm_kernel_pair.cuh"

namespace fgemm {

cudaError_t launch_gemm_pair(int bn, const KernelParams& p, int clusters, cudaStream_t stream) {
  switch (bn) {
    case 128: return launch_gemm_pair_t<128>(p, clusters, stream);
    case 256: return launch_gemm_pair_t<256>(p, clusters, stream);
    default: return cudaErrorInvalidValue;
  }
}

int gemm_pair_clusters_fit(int bn) {
  switch (bn) {
    case 128: return gemm_pair_clusters_fit_t<128>();
    case 256: return gemm_pair_clusters_fit_t<256>();
    default: return 0;
  }
}

}  // namespace fgemm
