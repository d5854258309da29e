// Classical (depth 0) instantiations of the persistent tcgen05 GEMM, the
// K == 0 fill kernel and the launch dispatcher.
#include "fgemm_kernel.cuh"

namespace fgemm {

cudaError_t launch_gemm_depth1(int bn, const KernelParams& p, const StrassenTable& tab, int grid,
                               cudaStream_t stream);
cudaError_t launch_gemm_depth2(int bn, const KernelParams& p, const StrassenTable& tab, int grid,
                               cudaStream_t stream);

size_t kernel_smem_bytes(int bn, int depth) {
  (void)depth;
  switch (bn) {
    case 64: return TileCfg<64>::kSmemBytes;
    case 128: return TileCfg<128>::kSmemBytes;
    case 256: return TileCfg<256>::kSmemBytes;
    default: return 0;
  }
}

int kernel_threads(int depth) {
  return depth == 0 ? RoleCfg<0>::kThreads : RoleCfg<1>::kThreads;
}

cudaError_t launch_gemm(int bn, int depth, const KernelParams& p, const StrassenTable* tab, int grid,
                        cudaStream_t stream) {
  if (depth == 1) return tab ? launch_gemm_depth1(bn, p, *tab, grid, stream) : cudaErrorInvalidValue;
  if (depth == 2) return tab ? launch_gemm_depth2(bn, p, *tab, grid, stream) : cudaErrorInvalidValue;
  if (depth != 0) return cudaErrorInvalidValue;
  switch (bn) {
    case 64: return launch_gemm_t<64, 0>(p, nullptr, grid, stream);
    case 128: return launch_gemm_t<128, 0>(p, nullptr, grid, stream);
    case 256: return launch_gemm_t<256, 0>(p, nullptr, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// C = epi(bias) when the product is empty (K == 0): alpha * 0 + bias.
__global__ void k0_fill_kernel(const __grid_constant__ KernelParams p) {
  const long long total = static_cast<long long>(p.M) * p.n_out;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(idx / p.n_out);
    const int col = static_cast<int>(idx % p.n_out);
    float v = p.bias ? ld_bias(p, col) : 0.0f;
    if (p.epi == kEpiSwiglu) {
      const float u = p.bias ? ld_bias(p, p.n_out + col) : 0.0f;
      v = silu(v) * u;
    } else if (p.epi == kEpiSilu) {
      v = silu(v);
    }
    p.C[static_cast<long long>(row) * p.ldc + col] = pack1(v, p.is_bf16);
  }
}

// Nothing ever arrives on `bar`, so the wait for its phase 0 can only end
// by its time limit; the helper then latches the timeout in p.err.
__global__ void selftest_wait_kernel(const __grid_constant__ KernelParams p) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_one(ptx::smem_u32(&bar), 0, p, 0);
  __syncthreads();
}

cudaError_t launch_selftest_wait(const KernelParams& p, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_k0_fill(const KernelParams& p, cudaStream_t stream) {
  const long long total = static_cast<long long>(p.M) * p.n_out;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  k0_fill_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fgemm
