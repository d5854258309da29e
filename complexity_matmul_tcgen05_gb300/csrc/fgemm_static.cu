// fgemm_static.cu -- a Strassen product that allocates no device memory.
//
// fgemm_matmul_ex keeps the Strassen partial tiles in a workspace that the
// handle grows with cudaMalloc, and a handle itself allocates its error word.
// Some callers cannot do that: a host framework that owns all device memory
// through its own pool and forbids allocations once it has started, a
// latency-critical serving loop that must not hit cudaMalloc's implicit
// device synchronisation, or a plug-in that is only handed a stream.
// fgemm_strassen_matmul_static serves them: it runs the same Strassen kernel,
// with its scratch (error word + partial tiles) in the file-scope array
// below, which is part of the library image.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/fgemm.h"
#include "fgemm_internal.h"

namespace fgemm {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
void set_thread_message(const std::string& text);
}  // namespace fgemm

namespace {

// 64 MiB of scratch on every device that loads the library, held until the
// process exits.  Bytes [0, 256) hold the kernel's error word; the rest holds
// 4^depth fp32 partial tiles of 128 x tile_n per CTA of the launch.
constexpr size_t kScratchBytes = size_t{64} << 20;
constexpr size_t kScratchHeader = 256;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};

fgemm_status_t fail(fgemm_status_t s, const std::string& text) {
  fgemm::set_thread_message(text);
  return s;
}

// Once per device, with that device current: the device address of the
// scratch array (its host-side name is only a stand-in) and the SM count.
fgemm_status_t setup_device(int dev, void** addr, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return fail(FGEMM_ERR_NO_DEVICE, "device index out of range");
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    int major = 0, minor = 0, n = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3 || n <= 0)
      return fail(FGEMM_ERR_NO_DEVICE, "this library is built for sm_103a only");
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
    if (e != cudaSuccess || !ptr)
      return fail(FGEMM_ERR_CUDA,
                  std::string("cudaGetSymbolAddress(static scratch): ") + cudaGetErrorString(e));
    g_scratch_addr[dev] = ptr;
    g_num_sms[dev] = n;
  }
  *addr = g_scratch_addr[dev];
  *sms = g_num_sms[dev];
  return FGEMM_OK;
}

fgemm_status_t encode(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                      uint32_t box_outer, int bf16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = fgemm::tensor_map_encoder();
  if (!enc) return fail(FGEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
          const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")");
  return FGEMM_OK;
}

}  // namespace

extern "C" fgemm_status_t fgemm_strassen_matmul_static(
    int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
    void* C, int64_t ldc, fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, int32_t depth,
    int32_t tile_n, void* cuda_stream) {
  if (depth != 1 && depth != 2) return fail(FGEMM_ERR_INVALID_ARG, "depth must be 1 or 2");
  if (tile_n == 0) tile_n = 128;
  const fgemm_algo_t algo = depth == 1 ? FGEMM_ALGO_STRASSEN1 : FGEMM_ALGO_STRASSEN2;
  fgemm_status_t s =
      fgemm_validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, fgemm::kBM, tile_n);
  if (s != FGEMM_OK) return s;
  const int32_t kind = epi ? epi->kind : FGEMM_EPI_NONE;
  const int64_t n_out = kind == FGEMM_EPI_SWIGLU ? N / 2 : N;
  if (M == 0 || n_out == 0) return FGEMM_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FGEMM_ERR_NO_DEVICE, "cudaGetDevice failed");
  void* scratch = nullptr;
  int sms = 0;
  s = setup_device(dev, &scratch, &sms);
  if (s != FGEMM_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  fgemm::KernelParams p;
  std::memset(&p, 0, sizeof(p));
  p.A = static_cast<const uint16_t*>(A);
  p.B = static_cast<const uint16_t*>(B);
  p.C = static_cast<uint16_t*>(C);
  p.bias = epi ? static_cast<const uint16_t*>(epi->bias) : nullptr;
  p.err = static_cast<unsigned int*>(scratch);
  p.workspace = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kScratchHeader);
  p.lda = lda;
  p.ldb = ldb;
  p.ldc = ldc;
  const char* spin = std::getenv("FGEMM_SPIN_LIMIT_MS");
  const double spin_ms = spin && *spin ? std::max(1.0, std::atof(spin)) : 1000.0;
  p.spin_ns = static_cast<unsigned long long>(spin_ms * 1e6);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.n_out = static_cast<int>(n_out);
  p.epi = kind;
  p.is_bf16 = dtype == FGEMM_BF16 ? 1 : 0;
  p.alpha = epi ? epi->alpha : 1.0f;

  cudaError_t e;
  if (K == 0) {
    e = fgemm::launch_k0_fill(p, stream);
    return e == cudaSuccess ? FGEMM_OK
                            : fail(FGEMM_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
  }

  p.sub_m = static_cast<int>(M >> depth);
  p.sub_n = static_cast<int>(N >> depth);
  p.sub_k = static_cast<int>(K >> depth);
  p.tiles_m = p.sub_m / fgemm::kBM;
  p.tiles_n = p.sub_n / tile_n;
  const long long units = static_cast<long long>(p.tiles_m) * p.tiles_n;
  p.num_units = static_cast<int>(units);
  p.k_blocks = p.sub_k / fgemm::kBK;
  p.raster_group = 8;
  const uint32_t fmt = p.is_bf16 ? 1u : 0u;
  p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 16) |
            (static_cast<uint32_t>(tile_n >> 3) << 17) |
            (static_cast<uint32_t>(fgemm::kBM >> 4) << 24);
  p.num_products = depth == 1 ? 7 : 49;
  const fgemm::StrassenTable& tab = fgemm::strassen_table(depth);

  const int grid = static_cast<int>(std::min<long long>(units, sms));
  const size_t per_cta = (size_t{1} << (2 * depth)) * fgemm::kBM * static_cast<size_t>(tile_n) * 4;
  const size_t need = per_cta * static_cast<size_t>(grid);
  if (need > kScratchBytes - kScratchHeader) {
    return fail(FGEMM_ERR_UNSUPPORTED,
                "this product needs " + std::to_string(need >> 20) + " MiB of partial tiles (" +
                    std::to_string(grid) + " CTAs x " + std::to_string(per_cta >> 10) +
                    " KiB) but the static scratch holds " +
                    std::to_string((kScratchBytes - kScratchHeader) >> 20) +
                    " MiB; use a smaller tile_n or depth, or fgemm_matmul_ex");
  }
  s = encode(&p.tmap_a, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
             static_cast<uint64_t>(lda), fgemm::kBM, p.is_bf16);
  if (s != FGEMM_OK) return s;
  s = encode(&p.tmap_b, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K),
             static_cast<uint64_t>(ldb), fgemm::kBK, p.is_bf16);
  if (s != FGEMM_OK) return s;
  // The partial tiles need no clearing: each product's first contribution to
  // a block stores instead of adding.  The error word is not cleared here: it
  // starts at zero when the library is loaded, a timeout latches into it and
  // stays until fgemm_strassen_static_get_error reads and clears it, so a
  // failed call cannot be hidden by a later one.
  e = fgemm::launch_gemm(tile_n, depth, p, &tab, grid, stream);
  if (e != cudaSuccess) return fail(FGEMM_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
  return FGEMM_OK;
}

extern "C" fgemm_status_t fgemm_strassen_static_get_error(void* cuda_stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FGEMM_ERR_NO_DEVICE, "cudaGetDevice failed");
  void* scratch = nullptr;
  int sms = 0;
  fgemm_status_t s = setup_device(dev, &scratch, &sms);
  if (s != FGEMM_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess)
    return fail(FGEMM_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  unsigned int word = 0;
  e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess)
    return fail(FGEMM_ERR_CUDA, std::string("reading the error word: ") + cudaGetErrorString(e));
  if (word == 0) {
    fgemm::set_thread_message("");
    return FGEMM_OK;
  }
  e = cudaMemset(scratch, 0, sizeof(unsigned int));
  if (e != cudaSuccess)
    return fail(FGEMM_ERR_CUDA, std::string("clearing the error word: ") + cudaGetErrorString(e));
  static const char* roles[] = {"producer", "mma", "epilogue", "operand-sum"};
  const unsigned role = (word >> 24) & 0xF;
  char text[160];
  std::snprintf(text, sizeof(text),
                "a bounded wait ran out in the %s role of block %u (word 0x%08x)",
                role < 4 ? roles[role] : "?", word & 0xFFFFFFu, word);
  return fail(FGEMM_ERR_TIMEOUT, text);
}

extern "C" fgemm_status_t fgemm_strassen_static_selftest_timeout(int32_t limit_ms,
                                                                 void* cuda_stream) {
  if (limit_ms < 1 || limit_ms > 10000) return fail(FGEMM_ERR_INVALID_ARG, "limit_ms must be in 1..10000");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FGEMM_ERR_NO_DEVICE, "cudaGetDevice failed");
  void* scratch = nullptr;
  int sms = 0;
  fgemm_status_t s = setup_device(dev, &scratch, &sms);
  if (s != FGEMM_OK) return s;
  fgemm::KernelParams p;
  std::memset(&p, 0, sizeof(p));
  p.err = static_cast<unsigned int*>(scratch);
  p.spin_ns = static_cast<unsigned long long>(limit_ms) * 1000000ull;
  const cudaError_t e = fgemm::launch_selftest_wait(p, static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? FGEMM_OK
                          : fail(FGEMM_ERR_CUDA, std::string("self-test launch: ") + cudaGetErrorString(e));
}
