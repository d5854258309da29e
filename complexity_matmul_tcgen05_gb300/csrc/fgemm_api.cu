// fgemm_api.cpp -- the C ABI (include/fgemm.h): handles, argument checks,
// plan cache, tensor-map encoding, Strassen coefficient tables, launches and
// calibration.  Host code only; kernels live in the fgemm_kern_*.cu files.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/fgemm.h"
#include "fgemm_internal.h"

namespace fgemm {
bool form_is_legal(int64_t M, int64_t N, int64_t K, int32_t epi_kind, fgemm_algo_t algo,
                   int32_t tile_m, int32_t tile_n);
// The decision: the form and tile of least predicted time among those that
// `algo` (AUTO: every form), `tile_m` / `tile_n` (0: any) and `min_tile_m`
// allow; under AUTO a low-complexity form only when its prediction is below
// (1 - lcma_margin) times the best classical one.  The time returned is the
// pick's own prediction.  FGEMM_ERR_UNSUPPORTED when nothing is legal.
fgemm_status_t model_search(const fgemm_device_model_t* dev, int64_t M, int64_t N, int64_t K,
                            int32_t epi_kind, fgemm_algo_t algo, int32_t tile_m, int32_t tile_n,
                            int32_t min_tile_m, fgemm_algo_t* algo_out, int32_t* tm_out, int32_t* tn_out,
                            double* us_out);
}

using fgemm::KernelParams;
using fgemm::StrassenTable;

namespace {

thread_local std::string g_thread_msg;

// ------------------------------------------------------------------ helpers

int depth_of(fgemm_algo_t a) {
  return (a == FGEMM_ALGO_STRASSEN1 || a == FGEMM_ALGO_WINOGRAD1) ? 1
                                                                 : (a == FGEMM_ALGO_STRASSEN2 ? 2 : 0);
}

constexpr fgemm_algo_t kForms[4] = {FGEMM_ALGO_CLASSICAL, FGEMM_ALGO_STRASSEN1, FGEMM_ALGO_STRASSEN2,
                                    FGEMM_ALGO_WINOGRAD1};

fgemm_status_t fail(std::string* msg, fgemm_status_t s, const std::string& text) {
  if (msg) *msg = text;
  return s;
}

// ------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct TmapKey {
  const void* ptr;
  uint64_t inner, outer, ld;
  uint32_t box_inner, box_outer;
  int bf16;
  bool operator==(const TmapKey& o) const {
    return ptr == o.ptr && inner == o.inner && outer == o.outer && ld == o.ld &&
           box_inner == o.box_inner && box_outer == o.box_outer && bf16 == o.bf16;
  }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey& k) const {
    size_t h = std::hash<const void*>()(k.ptr);
    h ^= std::hash<uint64_t>()(k.inner * 1000003u + k.outer) + 0x9e3779b97f4a7c15ull + (h << 6);
    h ^= std::hash<uint64_t>()(k.ld * 31u + k.box_outer * 7u + k.box_inner * 131u + k.bf16) + (h << 6) +
         (h >> 2);
    return h;
  }
};

struct PlanKey {
  int64_t M, N, K;
  int32_t epi, algo, tile_m, tile_n;
  int32_t wide_classical;  // plans restricted to classical 128/256-row tiles
  bool operator==(const PlanKey& o) const {
    return M == o.M && N == o.N && K == o.K && epi == o.epi && algo == o.algo &&
           tile_m == o.tile_m && tile_n == o.tile_n && wide_classical == o.wide_classical;
  }
};
struct PlanKeyHash {
  size_t operator()(const PlanKey& k) const {
    size_t h = std::hash<int64_t>()(k.M);
    h = h * 1000003u ^ std::hash<int64_t>()(k.N);
    h = h * 1000003u ^ std::hash<int64_t>()(k.K);
    h = h * 1000003u ^ static_cast<size_t>(k.epi * 512 + k.algo * 64 + (k.tile_m >> 4) + (k.tile_n >> 6) +
                                           k.wide_classical * 4096);
    return h;
  }
};
struct Plan {
  fgemm_algo_t algo;
  int32_t tile_m;
  int32_t tile_n;
  double predicted_us;
};

}  // namespace

namespace fgemm {
// The tensor-map encoder, for other host translation units.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return get_encode_fn(); }
void set_thread_message(const std::string& text) { g_thread_msg = text; }
}  // namespace fgemm

struct fgemm_handle_s {
  int device = 0;
  int num_sms = 0;
  cudaStream_t stream = nullptr;
  unsigned int* d_err = nullptr;
  float* workspace = nullptr;
  size_t ws_bytes = 0;
  void* mx_buf = nullptr;             // bf16 values of MX inputs
  size_t mx_bytes = 0;
  unsigned int* split_ctr = nullptr;  // K-split arrival counters (zeroed once)
  size_t split_ctr_count = 0;
  unsigned int split_gen = 0;         // generation of the last split launch
  int split_mode = 1;                 // 0 never, 1 auto, 2 whenever possible
  int lcma_formation = 0;             // 0 auto, 1 pre-pass launch, 2 inside the product kernel
  unsigned int* form_ctr = nullptr;   // band counters of the in-kernel formation (3 words)
  // fgemm_matmul_host: two device slots each of B (with the bias), of A row
  // blocks and of C row blocks; an upload and a download stream; the events
  // that order them with the handle's stream; the host ranges of C the last
  // two calls write, with the events that mark them written
  void* host_buf = nullptr;
  size_t host_cap_b = 0, host_cap_a = 0, host_cap_c = 0;  // bytes of one slot of each kind
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t ev_start = nullptr, ev_b = nullptr, ev_a[2] = {nullptr, nullptr}, ev_c[2] = {nullptr, nullptr},
              ev_d[2] = {nullptr, nullptr}, ev_bfree[2] = {nullptr, nullptr}, ev_done[2] = {nullptr, nullptr};
  unsigned long long host_calls = 0, host_blocks = 0;
  uintptr_t c_lo[2] = {0, 0}, c_hi[2] = {0, 0};
  unsigned long long spin_ns = 1000000000ull;
  fgemm_device_model_t model{};
  std::unordered_map<PlanKey, Plan, PlanKeyHash> plans;
  std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> tmaps;
  std::string msg;
};

namespace {

fgemm_status_t set_msg(fgemm_handle_t h, fgemm_status_t s, const std::string& text) {
  if (h)
    h->msg = text;
  else
    g_thread_msg = text;
  return s;
}

fgemm_status_t cuda_fail(fgemm_handle_t h, cudaError_t e, const char* what) {
  std::string t = std::string(what) + ": " + cudaGetErrorString(e);
  return set_msg(h, FGEMM_ERR_CUDA, t);
}

// A 2D map of 16-bit elements (inner x outer, row pitch ld elements) with
// boxes of box_inner x box_outer.  Boxes 64 elements wide (128-byte rows)
// use the 128-byte swizzle, 32 wide the 64-byte one.
fgemm_status_t encode_tmap(fgemm_handle_t h, CUtensorMap* out, const void* ptr, uint64_t inner,
                           uint64_t outer, uint64_t ld, uint32_t box_outer, int bf16,
                           uint32_t box_inner = 64) {
  TmapKey key{ptr, inner, outer, ld, box_inner, box_outer, bf16};
  auto it = h->tmaps.find(key);
  if (it != h->tmaps.end()) {
    *out = it->second;
    return FGEMM_OK;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc) return set_msg(h, FGEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  CUtensorMap m;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_inner == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_msg(h, FGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")");
  if (h->tmaps.size() > 256) h->tmaps.clear();
  h->tmaps.emplace(key, m);
  *out = m;
  return FGEMM_OK;
}

// The checks fgemm_matmul_ex makes before launching (see fgemm.h).
fgemm_status_t validate(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                        int64_t ldb, const void* C, int64_t ldc, fgemm_dtype_t dtype,
                        const fgemm_epilogue_t* epi, fgemm_algo_t algo, int32_t tile_m,
                        int32_t tile_n, std::string* msg) {
  const int32_t kind = epi ? epi->kind : FGEMM_EPI_NONE;
  if (dtype != FGEMM_F16 && dtype != FGEMM_BF16)
    return fail(msg, FGEMM_ERR_INVALID_ARG, "dtype must be FGEMM_F16 or FGEMM_BF16");
  if (kind < FGEMM_EPI_NONE || kind > FGEMM_EPI_SWIGLU)
    return fail(msg, FGEMM_ERR_INVALID_ARG, "unknown epilogue kind");
  if (algo < FGEMM_ALGO_AUTO || algo > FGEMM_ALGO_WINOGRAD1)
    return fail(msg, FGEMM_ERR_INVALID_ARG, "unknown algorithm");
  if (tile_n != 0 && tile_n != 64 && tile_n != 128 && tile_n != 256)
    return fail(msg, FGEMM_ERR_INVALID_ARG, "tile_n must be 0, 64, 128 or 256");
  if (tile_m != 0 && tile_m != 16 && tile_m != 32 && tile_m != 64 && tile_m != 128 && tile_m != 256)
    return fail(msg, FGEMM_ERR_INVALID_ARG, "tile_m must be 0, 16, 32, 64, 128 or 256");
  if (M < 0 || N < 0 || K < 0) return fail(msg, FGEMM_ERR_INVALID_ARG, "negative dimension");
  const int64_t kMax = (int64_t{1} << 31) - 1;
  if (M > kMax || N > kMax || K > kMax)
    return fail(msg, FGEMM_ERR_INVALID_ARG, "dimension above 2^31 - 1");
  if (kind == FGEMM_EPI_SWIGLU && (N % 2) != 0)
    return fail(msg, FGEMM_ERR_INVALID_ARG, "SWIGLU needs an even N (gate | up)");
  const int64_t n_out = kind == FGEMM_EPI_SWIGLU ? N / 2 : N;
  if (kind == FGEMM_EPI_SCALE_BIAS && (!epi || !epi->bias))
    return fail(msg, FGEMM_ERR_INVALID_ARG, "SCALE_BIAS needs a bias vector");
  if (epi && epi->bias && (reinterpret_cast<uintptr_t>(epi->bias) & 1u))
    return fail(msg, FGEMM_ERR_ALIGNMENT, "bias must be 2-byte aligned");
  if (M == 0 || n_out == 0) return FGEMM_OK;  // nothing to compute
  if (!C) return fail(msg, FGEMM_ERR_INVALID_ARG, "C is NULL");
  if (ldc < n_out) return fail(msg, FGEMM_ERR_INVALID_ARG, "ldc < output width");
  if ((reinterpret_cast<uintptr_t>(C) & 15u) || (ldc % 8) != 0)
    return fail(msg, FGEMM_ERR_ALIGNMENT, "C must be 16-byte aligned with ldc a multiple of 8");
  if (K == 0) return FGEMM_OK;  // C = epi(bias), A and B unused
  if (!A || !B) return fail(msg, FGEMM_ERR_INVALID_ARG, "A or B is NULL");
  if (lda < K) return fail(msg, FGEMM_ERR_INVALID_ARG, "lda < K");
  if (ldb < N) return fail(msg, FGEMM_ERR_INVALID_ARG, "ldb < N");
  if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u))
    return fail(msg, FGEMM_ERR_ALIGNMENT, "A and B must be 16-byte aligned");
  if ((lda % 8) != 0 || (ldb % 8) != 0)
    return fail(msg, FGEMM_ERR_ALIGNMENT, "lda and ldb must be multiples of 8 elements");
  if (kind == FGEMM_EPI_SWIGLU && (N % 16) != 0)
    return fail(msg, FGEMM_ERR_ALIGNMENT, "SWIGLU needs N a multiple of 16 (up half 16-byte aligned)");
  if (algo != FGEMM_ALGO_AUTO || tile_m != 0 || tile_n != 0) {
    bool any = false;
    for (fgemm_algo_t a : kForms) {
      if (algo != FGEMM_ALGO_AUTO && a != algo) continue;
      for (int32_t tm : {16, 32, 64, 128, 256}) {
        if (tile_m != 0 && tm != tile_m) continue;
        for (int32_t tn : {64, 128, 256}) {
          if (tile_n != 0 && tn != tile_n) continue;
          any = any || fgemm::form_is_legal(M, N, K, kind, a, tm, tn);
        }
      }
    }
    if (!any)
      return fail(msg, FGEMM_ERR_UNSUPPORTED,
                  "no legal form/tile: Strassen and Winograd forms need M, N, K divisible into "
                  "2^d blocks of whole 128 x tile_n x 64 tiles; 256-row tiles are classical or "
                  "one Strassen level only; tile_m 16/32/64 (small M) needs M <= tile_m, "
                  "tile_n 128, classical, no SWIGLU; SWIGLU needs tile_n >= 128");
  }
  return FGEMM_OK;
}

fgemm_status_t choose_plan(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, int32_t kind,
                           fgemm_algo_t algo, int32_t tile_m, int32_t tile_n, Plan* out,
                           bool wide_classical = false) {
  PlanKey key{M, N, K, kind, static_cast<int32_t>(algo), tile_m, tile_n, wide_classical ? 1 : 0};
  auto it = h->plans.find(key);
  if (it != h->plans.end()) {
    *out = it->second;
    return FGEMM_OK;
  }
  Plan p{FGEMM_ALGO_CLASSICAL, 0, 0, INFINITY};
  // the same decision as fgemm_model_plan (under AUTO, the margin a
  // low-complexity form must win by)
  if (fgemm::model_search(&h->model, M, N, K, kind, wide_classical ? FGEMM_ALGO_CLASSICAL : algo, tile_m,
                          tile_n, wide_classical ? 128 : 0, &p.algo, &p.tile_m, &p.tile_n,
                          &p.predicted_us) != FGEMM_OK)
    return set_msg(h, FGEMM_ERR_UNSUPPORTED, "no legal form/tile for this shape");
  if (h->plans.size() > 4096) h->plans.clear();
  h->plans.emplace(key, p);
  *out = p;
  return FGEMM_OK;
}

fgemm_status_t ensure_workspace(fgemm_handle_t h, size_t bytes) {
  if (bytes <= h->ws_bytes) return FGEMM_OK;
  if (h->workspace) {
    cudaError_t e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
    cudaFree(h->workspace);
    h->workspace = nullptr;
    h->ws_bytes = 0;
  }
  cudaError_t e = cudaMalloc(&h->workspace, bytes);
  if (e != cudaSuccess) {
    h->workspace = nullptr;
    return cuda_fail(h, e, "cudaMalloc(partial-tile workspace)");
  }
  h->ws_bytes = bytes;
  return FGEMM_OK;
}

// Arrival counters for pieces (at least `ctrs`), zeroed when (re)allocated,
// and the next launch generation (1 .. 2^24 - 1) in h->split_gen.
fgemm_status_t ensure_counters(fgemm_handle_t h, size_t ctrs) {
  if (ctrs > h->split_ctr_count) {
    if (h->split_ctr) {
      cudaError_t e = cudaStreamSynchronize(h->stream);
      if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
      cudaFree(h->split_ctr);
      h->split_ctr = nullptr;
      h->split_ctr_count = 0;
    }
    const size_t n = std::max<size_t>(ctrs, static_cast<size_t>(8) * h->num_sms);
    cudaError_t e = cudaMalloc(&h->split_ctr, n * sizeof(unsigned int));
    if (e != cudaSuccess) {
      h->split_ctr = nullptr;
      return cuda_fail(h, e, "cudaMalloc(split counters)");
    }
    e = cudaMemset(h->split_ctr, 0, n * sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemset(split counters)");
    h->split_ctr_count = n;
    h->split_gen = 0;
  }
  // Counters hold gen << 8 | arrivals; a counter tagged with an older
  // generation (e.g. left by a launch that ended on an error) reads as zero
  // arrivals.  When the 24-bit generation wraps, clear them all.
  if (++h->split_gen >= (1u << 24)) {
    cudaError_t e =
        cudaMemsetAsync(h->split_ctr, 0, h->split_ctr_count * sizeof(unsigned int), h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemsetAsync(split counters)");
    h->split_gen = 1;
  }
  return FGEMM_OK;
}

// Workspace, counters and generation of a K-split pair launch.
fgemm_status_t prepare_split(fgemm_handle_t h, KernelParams* p, int split, int pieces, int bn) {
  const size_t slots = static_cast<size_t>(split) * pieces * 2;
  fgemm_status_t s =
      ensure_workspace(h, slots * fgemm::kBM * static_cast<size_t>(bn) * sizeof(float));
  if (s != FGEMM_OK) return s;
  s = ensure_counters(h, static_cast<size_t>(split) * 8);  // 2 CTAs x 4 epilogue warps
  if (s != FGEMM_OK) return s;
  p->split_tiles = split;
  p->split_pieces = pieces;
  p->split_gen = h->split_gen;
  p->split_ctr = h->split_ctr;
  p->split_ws = h->workspace;
  return FGEMM_OK;
}


// One Strassen-like level on CTA pairs with the summed operands streamed
// through HBM: the scheme's distinct summed operands become temporaries
// (formed by one pre-pass launch), the product kernel reads every operand
// through a tensor map of A, B or the temporaries.  Workspace layout: the
// product kernel's partial tiles, then the A and the B temporaries.
// Whether product k of the table reads a sum of A's blocks (bit 0) and of
// B's (bit 1); a single positive term is a raw block, read in place.
int lcma_needs(const StrassenTable& tab, int k) {
  auto sum = [](int n, const uint8_t* c) { return !(n == 1 && !(c[0] & fgemm::kTermNeg)); };
  return (sum(tab.na[k], tab.a[k]) ? 1 : 0) | (sum(tab.nb[k], tab.b[k]) ? 2 : 0);
}

// The order in which the pair kernel runs a scheme's products (and folds
// them): those that read no sum first, then those that read sums of A only,
// then of B only, then of both, each group in table order.  Winograd's
// stays as it is (A11 B11, A12 B21 first); Strassen's becomes M2, M5, M3,
// M4, M1, M6, M7.  The order is the same whoever forms the sums, so the
// result is too.
void lcma_order(const StrassenTable& tab, int np, int (&order)[fgemm::kLcmaProducts]) {
  int n = 0;
  for (int key = 0; key < 4; ++key)
    for (int k = 0; k < np; ++k)
      if (lcma_needs(tab, k) == key) order[n++] = k;
}

// Which sides' sums the product kernel forms itself (bit 0: A's, bit 1:
// B's; the pre-pass forms the others), and how many products run before the
// first that reads one of them (*lead).  Both sides when the scheme has
// products that read no sum (Winograd), else B's side alone when it has
// products that read no sum of B (Strassen: M2 and M5).  Mode 2 of the
// handle asks for it whenever possible, mode 0 (auto) when those products
// span at least kFusedMinWaves waves; the matrices must cut into whole
// formation bands.
int lcma_formation_plan(fgemm_handle_t h, const StrassenTable& tab, long long positions, int clusters, int sub_m,
                        int sub_k, int* lead) {
  constexpr int np = 7;  // one level (two levels always take the pre-pass)
  int order[fgemm::kLcmaProducts];
  lcma_order(tab, np, order);
  int none = 0, no_b = 0;
  while (none < np && lcma_needs(tab, order[none]) == 0) ++none;
  while (no_b < np && !(lcma_needs(tab, order[no_b]) & 2)) ++no_b;
  const int mask = none > 0 ? 3 : (no_b > 0 ? 2 : 0);
  const int ld = none > 0 ? none : no_b;
  if (lead) *lead = ld;
  const long long whole = positions / std::max(clusters, 1);
  const bool whole_bands = sub_m % fgemm::kFormRows == 0 && sub_k % fgemm::kFormRows == 0;
  if (mask == 0 || !whole_bands || h->lcma_formation == 1) return 0;
  if (h->lcma_formation == 2 || ld * whole >= fgemm::kFusedMinWaves) return mask;
  return 0;
}

fgemm_status_t launch_lcma(fgemm_handle_t h, KernelParams& p, const StrassenTable& tab, int depth, int bn,
                           const void* A, int64_t lda, const void* B, int64_t ldb) {
  using fgemm::LcmaFormParams;
  using fgemm::LcmaParams;
  LcmaParams L;
  std::memset(&L, 0, sizeof(L));
  LcmaFormParams F;
  std::memset(&F, 0, sizeof(F));
  const int np = depth == 1 ? 7 : 49;
  const int nblk = 1 << (2 * depth);  // blocks of each matrix, and output blocks
  // the distinct summed operands of each side (a single positive term is a
  // raw block of A or B, read in place)
  auto operand = [&](int n, const uint8_t* codes, fgemm::LcmaFormJob& J, uint8_t* is_temp,
                     uint8_t* idx) {
    if (n == 1 && !(codes[0] & fgemm::kTermNeg)) {
      *is_temp = 0;
      *idx = codes[0] & fgemm::kTermIndexMask;
      return;
    }
    int8_t coef[fgemm::kLcmaMaxBlocks] = {0};
    for (int i = 0; i < n; ++i)
      coef[codes[i] & fgemm::kTermIndexMask] += (codes[i] & fgemm::kTermNeg) ? -1 : 1;
    int t = 0;
    while (t < J.ntemp && std::memcmp(J.coef[t], coef, sizeof(coef)) != 0) ++t;
    if (t == J.ntemp) {
      std::memcpy(J.coef[t], coef, sizeof(coef));
      for (int q = 0; q < nblk; ++q)
        if (coef[q] != 0) J.block_mask |= 1u << q;
      ++J.ntemp;
    }
    *is_temp = 1;
    *idx = static_cast<uint8_t>(t);
  };
  // the products in the kernel's order (lcma_order): L.prod[pr] is table
  // product order[pr]
  // (two levels: table order; every product but four reads sums, all
  // formed by the pre-pass)
  int order[fgemm::kLcmaProducts];
  if (depth == 1)
    lcma_order(tab, np, order);
  else
    for (int k = 0; k < np; ++k) order[k] = k;
  int first_of[fgemm::kLcmaMaxBlocks], last_of[fgemm::kLcmaMaxBlocks];  // product per output block
  for (int b = 0; b < fgemm::kLcmaMaxBlocks; ++b) first_of[b] = last_of[b] = -1;
  for (int pr = 0; pr < np; ++pr) {
    fgemm::LcmaProduct& P = L.prod[pr];
    const int k = order[pr];
    operand(tab.na[k], tab.a[k], F.job[0], &P.a_temp, &P.a_idx);
    operand(tab.nb[k], tab.b[k], F.job[1], &P.b_temp, &P.b_idx);
    P.nc = tab.nc[k];
    for (int t = 0; t < P.nc; ++t) {
      P.c[t] = static_cast<uint8_t>(tab.c[k][t] & (fgemm::kTermIndexMask | fgemm::kTermNeg));
      const int blk = P.c[t] & fgemm::kTermIndexMask;
      if (first_of[blk] < 0) first_of[blk] = pr;
      last_of[blk] = pr;
    }
  }
  // where each output is complete (fin: the block, or for SwiGLU the block
  // row, whose value is known once this product is in), the first
  // contribution to each block (stored, not added) and the contribution
  // that completes a block's output (kTermLast: kept out of the partial, the
  // output is finished from the partial and the accumulator).  For SwiGLU a
  // block's last contribution can come before its row is complete (C12's
  // M5 before the gate's M7): it is folded like any other.
  const bool swiglu = p.epi == FGEMM_EPI_SWIGLU;
  for (int pr = 0; pr < np; ++pr) {
    fgemm::LcmaProduct& P = L.prod[pr];
    P.fin = 0;
    P.groups = 0;
    for (int b = 0; b < nblk; ++b)
      if (!swiglu && last_of[b] == pr) P.fin |= static_cast<uint16_t>(1u << b);
    for (int sr = 0; sr < 2; ++sr)
      if (swiglu && std::max(last_of[2 * sr], last_of[2 * sr + 1]) == pr)
        P.fin |= static_cast<uint16_t>(1u << sr);
    for (int t = 0; t < P.nc; ++t) {
      const int blk = P.c[t] & fgemm::kTermIndexMask;
      const int group = swiglu ? blk >> 1 : blk;
      if (first_of[blk] == pr) P.c[t] |= fgemm::kTermFirst;
      if (last_of[blk] == pr && ((P.fin >> group) & 1u)) P.c[t] |= fgemm::kTermLast;
      P.groups |= static_cast<uint16_t>(1u << group);
    }
  }
  for (int g = 0; g < nblk; ++g) {
    int n = 0;
    for (int pr = 0; pr < np; ++pr) n += (L.prod[pr].groups >> g) & 1u;
    L.group_pieces[g] = static_cast<uint8_t>(n);
  }
  if (depth == 2) {
    // the two-level pre-pass forms product (p, q)'s operand as the inner
    // combination q of the outer combination p (fgemm::strassen_coef): it
    // must be the table's operand
    for (int side = 0; side < 2; ++side) {
      fgemm::LcmaFormJob& J = F.job[side];
      for (int k = 0; k < np; ++k) {
        const fgemm::LcmaProduct& P = L.prod[k];
        const int n = side == 0 ? tab.na[k] : tab.nb[k];
        const uint8_t* codes = side == 0 ? tab.a[k] : tab.b[k];
        int8_t want[fgemm::kLcmaMaxBlocks] = {0}, got[fgemm::kLcmaMaxBlocks] = {0};
        for (int i = 0; i < n; ++i)
          want[codes[i] & fgemm::kTermIndexMask] += (codes[i] & fgemm::kTermNeg) ? -1 : 1;
        for (int i = 0; i < 4; ++i)
          for (int j = 0; j < 4; ++j)
            got[(2 * (i >> 1) + (j >> 1)) * 4 + 2 * (i & 1) + (j & 1)] = static_cast<int8_t>(
                fgemm::strassen_coef(side, k / 7, i) * fgemm::strassen_coef(side, k % 7, j));
        if (std::memcmp(want, got, sizeof(want)) != 0)
          return set_msg(h, FGEMM_ERR_UNSUPPORTED, "two-level operand table does not match the pre-pass");
        const bool temp = side == 0 ? P.a_temp : P.b_temp;
        J.leaf_temp[k] = temp ? static_cast<int8_t>(side == 0 ? P.a_idx : P.b_idx) : static_cast<int8_t>(-1);
      }
    }
  }
  const int ntA = F.job[0].ntemp, ntB = F.job[1].ntemp;
  const int fit = fgemm::lcma_pair_clusters_fit(bn, depth);
  if (fit <= 0) return set_msg(h, FGEMM_ERR_CUDA, "cannot size the Strassen pair launch");
  const long long positions = p.num_units;
  L.units = positions * np;
  const int clusters = static_cast<int>(fgemm_lcma_pair_clusters(positions, depth, fit));
  // the positions of the partial last wave run as separate product units;
  // every CTA keeps the partials of each of its whole positions
  const long long tail_positions = positions % clusters;
  const long long whole = positions / clusters;
  const size_t slot_bytes = static_cast<size_t>(2) * clusters * static_cast<size_t>(std::max<long long>(whole, 1)) *
                            fgemm::lcma_slot_floats(bn, depth) * sizeof(float);
  const size_t tail_bytes =
      static_cast<size_t>(tail_positions) * np * 2 * fgemm::kBM * static_cast<size_t>(bn) * sizeof(float);
  const size_t ta_elems = static_cast<size_t>(ntA) * p.sub_m * p.sub_k;
  const size_t tb_elems = static_cast<size_t>(ntB) * p.sub_k * p.sub_n;
  auto align = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t tail_off = align(slot_bytes);
  const size_t ta_off = tail_off + align(tail_bytes), tb_off = ta_off + align(ta_elems * 2);
  fgemm_status_t s = ensure_workspace(h, tb_off + align(tb_elems * 2));
  if (s != FGEMM_OK) return s;
  // 4^depth output groups x 2 CTAs x 4 epilogue warps per tail position
  s = ensure_counters(h, static_cast<size_t>(std::max<long long>(tail_positions, 1)) * nblk * 8);
  if (s != FGEMM_OK) return s;
  uint8_t* ws = reinterpret_cast<uint8_t*>(h->workspace);
  uint16_t* TA = reinterpret_cast<uint16_t*>(ws + ta_off);
  uint16_t* TB = reinterpret_cast<uint16_t*>(ws + tb_off);
  p.workspace = h->workspace;
  p.split_ws = reinterpret_cast<float*>(ws + tail_off);
  p.split_ctr = h->split_ctr;
  p.split_gen = h->split_gen;
  p.num_products = np;
  L.tmap_ta = p.tmap_a;
  L.tmap_tb = p.tmap_b;
  if (ntA > 0) {
    s = encode_tmap(h, &L.tmap_ta, TA, static_cast<uint64_t>(p.sub_k),
                    static_cast<uint64_t>(ntA) * p.sub_m, static_cast<uint64_t>(p.sub_k), fgemm::kBM,
                    p.is_bf16);
    if (s != FGEMM_OK) return s;
  }
  if (ntB > 0) {
    s = encode_tmap(h, &L.tmap_tb, TB, static_cast<uint64_t>(p.sub_n),
                    static_cast<uint64_t>(ntB) * p.sub_k, static_cast<uint64_t>(p.sub_n), fgemm::kBK,
                    p.is_bf16);
    if (s != FGEMM_OK) return s;
  }
  L.k = p;
  F.is_bf16 = p.is_bf16;
  F.job[0].src = static_cast<const uint16_t*>(A);
  F.job[0].ld = lda;
  F.job[0].dst = TA;
  F.job[0].rows = p.sub_m;
  F.job[0].cols = p.sub_k;
  F.job[1].src = static_cast<const uint16_t*>(B);
  F.job[1].ld = ldb;
  F.job[1].dst = TB;
  F.job[1].rows = p.sub_k;
  F.job[1].cols = p.sub_n;
  // Where the operands are formed: each side by the pre-pass launch, or
  // inside the product kernel while the leading products that do not read
  // that side's sums run (lcma_formation_plan).
  int lead = 0;
  const int mask = depth == 1 ? lcma_formation_plan(h, tab, positions, clusters, p.sub_m, p.sub_k, &lead) : 0;
  const bool fused = mask != 0;
  // A pair's tail units (positions of the partial last wave, one product
  // each) run after its whole positions' first tail_at products, so that the
  // combinations of their accumulators overlap the MMAs of the products that
  // follow: first thing when the pre-pass formed every sum, else after two
  // more products than those that read no sum the kernel forms (then they
  // are stored by the time the tail units read them).
  L.tail_at = fused ? std::min(lead + 2, np) : 0;
  cudaError_t e = cudaSuccess;
  // the pre-pass forms the sides the product kernel does not
  LcmaFormParams pre = F;
  for (int j = 0; j < 2; ++j)
    if ((mask >> j) & 1) pre.job[j].ntemp = 0;
  if (pre.job[0].ntemp > 0 || pre.job[1].ntemp > 0) {
    e = fgemm::launch_lcma_form(pre, depth, h->num_sms, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "operand-sum pre-pass launch");
  }
  if (fused) {
    if (!h->form_ctr) {
      e = cudaMalloc(&h->form_ctr, 4 * sizeof(unsigned int));
      if (e != cudaSuccess) {
        h->form_ctr = nullptr;
        return cuda_fail(h, e, "cudaMalloc(formation counters)");
      }
    }
    e = cudaMemsetAsync(h->form_ctr, 0, 4 * sizeof(unsigned int), h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemsetAsync(formation counters)");
    L.form = F;
    L.form_ctr = h->form_ctr;
    for (int j = 0; j < 2; ++j)
      L.form_tasks[j] = ((mask >> j) & 1) && F.job[j].ntemp > 0 ? F.job[j].rows / fgemm::kFormRows : 0;
  }
  e = fgemm::launch_lcma_pair(bn, depth, L, clusters, h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "Strassen pair kernel launch");
  return FGEMM_OK;
}

// The small-M kernel (tile_m = mp in {16, 32, 64}, M <= mp): C^T = B^T A^T
// over 128-column tiles of C, the K blocks of all tiles shared out over the
// SMs.  A's descriptor uses an {64, mp} box; partial slots and counters are
// two and eight per CTA.
fgemm_status_t launch_small_m(fgemm_handle_t h, KernelParams& p, int64_t M, int64_t N, int64_t K,
                              const void* A, int64_t lda, const void* B, int64_t ldb, int mp) {
  const long long tiles = (static_cast<long long>(p.n_out) + 127) / 128;
  if (tiles > (1ll << 30)) return set_msg(h, FGEMM_ERR_UNSUPPORTED, "too many tiles");
  p.num_units = static_cast<int>(tiles);
  p.tiles_m = 1;
  p.tiles_n = p.num_units;
  p.k_blocks = static_cast<int>((K + fgemm::kBK - 1) / fgemm::kBK);
  const uint32_t fmt = p.is_bf16 ? 1u : 0u;
  // tcgen05 instruction descriptor: fp32 accumulator, A = B^T (MN-major, bit
  // 15), B = A^T (K-major), N = mp, M = 128
  p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 15) |
            (static_cast<uint32_t>(mp >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
  fgemm_status_t s = encode_tmap(h, &p.tmap_a, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                                 static_cast<uint64_t>(lda), static_cast<uint32_t>(mp), p.is_bf16);
  if (s != FGEMM_OK) return s;
  s = encode_tmap(h, &p.tmap_b, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                  static_cast<uint64_t>(ldb), fgemm::kBK, p.is_bf16);
  if (s != FGEMM_OK) return s;
  // every CTA streams at least 8 K blocks, so that a tile is not cut into
  // more pieces than its sum can absorb cheaply; among such grids, one whose
  // shares start at few K offsets of a tile, so that the CTAs read the same
  // rows of B together
  const int ctas = fgemm_small_m_grid(tiles, p.k_blocks, h->num_sms, nullptr);
  if (ctas <= 0) return set_msg(h, FGEMM_ERR_UNSUPPORTED, "cannot size the small-M grid");
  s = ensure_workspace(h, static_cast<size_t>(ctas) * 2 * 128 * static_cast<size_t>(mp) * sizeof(float));
  if (s != FGEMM_OK) return s;
  s = ensure_counters(h, static_cast<size_t>(ctas) * 8);
  if (s != FGEMM_OK) return s;
  p.split_ws = h->workspace;
  p.split_ctr = h->split_ctr;
  p.split_gen = h->split_gen;
  cudaError_t e = fgemm::launch_gemm_skinny(mp, p, ctas, h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "small-M kernel launch");
  return FGEMM_OK;
}

double getenv_double(const char* name, double dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  double d = std::strtod(v, &end);
  return (end && end != v) ? d : dflt;
}

// ------------------------------------------------- calibration JSON I/O

fgemm_status_t load_calibration(fgemm_handle_t h, const char* path) {
  fgemm_device_model_t m = h->model;
  const fgemm_status_t s = fgemm_model_load_json(path, &m);
  if (s != FGEMM_OK)
    return set_msg(h, s == FGEMM_ERR_CALIBRATION ? s : FGEMM_ERR_CALIBRATION,
                   std::string("calibration file unreadable or malformed: ") + path);
  h->model = m;
  h->plans.clear();
  return FGEMM_OK;
}

}  // namespace

// ====================================================================== ABI

extern "C" {

const char* fgemm_status_string(fgemm_status_t s) {
  switch (s) {
    case FGEMM_OK: return "FGEMM_OK";
    case FGEMM_ERR_INVALID_ARG: return "FGEMM_ERR_INVALID_ARG";
    case FGEMM_ERR_ALIGNMENT: return "FGEMM_ERR_ALIGNMENT";
    case FGEMM_ERR_UNSUPPORTED: return "FGEMM_ERR_UNSUPPORTED";
    case FGEMM_ERR_CUDA: return "FGEMM_ERR_CUDA";
    case FGEMM_ERR_TIMEOUT: return "FGEMM_ERR_TIMEOUT";
    case FGEMM_ERR_NO_DEVICE: return "FGEMM_ERR_NO_DEVICE";
    case FGEMM_ERR_CALIBRATION: return "FGEMM_ERR_CALIBRATION";
  }
  return "FGEMM_ERR_UNKNOWN";
}

const char* fgemm_last_message(fgemm_handle_t h) {
  return h ? h->msg.c_str() : g_thread_msg.c_str();
}

fgemm_status_t fgemm_validate(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                              const void* B, int64_t ldb, const void* C, int64_t ldc,
                              fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                              int32_t tile_m, int32_t tile_n) {
  std::string msg;
  fgemm_status_t s =
      validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, tile_m, tile_n, &msg);
  g_thread_msg = msg;
  return s;
}

fgemm_status_t fgemm_create(fgemm_handle_t* out) {
  if (!out) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int dev = 0, count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    return set_msg(nullptr, FGEMM_ERR_NO_DEVICE, "no CUDA device");
  }
  if (cudaGetDevice(&dev) != cudaSuccess) return set_msg(nullptr, FGEMM_ERR_NO_DEVICE, "cudaGetDevice failed");
  int major = 0, minor = 0, sms = 0, l2 = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  if (major != 10 || minor != 3)
    return set_msg(nullptr, FGEMM_ERR_NO_DEVICE,
                   "device is sm_" + std::to_string(major) + std::to_string(minor) +
                       "; this library is built for sm_103a only");
  fgemm_handle_t h = new fgemm_handle_s();
  h->device = dev;
  h->num_sms = sms;
  fgemm_model_default(&h->model, sms, getenv_double("FGEMM_PEAK_TFLOPS", 0.0),
                      getenv_double("FGEMM_HBM_GBS", 0.0));
  if (l2 > 0) h->model.l2_bytes = l2;
  const double spin_ms = getenv_double("FGEMM_SPIN_LIMIT_MS", 1000.0);
  h->spin_ns = static_cast<unsigned long long>(std::max(1.0, spin_ms) * 1e6);
  cudaError_t e = cudaMalloc(&h->d_err, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(unsigned int));
  if (e != cudaSuccess) {
    fgemm_status_t s = cuda_fail(nullptr, e, "cudaMalloc(error word)");
    if (h->d_err) cudaFree(h->d_err);
    delete h;
    return s;
  }
  if (const char* calib = std::getenv("FGEMM_CALIB")) {
    if (*calib) {
      fgemm_status_t s = load_calibration(h, calib);
      if (s != FGEMM_OK) {
        g_thread_msg = h->msg;
        cudaFree(h->d_err);
        delete h;
        return s;
      }
    }
  }
  *out = h;
  return FGEMM_OK;
}

fgemm_status_t fgemm_destroy(fgemm_handle_t h) {
  if (!h) return FGEMM_OK;
  cudaStreamSynchronize(h->stream);
  if (h->workspace) cudaFree(h->workspace);
  if (h->split_ctr) cudaFree(h->split_ctr);
  if (h->form_ctr) cudaFree(h->form_ctr);
  if (h->host_buf) cudaFree(h->host_buf);
  for (cudaStream_t st : {h->up, h->down})
    if (st) cudaStreamDestroy(st);
  for (cudaEvent_t ev : {h->ev_start, h->ev_b, h->ev_a[0], h->ev_a[1], h->ev_c[0], h->ev_c[1], h->ev_d[0],
                         h->ev_d[1], h->ev_bfree[0], h->ev_bfree[1], h->ev_done[0], h->ev_done[1]})
    if (ev) cudaEventDestroy(ev);
  if (h->mx_buf) cudaFree(h->mx_buf);
  if (h->d_err) cudaFree(h->d_err);
  delete h;
  return FGEMM_OK;
}

fgemm_status_t fgemm_set_split_mode(fgemm_handle_t h, int32_t mode) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (mode < 0 || mode > 2) return set_msg(h, FGEMM_ERR_INVALID_ARG, "split mode must be 0, 1 or 2");
  h->split_mode = mode;
  return FGEMM_OK;
}

fgemm_status_t fgemm_set_lcma_formation(fgemm_handle_t h, int32_t mode) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (mode < 0 || mode > 2) return set_msg(h, FGEMM_ERR_INVALID_ARG, "formation mode must be 0, 1 or 2");
  h->lcma_formation = mode;
  return FGEMM_OK;
}

fgemm_status_t fgemm_set_stream(fgemm_handle_t h, void* cuda_stream) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  return FGEMM_OK;
}

fgemm_status_t fgemm_get_device_model(fgemm_handle_t h, fgemm_device_model_t* out) {
  if (!h || !out) return set_msg(h, FGEMM_ERR_INVALID_ARG, "NULL argument");
  *out = h->model;
  return FGEMM_OK;
}

fgemm_status_t fgemm_set_device_model(fgemm_handle_t h, const fgemm_device_model_t* model) {
  if (!h || !model) return set_msg(h, FGEMM_ERR_INVALID_ARG, "NULL argument");
  if (model->num_sms <= 0 || !(model->peak_tflops > 0) || !(model->hbm_gbs > 0))
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "model needs positive SM count, peak and bandwidth");
  h->model = *model;
  h->plans.clear();
  return FGEMM_OK;
}

fgemm_status_t fgemm_plan(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, fgemm_dtype_t dtype,
                          const fgemm_epilogue_t* epi, fgemm_algo_t* algo_out, int32_t* tile_m,
                          int32_t* tile_n, double* predicted_us) {
  return fgemm_plan_ex(h, M, N, K, dtype, epi, FGEMM_ALGO_AUTO, 0, 0, algo_out, tile_m, tile_n,
                       predicted_us);
}

fgemm_status_t fgemm_plan_ex(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                             fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                             int32_t tile_m_in, int32_t tile_n_in, fgemm_algo_t* algo_out,
                             int32_t* tile_m, int32_t* tile_n, double* predicted_us) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (dtype != FGEMM_F16 && dtype != FGEMM_BF16)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "dtype must be FGEMM_F16 or FGEMM_BF16");
  if (algo < FGEMM_ALGO_AUTO || algo > FGEMM_ALGO_WINOGRAD1)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "unknown algorithm");
  const int32_t kind = epi ? epi->kind : FGEMM_EPI_NONE;
  Plan p;
  fgemm_status_t s = choose_plan(h, M, N, K, kind, algo, tile_m_in, tile_n_in, &p);
  if (s != FGEMM_OK) return s;
  if (algo_out) *algo_out = p.algo;
  if (tile_m) *tile_m = p.tile_m;
  if (tile_n) *tile_n = p.tile_n;
  if (predicted_us) *predicted_us = p.predicted_us;
  return FGEMM_OK;
}

fgemm_status_t fgemm_call_launches(fgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                   const fgemm_epilogue_t* epi, fgemm_algo_t algo, int32_t tile_m_in,
                                   int32_t tile_n_in, int32_t* launches) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (!launches) return set_msg(h, FGEMM_ERR_INVALID_ARG, "launches is NULL");
  if (algo < FGEMM_ALGO_AUTO || algo > FGEMM_ALGO_WINOGRAD1)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "unknown algorithm");
  const int32_t kind = epi ? epi->kind : FGEMM_EPI_NONE;
  const int64_t n_out = kind == FGEMM_EPI_SWIGLU ? N / 2 : N;
  if (M == 0 || n_out == 0) {
    *launches = 0;
    return FGEMM_OK;
  }
  if (K == 0) {
    *launches = 1;  // the bias / zero fill
    return FGEMM_OK;
  }
  Plan p;
  fgemm_status_t s = choose_plan(h, M, N, K, kind, algo, tile_m_in, tile_n_in, &p);
  if (s != FGEMM_OK) return s;
  *launches = 1;
  if (p.tile_m == 256 && depth_of(p.algo) == 2) {
    *launches = 2;  // the pre-pass, then the products
  } else if (p.tile_m == 256 && depth_of(p.algo) == 1) {
    const int sub_m = static_cast<int>(M / 2), sub_n = static_cast<int>(N / 2), sub_k = static_cast<int>(K / 2);
    const long long positions = fgemm_model_tiles(sub_m, sub_n, 256, p.tile_n);
    const int fit = fgemm::lcma_pair_clusters_fit(p.tile_n, 1);
    if (fit <= 0) return set_msg(h, FGEMM_ERR_CUDA, "cannot size the Strassen pair launch");
    const int clusters = static_cast<int>(fgemm_lcma_pair_clusters(positions, 1, fit));
    const StrassenTable& tab =
        p.algo == FGEMM_ALGO_WINOGRAD1 ? fgemm::winograd_table() : fgemm::strassen_table(1);
    // the pre-pass runs unless the product kernel forms both sides' sums
    if (lcma_formation_plan(h, tab, positions, clusters, sub_m, sub_k, nullptr) != 3) *launches = 2;
  }
  return FGEMM_OK;
}

namespace {

fgemm_status_t matmul_impl(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                           int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                           fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                           int32_t tile_m, int32_t tile_n, const fgemm_rms_t* rms) {
  fgemm_status_t s =
      validate(M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, tile_m, tile_n, &h->msg);
  if (s != FGEMM_OK) return s;
  const bool with_rms = rms && (rms->sumsq_out || rms->sumsq_in);
  const int32_t kind = epi ? epi->kind : FGEMM_EPI_NONE;
  const int64_t n_out = kind == FGEMM_EPI_SWIGLU ? N / 2 : N;
  if (M == 0 || n_out == 0) return FGEMM_OK;

  KernelParams p;
  std::memset(&p, 0, sizeof(p));
  p.A = static_cast<const uint16_t*>(A);
  p.B = static_cast<const uint16_t*>(B);
  p.C = static_cast<uint16_t*>(C);
  p.bias = epi ? static_cast<const uint16_t*>(epi->bias) : nullptr;
  p.err = h->d_err;
  p.lda = lda;
  p.ldb = ldb;
  p.ldc = ldc;
  p.spin_ns = h->spin_ns;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.n_out = static_cast<int>(n_out);
  p.epi = kind;
  p.is_bf16 = dtype == FGEMM_BF16 ? 1 : 0;
  p.alpha = epi ? epi->alpha : 1.0f;
  if (with_rms) {
    p.sumsq_out = rms->sumsq_out;
    p.sumsq_in = rms->sumsq_in;
    p.sumsq_parts = rms->sumsq_in ? rms->sumsq_parts : 0;
    p.rms_inv_n = rms->sumsq_in ? static_cast<float>(1.0 / static_cast<double>(rms->norm_width)) : 0.0f;
    p.rms_eps = rms->eps;
  }

  if (K == 0) {
    if (with_rms) return set_msg(h, FGEMM_ERR_UNSUPPORTED, "RMSNorm statistics need K >= 1");
    cudaError_t e = fgemm::launch_k0_fill(p, h->stream);
    return e == cudaSuccess ? FGEMM_OK : cuda_fail(h, e, "K == 0 fill launch");
  }

  Plan plan;
  s = choose_plan(h, M, N, K, kind, with_rms ? FGEMM_ALGO_CLASSICAL : algo, tile_m, tile_n, &plan,
                  with_rms);
  if (s != FGEMM_OK) return s;
  const int d = depth_of(plan.algo);
  const int bn = plan.tile_n;
  const int bm = plan.tile_m;  // 256: CTA pair; 16, 32, 64: the small-M kernel
  if (bm < fgemm::kBM) return launch_small_m(h, p, M, N, K, A, lda, B, ldb, bm);

  p.sub_m = static_cast<int>(M >> d);
  p.sub_n = static_cast<int>(N >> d);
  p.sub_k = static_cast<int>(K >> d);
  p.tiles_m = static_cast<int>((p.sub_m + bm - 1) / bm);
  if (d == 0 && kind == FGEMM_EPI_SWIGLU)
    p.tiles_n = static_cast<int>((n_out + bn / 2 - 1) / (bn / 2));
  else
    p.tiles_n = (p.sub_n + bn - 1) / bn;
  const long long units = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (units > (1ll << 31) - 1) return set_msg(h, FGEMM_ERR_UNSUPPORTED, "too many tiles");
  p.num_units = static_cast<int>(units);
  p.k_blocks = (p.sub_k + fgemm::kBK - 1) / fgemm::kBK;
  p.raster_group = 8;
  const uint32_t fmt = p.is_bf16 ? 1u : 0u;
  // tcgen05 instruction descriptor: fp32 accumulator, A/B fp16 (0) or bf16
  // (1), A K-major, B MN-major, N >> 3, M >> 4 (M = 256 on a CTA pair)
  p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 16) |
            (static_cast<uint32_t>(bn >> 3) << 17) | (static_cast<uint32_t>(bm >> 4) << 24);
  p.num_products = d == 0 ? 1 : (d == 1 ? 7 : 49);
  const bool wino = plan.algo == FGEMM_ALGO_WINOGRAD1;
  const StrassenTable& tab = wino ? fgemm::winograd_table() : fgemm::strassen_table(d);

  s = encode_tmap(h, &p.tmap_a, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                  static_cast<uint64_t>(lda), fgemm::kBM, p.is_bf16);
  if (s != FGEMM_OK) return s;
  s = encode_tmap(h, &p.tmap_b, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                  static_cast<uint64_t>(ldb), fgemm::kBK, p.is_bf16);
  if (s != FGEMM_OK) return s;

  if (bm == 256 && d >= 1) return launch_lcma(h, p, tab, d, bn, A, lda, B, ldb);
  if (bm == 256) {
    const int fit = fgemm::gemm_pair_clusters_fit(bn);
    if (fit <= 0) return set_msg(h, FGEMM_ERR_CUDA, "cannot size the CTA-pair launch");
    // C leaves this kernel by TMA stores of 32 x 32 boxes
    s = encode_tmap(h, &p.tmap_c, C, static_cast<uint64_t>(p.n_out), static_cast<uint64_t>(M),
                    static_cast<uint64_t>(ldc), 32, p.is_bf16, 32);
    if (s != FGEMM_OK) return s;
    int32_t pieces = 1;
    const int split = with_rms ? 0
                               : fgemm_model_split_tail(&h->model, units, fit, p.k_blocks, bn,
                                                        h->split_mode, &pieces);
    int clusters = static_cast<int>(std::min<long long>(fit, units));
    if (split > 0) {
      clusters = fit;  // the schedule is planned for every pair that fits
      s = prepare_split(h, &p, split, pieces, bn);
      if (s != FGEMM_OK) return s;
    }
    cudaError_t e = fgemm::launch_gemm_pair(bn, p, clusters, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "GEMM pair kernel launch");
    return FGEMM_OK;
  }
  const int grid = static_cast<int>(std::min<long long>(units, h->num_sms));
  if (d > 0) {
    const size_t per_cta = (size_t{1} << (2 * d)) * fgemm::kBM * static_cast<size_t>(bn) * sizeof(float);
    s = ensure_workspace(h, per_cta * static_cast<size_t>(grid));
    if (s != FGEMM_OK) return s;
    p.workspace = h->workspace;
  }
  cudaError_t e = wino ? fgemm::launch_gemm_winograd1(bn, p, tab, grid, h->stream)
                       : fgemm::launch_gemm(bn, d, p, &tab, grid, h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "GEMM kernel launch");
  return FGEMM_OK;
}

}  // namespace

fgemm_status_t fgemm_matmul_ex(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                               int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                               fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                               int32_t tile_m, int32_t tile_n) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  return matmul_impl(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, tile_m, tile_n, nullptr);
}

// Byte span [lo, hi) of a rows x cols matrix of 2-byte elements with row
// pitch ld elements at p (empty when p is null or the matrix is).
static void host_span(const void* p, int64_t rows, int64_t cols, int64_t ld, uintptr_t& lo, uintptr_t& hi) {
  lo = hi = 0;
  if (!p || rows <= 0 || cols <= 0) return;
  lo = reinterpret_cast<uintptr_t>(p);
  hi = lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * 2);
}

// C = epi(alpha A B + bias) with A, B, C and the bias in host memory.  B (and
// the bias) go up first into one of two device slots; A is cut into row
// blocks that go up on the upload stream while earlier blocks are multiplied
// on the handle's stream and their C blocks come down on the download
// stream, two slots each of A and C.  Every slot is reused only after the
// event that marks its last reader or writer done.  Everything is ordered on
// the handle's stream when the call returns.  With FGEMM_HOST_OVERLAP the
// uploads start without waiting for earlier work on the handle's stream
// (only for the slots they reuse, and for the earlier calls whose C they
// read), so they run under the previous call's products.
fgemm_status_t fgemm_matmul_host_ex(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                                    int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                                    fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                                    int32_t tile_m, int32_t tile_n, int32_t flags) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (dtype != FGEMM_F16 && dtype != FGEMM_BF16)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "dtype must be FGEMM_F16 or FGEMM_BF16");
  if (flags & ~FGEMM_HOST_OVERLAP) return set_msg(h, FGEMM_ERR_INVALID_ARG, "unknown flags");
  if (M < 0 || N < 0 || K < 0) return set_msg(h, FGEMM_ERR_INVALID_ARG, "negative size");
  const int32_t kind = epi ? epi->kind : FGEMM_EPI_NONE;
  const int64_t n_out = kind == FGEMM_EPI_SWIGLU ? N / 2 : N;
  if (M == 0 || n_out == 0) return FGEMM_OK;
  if ((K > 0 && (!A || !B)) || !C) return set_msg(h, FGEMM_ERR_INVALID_ARG, "NULL host matrix");
  if ((K > 0 && (lda < K || ldb < N)) || ldc < n_out)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "leading dimension smaller than the row");
  // row blocks: at least ~6 waves of 256 x 256 pair tiles each, at most 8
  // blocks, a multiple of 512 rows that divides M (so every block takes the
  // same form); otherwise one block
  int64_t mb = M;
  const int64_t min_rows = std::max<int64_t>(512, (6 * 76 * 65536 + N - 1) / std::max<int64_t>(N, 1));
  for (int nb = 8; nb >= 2; --nb) {
    if (M % nb != 0) continue;
    const int64_t r = M / nb;
    if (r % 512 == 0 && r >= min_rows) {
      mb = r;
      break;
    }
  }
  const int64_t nblocks = M / mb;
  const size_t esz = 2;
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  // device row pitches: multiples of 8 elements (16 bytes), as the kernels need
  const int64_t pk = (std::max<int64_t>(K, 1) + 7) / 8 * 8, pn = (N + 7) / 8 * 8, po = (n_out + 7) / 8 * 8;
  const size_t b_bytes = al(static_cast<size_t>(K) * pn * esz) + al(static_cast<size_t>(N) * esz);
  const size_t a_bytes = al(static_cast<size_t>(mb) * pk * esz), c_bytes = al(static_cast<size_t>(mb) * po * esz);
  // The slots keep fixed places (their capacities) from call to call, since
  // earlier calls may still be using theirs; they grow, after everything in
  // flight is done, only when a call needs more.
  cudaError_t e = cudaSuccess;
  if (!h->host_buf || b_bytes > h->host_cap_b || a_bytes > h->host_cap_a || c_bytes > h->host_cap_c) {
    e = cudaStreamSynchronize(h->stream);
    for (cudaStream_t st : {h->up, h->down})
      if (e == cudaSuccess && st) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
    if (h->host_buf) cudaFree(h->host_buf);
    h->host_buf = nullptr;
    h->host_cap_b = std::max(h->host_cap_b, b_bytes);
    h->host_cap_a = std::max(h->host_cap_a, a_bytes);
    h->host_cap_c = std::max(h->host_cap_c, c_bytes);
    e = cudaMalloc(&h->host_buf, 2 * (h->host_cap_b + h->host_cap_a + h->host_cap_c));
    if (e != cudaSuccess) {
      h->host_buf = nullptr;
      h->host_cap_b = h->host_cap_a = h->host_cap_c = 0;
      return cuda_fail(h, e, "cudaMalloc(host-call buffers)");
    }
  }
  if (!h->up) {
    e = cudaStreamCreateWithFlags(&h->up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->down, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&h->ev_start, &h->ev_b, &h->ev_a[0], &h->ev_a[1], &h->ev_c[0], &h->ev_c[1],
                            &h->ev_d[0], &h->ev_d[1], &h->ev_bfree[0], &h->ev_bfree[1], &h->ev_done[0],
                            &h->ev_done[1]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(h, e, "creating the host-call streams and events");
  }
  const int bs = static_cast<int>(h->host_calls & 1u);  // this call's B slot
  uint8_t* base = static_cast<uint8_t*>(h->host_buf);
  const size_t cb = h->host_cap_b, ca = h->host_cap_a, cc = h->host_cap_c;
  uint8_t* dB = base + bs * cb;
  uint8_t* dbias = dB + al(static_cast<size_t>(K) * pn * esz);
  uint8_t* dA[2] = {base + 2 * cb, base + 2 * cb + ca};
  uint8_t* dC[2] = {base + 2 * cb + 2 * ca, base + 2 * cb + 2 * ca + cc};
  fgemm_epilogue_t dev_epi{kind, epi ? epi->alpha : 1.0f, nullptr};
  if (!(flags & FGEMM_HOST_OVERLAP)) {
    // the uploads start after everything already on the handle's stream
    e = cudaEventRecord(h->ev_start, h->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->up, h->ev_start, 0);
  } else {
    // ... or only after the earlier calls (of the last two) whose C this
    // call's inputs overlap have written it
    uintptr_t lo[3], hi[3];
    host_span(A, M, K, lda, lo[0], hi[0]);
    host_span(B, K, N, ldb, lo[1], hi[1]);
    host_span(epi ? epi->bias : nullptr, 1, N, N, lo[2], hi[2]);
    for (int j = 0; j < 2 && e == cudaSuccess; ++j)
      for (int t = 0; t < 3; ++t)
        if (lo[t] < h->c_hi[j] && h->c_lo[j] < hi[t]) {
          e = cudaStreamWaitEvent(h->up, h->ev_done[j], 0);
          break;
        }
  }
  // B (and the bias) into this call's slot once the products of the call
  // that used the slot last are done
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->up, h->ev_bfree[bs], 0);
  if (e == cudaSuccess && K > 0)
    e = cudaMemcpy2DAsync(dB, static_cast<size_t>(pn) * esz, B, static_cast<size_t>(ldb) * esz,
                          static_cast<size_t>(N) * esz, static_cast<size_t>(K), cudaMemcpyHostToDevice, h->up);
  if (e == cudaSuccess && epi && epi->bias) {
    e = cudaMemcpyAsync(dbias, epi->bias, static_cast<size_t>(N) * esz, cudaMemcpyHostToDevice, h->up);
    dev_epi.bias = dbias;
  }
  if (e == cudaSuccess) e = cudaEventRecord(h->ev_b, h->up);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->stream, h->ev_b, 0);
  if (e != cudaSuccess) return cuda_fail(h, e, "host-call upload of B");
  for (int64_t i = 0; i < nblocks; ++i) {
    // the slots alternate over all blocks of the handle's calls: a block
    // uses the slot the previous block (of this or the last call) did not
    const int sl = static_cast<int>(h->host_blocks++ & 1u);
    const uint8_t* Ai = static_cast<const uint8_t*>(A) + static_cast<size_t>(i * mb) * lda * esz;
    uint8_t* Ci = static_cast<uint8_t*>(C) + static_cast<size_t>(i * mb) * ldc * esz;
    // A block i into its slot once the last product that read the slot is done
    e = cudaStreamWaitEvent(h->up, h->ev_c[sl], 0);
    if (e == cudaSuccess && K > 0)
      e = cudaMemcpy2DAsync(dA[sl], static_cast<size_t>(pk) * esz, Ai, static_cast<size_t>(lda) * esz,
                            static_cast<size_t>(K) * esz, static_cast<size_t>(mb), cudaMemcpyHostToDevice, h->up);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_a[sl], h->up);
    // the product, once A block i is up and the slot's last C block is down
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->stream, h->ev_a[sl], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->stream, h->ev_d[sl], 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "host-call upload of A");
    fgemm_status_t s = matmul_impl(h, mb, N, K, dA[sl], pk, dB, pn, dC[sl], po, dtype, &dev_epi, algo, tile_m,
                                   tile_n, nullptr);
    if (s != FGEMM_OK) return s;
    e = cudaEventRecord(h->ev_c[sl], h->stream);
    // C block i down
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->down, h->ev_c[sl], 0);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(Ci, static_cast<size_t>(ldc) * esz, dC[sl], static_cast<size_t>(po) * esz,
                            static_cast<size_t>(n_out) * esz, static_cast<size_t>(mb), cudaMemcpyDeviceToHost,
                            h->down);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_d[sl], h->down);
    if (e != cudaSuccess) return cuda_fail(h, e, "host-call download of C");
  }
  // B's slot is free once this call's products are done; C is written once
  // the last download is done, and the handle's stream ends there
  const int dj = static_cast<int>(h->host_calls & 1u);
  e = cudaEventRecord(h->ev_bfree[bs], h->stream);
  if (e == cudaSuccess) e = cudaEventRecord(h->ev_done[dj], h->down);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->stream, h->ev_done[dj], 0);
  if (e != cudaSuccess) return cuda_fail(h, e, "host-call completion events");
  host_span(C, M, n_out, ldc, h->c_lo[dj], h->c_hi[dj]);
  ++h->host_calls;
  return FGEMM_OK;
}

fgemm_status_t fgemm_matmul_host(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                                 int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                                 fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                                 int32_t tile_m, int32_t tile_n) {
  return fgemm_matmul_host_ex(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, tile_m, tile_n, 0);
}

fgemm_status_t fgemm_matmul_rms(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                                int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                                fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo,
                                int32_t tile_m, int32_t tile_n, const fgemm_rms_t* rms) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (rms && (rms->sumsq_out || rms->sumsq_in)) {
    if (algo != FGEMM_ALGO_AUTO && algo != FGEMM_ALGO_CLASSICAL)
      return set_msg(h, FGEMM_ERR_UNSUPPORTED, "RMSNorm statistics: classical form only");
    if (tile_m != 0 && tile_m != 128 && tile_m != 256)
      return set_msg(h, FGEMM_ERR_UNSUPPORTED, "RMSNorm statistics: tile_m 128 or 256 only");
    if ((reinterpret_cast<uintptr_t>(rms->sumsq_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(rms->sumsq_in) & 3u))
      return set_msg(h, FGEMM_ERR_ALIGNMENT, "sumsq buffers must be 4-byte aligned");
    if (rms->sumsq_in && (rms->sumsq_parts < 1 || rms->norm_width < 1 || !(rms->eps >= 0.0f) ||
                          !std::isfinite(rms->eps)))
      return set_msg(h, FGEMM_ERR_INVALID_ARG,
                     "sumsq_in needs sumsq_parts >= 1, norm_width >= 1 and a finite eps >= 0");
  }
  return matmul_impl(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, tile_m, tile_n, rms);
}

fgemm_status_t fgemm_mx_to_bf16(fgemm_handle_t h, int64_t rows, int64_t cols, const void* X,
                                int64_t ldx, const void* S, int64_t lds, int32_t format,
                                int32_t along, void* Y, int64_t ldy) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (format != FGEMM_FP8_E4M3 && format != FGEMM_FP8_E5M2)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "format must be FGEMM_FP8_E4M3 or FGEMM_FP8_E5M2");
  if (along != 0 && along != 1) return set_msg(h, FGEMM_ERR_INVALID_ARG, "along must be 0 or 1");
  if (rows < 0 || cols < 0) return set_msg(h, FGEMM_ERR_INVALID_ARG, "negative dimension");
  if (rows == 0 || cols == 0) return FGEMM_OK;
  if (cols > (int64_t{1} << 31) - 1) return set_msg(h, FGEMM_ERR_INVALID_ARG, "cols above 2^31 - 1");
  if (!X || !S || !Y) return set_msg(h, FGEMM_ERR_INVALID_ARG, "X, S and Y must not be NULL");
  const int64_t need_s = along == 0 ? (cols + 31) / 32 : cols;
  if (ldx < cols || ldy < cols || lds < need_s)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "ldx, ldy >= cols and lds >= the scales per row");
  if (reinterpret_cast<uintptr_t>(Y) & 1u) return set_msg(h, FGEMM_ERR_ALIGNMENT, "Y must be 2-byte aligned");
  const fgemm::MxJob job{static_cast<const uint8_t*>(X), ldx, static_cast<const uint8_t*>(S), lds, format,
                         along, rows, cols, static_cast<uint16_t*>(Y), ldy};
  cudaError_t e = fgemm::launch_mx_dequant(&job, 1, h->num_sms, h->stream);
  return e == cudaSuccess ? FGEMM_OK : cuda_fail(h, e, "MX to bf16 launch");
}

fgemm_status_t fgemm_matmul_mx(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                               int64_t lda, const void* scale_a, int64_t ld_sa, int32_t a_format,
                               const void* B, int64_t ldb, const void* scale_b, int64_t ld_sb,
                               int32_t b_format, void* C, int64_t ldc, const fgemm_epilogue_t* epi,
                               fgemm_algo_t algo, int32_t tile_m, int32_t tile_n) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if ((a_format != FGEMM_FP8_E4M3 && a_format != FGEMM_FP8_E5M2) ||
      (b_format != FGEMM_FP8_E4M3 && b_format != FGEMM_FP8_E5M2))
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "8-bit formats must be FGEMM_FP8_E4M3 or FGEMM_FP8_E5M2");
  if (M < 0 || N < 0 || K < 0) return set_msg(h, FGEMM_ERR_INVALID_ARG, "negative dimension");
  const int64_t kMax = (int64_t{1} << 31) - 1;
  if (M > kMax || N > kMax || K > kMax)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "dimension above 2^31 - 1");
  const int64_t kblocks = (K + 31) / 32;
  if (M > 0 && N > 0 && K > 0) {
    if (!A || !B || !scale_a || !scale_b)
      return set_msg(h, FGEMM_ERR_INVALID_ARG, "A, B and their scales must not be NULL");
    if (lda < K || ldb < N || ld_sa < kblocks || ld_sb < N)
      return set_msg(h, FGEMM_ERR_INVALID_ARG, "lda >= K, ldb >= N, ld_sa >= ceil(K/32), ld_sb >= N");
  }
  const int32_t kind = epi ? epi->kind : FGEMM_EPI_NONE;
  if (M == 0 || N == 0 || K == 0) {  // no 8-bit operand is read
    return matmul_impl(h, M, N, K, A, lda, B, ldb, C, ldc, FGEMM_BF16, epi, algo, tile_m, tile_n,
                       nullptr);
  }
  (void)kind;
  // bf16 copies, rows padded to 8 elements (16-byte rows for the copy engine)
  const int64_t kp = (K + 7) / 8 * 8, np = (N + 7) / 8 * 8;
  const size_t a_bytes = (static_cast<size_t>(M) * kp * 2 + 255) / 256 * 256;
  const size_t need = a_bytes + static_cast<size_t>(K) * np * 2;
  if (need > h->mx_bytes) {
    if (h->mx_buf) {
      cudaError_t e = cudaStreamSynchronize(h->stream);
      if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
      cudaFree(h->mx_buf);
      h->mx_buf = nullptr;
      h->mx_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&h->mx_buf, need);
    if (e != cudaSuccess) {
      h->mx_buf = nullptr;
      return cuda_fail(h, e, "cudaMalloc(MX bf16 values)");
    }
    h->mx_bytes = need;
  }
  uint16_t* Ab = static_cast<uint16_t*>(h->mx_buf);
  uint16_t* Bb = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(h->mx_buf) + a_bytes);
  const fgemm::MxJob jobs[2] = {
      {static_cast<const uint8_t*>(A), lda, static_cast<const uint8_t*>(scale_a), ld_sa, a_format, 0, M, K, Ab,
       kp},
      {static_cast<const uint8_t*>(B), ldb, static_cast<const uint8_t*>(scale_b), ld_sb, b_format, 1, K, N, Bb,
       np}};
  cudaError_t e = fgemm::launch_mx_dequant(jobs, 2, h->num_sms, h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "MX to bf16 launch");
  return matmul_impl(h, M, N, K, Ab, kp, Bb, np, C, ldc, FGEMM_BF16, epi, algo, tile_m, tile_n,
                     nullptr);
}

fgemm_status_t fgemm_matmul(fgemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                            int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                            fgemm_dtype_t dtype, const fgemm_epilogue_t* epi, fgemm_algo_t algo) {
  return fgemm_matmul_ex(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, epi, algo, 0, 0);
}

fgemm_status_t fgemm_selftest_wait_timeout(fgemm_handle_t h, int32_t limit_ms) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (limit_ms < 1 || limit_ms > 10000)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "limit_ms must be in 1..10000");
  KernelParams p;
  std::memset(&p, 0, sizeof(p));
  p.err = h->d_err;
  p.spin_ns = static_cast<unsigned long long>(limit_ms) * 1000000ull;
  cudaError_t e = fgemm::launch_selftest_wait(p, h->stream);
  return e == cudaSuccess ? FGEMM_OK : cuda_fail(h, e, "self-test launch");
}

fgemm_status_t fgemm_get_error(fgemm_handle_t h) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  unsigned int word = 0;
  e = cudaMemcpy(&word, h->d_err, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemcpy(error word)");
  if (word == 0) return FGEMM_OK;
  cudaMemset(h->d_err, 0, sizeof(unsigned int));
  static const char* roles[] = {"producer", "mma", "epilogue", "operand-sum"};
  const unsigned role = (word >> 24) & 0xF;
  char text[160];
  std::snprintf(text, sizeof(text), "a bounded wait ran out in the %s role of block %u (word 0x%08x)",
                role < 4 ? roles[role] : "?", word & 0xFFFFFFu, word);
  return set_msg(h, FGEMM_ERR_TIMEOUT, text);
}

}  // extern "C"

// ------------------------------------------------------------- calibration

namespace {

__global__ void fill_pattern_kernel(uint16_t* x, long long n, uint32_t seed, int is_bf16) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint32_t v = static_cast<uint32_t>(i) * 2654435761u ^ seed;
    v ^= v >> 15;
    v *= 2246822519u;
    v ^= v >> 13;
    const float f = (static_cast<float>(v & 0xFFFF) / 32768.0f) - 1.0f;  // [-1, 1)
    x[i] = is_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f)) : __half_as_ushort(__float2half_rn(f));
  }
}

}  // namespace

extern "C" fgemm_status_t fgemm_calibrate(fgemm_handle_t h, const char* json_out_path) {
  return fgemm_calibrate_ex(h, 8192, json_out_path);
}

extern "C" fgemm_status_t fgemm_calibrate_ex(fgemm_handle_t h, int64_t n, const char* json_out_path) {
  if (!h) return set_msg(nullptr, FGEMM_ERR_INVALID_ARG, "handle is NULL");
  if (n < 1024 || n > 16384 || n % 1024 != 0)
    return set_msg(h, FGEMM_ERR_INVALID_ARG, "calibration size must be a multiple of 1024 in [1024, 16384]");
  uint16_t *A = nullptr, *B = nullptr, *C = nullptr, *Xa = nullptr, *Xb = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  fgemm_status_t status = FGEMM_OK;
  fgemm_device_model_t m = h->model;
  const size_t elems = static_cast<size_t>(n) * n;
  const size_t copy_bytes = size_t{1} << 30;
  auto check = [&](cudaError_t e, const char* what) {
    if (e != cudaSuccess && status == FGEMM_OK) status = cuda_fail(h, e, what);
    return e == cudaSuccess;
  };
  auto time_gemm = [&](int64_t M, int64_t N, int64_t K, fgemm_algo_t algo, int32_t tm, int32_t tile,
                       double* us) {
    const int reps = 3;
    for (int r = 0; r < reps + 1; ++r) {
      if (r == 1) check(cudaEventRecord(e0, h->stream), "cudaEventRecord");
      fgemm_status_t s =
          fgemm_matmul_ex(h, M, N, K, A, K, B, N, C, N, FGEMM_BF16, nullptr, algo, tm, tile);
      if (s != FGEMM_OK) {
        if (status == FGEMM_OK) status = s;
        return false;
      }
    }
    check(cudaEventRecord(e1, h->stream), "cudaEventRecord");
    if (!check(cudaEventSynchronize(e1), "cudaEventSynchronize")) return false;
    float ms = 0;
    check(cudaEventElapsedTime(&ms, e0, e1), "cudaEventElapsedTime");
    *us = ms * 1e3 / reps;
    return status == FGEMM_OK;
  };
  do {
    if (!check(cudaMalloc(&A, elems * 2), "cudaMalloc")) break;
    if (!check(cudaMalloc(&B, elems * 2), "cudaMalloc")) break;
    if (!check(cudaMalloc(&C, elems * 2), "cudaMalloc")) break;
    if (!check(cudaMalloc(&Xa, copy_bytes), "cudaMalloc")) break;
    if (!check(cudaMalloc(&Xb, copy_bytes), "cudaMalloc")) break;
    check(cudaEventCreate(&e0), "cudaEventCreate");
    check(cudaEventCreate(&e1), "cudaEventCreate");
    fill_pattern_kernel<<<1024, 256, 0, h->stream>>>(A, static_cast<long long>(elems), 1u, 1);
    fill_pattern_kernel<<<1024, 256, 0, h->stream>>>(B, static_cast<long long>(elems), 2u, 1);
    if (!check(cudaGetLastError(), "fill launch")) break;
    const double flops = 2.0 * n * n * n;
    const int32_t tiles[3] = {64, 128, 256};
    for (int i = 0; i < 3 && status == FGEMM_OK; ++i) {
      double us = 0;
      if (!time_gemm(n, n, n, FGEMM_ALGO_CLASSICAL, 128, tiles[i], &us)) break;
      m.eff_classical[i] = flops / (us * 1e6) / m.peak_tflops;
    }
    const int saved_split = h->split_mode;
    h->split_mode = 0;  // mainloop efficiencies are taken on whole waves
    double pair256_us = 0;
    for (int i = 0; i < 2 && status == FGEMM_OK; ++i) {
      double us = 0;
      if (!time_gemm(n, n, n, FGEMM_ALGO_CLASSICAL, 256, tiles[i + 1], &us)) break;
      m.eff_pair[i] = flops / (us * 1e6) / m.peak_tflops;
      if (i == 1) pair256_us = us;
    }
    if (status == FGEMM_OK) {
      // split_fix_us: the split form's time against whole waves, less the
      // idle share of the last wave it removes
      h->split_mode = 2;
      double us = 0;
      const int fit = fgemm::gemm_pair_clusters_fit(256);
      const int64_t pair_tiles = (n / 256) * (n / 256);
      int32_t pieces = 1;
      const int split =
          fgemm_model_split_tail(nullptr, pair_tiles, fit, static_cast<int32_t>(n / 64), 256, 2, &pieces);
      if (split > 0 && time_gemm(n, n, n, FGEMM_ALGO_CLASSICAL, 256, 256, &us)) {
        // whole waves: W + 1 tile times; split: W + 1/S tile times + (S-1) * fix
        const int64_t waves = (pair_tiles + fit - 1) / fit;
        const double t_tile = pair256_us / static_cast<double>(waves);
        const double saved = (1.0 - 1.0 / pieces) * t_tile;
        m.split_fix_us = std::min(50.0, std::max(0.5, (us - pair256_us + saved) / (pieces - 1)));
      }
    }
    h->split_mode = saved_split;
    for (int d = 1; d <= 2 && status == FGEMM_OK; ++d) {
      for (int i = 0; i < 2 && status == FGEMM_OK; ++i) {
        double us = 0;
        if (!time_gemm(n, n, n, d == 1 ? FGEMM_ALGO_STRASSEN1 : FGEMM_ALGO_STRASSEN2, 128,
                       i == 0 ? 128 : 256, &us))
          break;
        const double executed = flops * std::pow(7.0 / 8.0, d);
        m.eff_strassen[d - 1][i] = executed / (us * 1e6) / m.peak_tflops;
      }
    }
    for (int d = 1; d <= 2 && status == FGEMM_OK; ++d) {
      for (int i = 0; i < 2 && status == FGEMM_OK; ++i) {
        // one or two levels on CTA pairs: a pre-pass plus the product
        // kernel, so the product kernel's rate is the one under which the
        // model predicts the measured time (found by bisection; the
        // prediction falls as it rises)
        const fgemm_algo_t a = d == 1 ? FGEMM_ALGO_STRASSEN1 : FGEMM_ALGO_STRASSEN2;
        const int32_t tn = i == 0 ? 128 : 256;
        if (!fgemm::form_is_legal(n, n, n, FGEMM_EPI_NONE, a, 256, tn)) continue;
        double us = 0;
        if (!time_gemm(n, n, n, a, 256, tn, &us)) break;
        double* eff = d == 1 ? &m.eff_strassen_pair[i] : &m.eff_strassen2_pair[i];
        double lo = 1e-3, hi = 4.0;
        for (int it = 0; it < 60; ++it) {
          const double mid = 0.5 * (lo + hi);
          *eff = mid;
          double pred = 0;
          fgemm_model_predict(&m, n, n, n, FGEMM_EPI_NONE, a, 256, tn, &pred);
          if (pred > us)
            lo = mid;
          else
            hi = mid;
        }
        *eff = 0.5 * (lo + hi);
      }
    }
    for (int i = 0; i < 2 && status == FGEMM_OK; ++i) {
      double us = 0;
      if (!time_gemm(n, n, n, FGEMM_ALGO_WINOGRAD1, 128, i == 0 ? 128 : 256, &us)) break;
      m.eff_winograd[i] = flops * 7.0 / 8.0 / (us * 1e6) / m.peak_tflops;
    }
    if (status != FGEMM_OK) break;
    {  // launch cost: back-to-back K = 0 products (one trivial kernel each)
      double us = 0;
      if (!time_gemm(128, 128, 0, FGEMM_ALGO_AUTO, 0, 0, &us)) break;
      m.launch_us = std::max(0.5, us);
      // pipeline fill and drain: one 128 x 128 tile at two K lengths, the
      // intercept of its time in K less the launch
      double t1 = 0, t2 = 0;
      if (!time_gemm(128, 128, 1024, FGEMM_ALGO_CLASSICAL, 128, 128, &t1)) break;
      if (!time_gemm(128, 128, 4096, FGEMM_ALGO_CLASSICAL, 128, 128, &t2)) break;
      const double intercept = t1 - (t2 - t1) / 3.0;
      m.tile_fill_us = std::max(0.5, intercept - m.launch_us);
    }
    {  // streaming bandwidth: device-to-device copy, read + write bytes
      check(cudaMemcpyAsync(Xb, Xa, copy_bytes, cudaMemcpyDeviceToDevice, h->stream), "copy");
      check(cudaEventRecord(e0, h->stream), "cudaEventRecord");
      for (int r = 0; r < 3; ++r)
        check(cudaMemcpyAsync(Xb, Xa, copy_bytes, cudaMemcpyDeviceToDevice, h->stream), "copy");
      check(cudaEventRecord(e1, h->stream), "cudaEventRecord");
      if (!check(cudaEventSynchronize(e1), "cudaEventSynchronize")) break;
      float ms = 0;
      check(cudaEventElapsedTime(&ms, e0, e1), "cudaEventElapsedTime");
      if (ms > 0) m.hbm_gbs = 3.0 * 2.0 * copy_bytes / (ms * 1e-3) / 1e9;
    }
  } while (false);
  cudaStreamSynchronize(h->stream);
  if (A) cudaFree(A);
  if (B) cudaFree(B);
  if (C) cudaFree(C);
  if (Xa) cudaFree(Xa);
  if (Xb) cudaFree(Xb);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (status != FGEMM_OK) return status;
  h->model = m;
  h->plans.clear();
  if (json_out_path && fgemm_model_save_json(&m, json_out_path) != FGEMM_OK)
    return set_msg(h, FGEMM_ERR_CALIBRATION, std::string("cannot write ") + json_out_path);
  return FGEMM_OK;
}
