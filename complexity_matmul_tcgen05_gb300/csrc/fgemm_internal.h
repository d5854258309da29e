// fgemm_internal.h -- definitions shared by the host API and the kernel
// translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fgemm {

constexpr int kBM = 128;          // output tile rows (tcgen05 M = 128, one CTA)
constexpr int kBK = 64;           // K per pipeline stage = one 128-byte swizzle row
constexpr int kMaxDepth = 2;      // Strassen recursion levels supported
constexpr int kMaxProducts = 49;  // 7^2
constexpr int kMaxTerms = 4;      // 2^depth source blocks per formed operand
constexpr int kMaxSplitPieces = 4;  // K pieces per split tile (each last piece reads S - 1)

// Term codes in the Strassen tables: bits [0,5) block index
// (row_block << depth | col_block) in the 2^depth x 2^depth block grid,
// bit 5 = last contribution to that output block (product kernel on CTA
// pairs only), bit 6 = first contribution, bit 7 = negative sign.
constexpr uint8_t kTermIndexMask = 0x1F;
constexpr uint8_t kTermLast = 0x20;
constexpr uint8_t kTermFirst = 0x40;
constexpr uint8_t kTermNeg = 0x80;

// Product p multiplies (sum of a-terms of A) by (sum of b-terms of B) and adds
// its result, with the c-terms' signs, into output blocks.  For depth 0 there
// is one product with one term of each kind.
struct StrassenTable {
  uint8_t na[kMaxProducts];
  uint8_t nb[kMaxProducts];
  uint8_t nc[kMaxProducts];
  uint8_t a[kMaxProducts][kMaxTerms];
  uint8_t b[kMaxProducts][kMaxTerms];
  uint8_t c[kMaxProducts][kMaxTerms];
};

enum EpiKind : int { kEpiNone = 0, kEpiScaleBias = 1, kEpiSilu = 2, kEpiSwiglu = 3 };

#ifdef __CUDACC__
#define FGEMM_HD __host__ __device__
#else
#define FGEMM_HD
#endif

// ---------------------------------------------------------------------------
// Work schedule of the persistent CTA-pair kernel, with the last partial
// wave split along K.
//
// With T output tiles on P clusters, R = T mod P tiles would run alone in a
// last, partly idle wave.  When 2R <= P, those R tiles (the FIRST R units in
// the rasterised order, so that they share row blocks of A with the first
// wave of whole tiles) are each cut into S = floor(P / R) pieces of equal K
// range; piece s of split tile t runs on cluster t * S + s, as that
// cluster's first work item.  Every cluster then runs its (T - R) / P whole
// tiles, units R + c, R + c + P, ...  The kernel takes W + 1/S tile times
// instead of W + 1.
//
// Every piece stores its fp32 partial tile; the piece that finishes last
// (per 32-row warp slice, decided by a counter) sums the pieces in piece
// order, so the result does not depend on which finished last, and applies
// the epilogue.  No CTA waits for another.  Its sum overlaps the MMAs of the
// cluster's first whole tile.
struct WorkItem {
  int unit;     // output tile (unit_coords order)
  int k0, k1;   // K blocks [k0, k1) of the tile
  int piece;    // index of this piece among the tile's pieces
  int npieces;  // 1 for a whole tile
};

// The n-th work item of `cluster` (false once its list is exhausted).
FGEMM_HD inline bool work_item(int num_units, int split_tiles, int split_pieces, int clusters,
                               int k_blocks, int cluster, int n, WorkItem& w) {
  const bool has_piece = split_tiles > 0 && cluster < split_tiles * split_pieces;
  if (has_piece && n == 0) {
    const int s = cluster % split_pieces;
    w.unit = cluster / split_pieces;
    w.k0 = static_cast<int>(static_cast<long long>(s) * k_blocks / split_pieces);
    w.k1 = static_cast<int>(static_cast<long long>(s + 1) * k_blocks / split_pieces);
    w.piece = s;
    w.npieces = split_pieces;
    return true;
  }
  const int i = n - (has_piece ? 1 : 0);
  const int whole = num_units - split_tiles;
  const int count = cluster < whole ? (whole - cluster + clusters - 1) / clusters : 0;
  if (i >= count) return false;
  w.unit = split_tiles + cluster + i * clusters;
  w.k0 = 0;
  w.k1 = k_blocks;
  w.piece = 0;
  w.npieces = 1;
  return true;
}

// How many work items `cluster` runs under the schedule of work_item.
FGEMM_HD inline int work_item_count(int num_units, int split_tiles, int split_pieces, int clusters,
                                    int cluster) {
  const bool has_piece = split_tiles > 0 && cluster < split_tiles * split_pieces;
  const int whole = num_units - split_tiles;
  const int count = cluster < whole ? (whole - cluster + clusters - 1) / clusters : 0;
  return count + (has_piece ? 1 : 0);
}

// ---------------------------------------------------------------------------
// Work schedule of the small-M kernel (stream-K).  Its tiles are 128 columns
// of C (all M <= 64 rows); the K blocks of all tiles, laid end to end tile
// after tile (tiles * k_blocks iterations), are cut into `ctas` contiguous
// shares of equal size (+-1), one per CTA.  A share meets each tile in one
// contiguous K range (a piece); the pieces of a tile run on consecutive CTAs
// and are numbered from 0 in K order.  As in the CTA-pair split, every piece
// of a tile with several pieces stores an fp32 partial and the last to finish
// sums them in piece order.

// The CTA whose share holds flat iteration x.
FGEMM_HD inline int stream_k_owner(long long x, long long total, int ctas) {
  return static_cast<int>(((x + 1) * ctas - 1) / total);
}

// The n-th work item of CTA `cta` (false once its share is exhausted).
FGEMM_HD inline bool stream_k_item(int tiles, int k_blocks, int ctas, int cta, int n, WorkItem& w) {
  const long long total = static_cast<long long>(tiles) * k_blocks;
  const long long lo = static_cast<long long>(cta) * total / ctas;
  const long long hi = static_cast<long long>(cta + 1) * total / ctas;
  if (hi <= lo) return false;
  const long long start = n == 0 ? lo : (lo / k_blocks + n) * k_blocks;
  if (start >= hi) return false;
  const long long t = start / k_blocks;
  const long long tile_lo = t * k_blocks;
  const long long end = hi < tile_lo + k_blocks ? hi : tile_lo + k_blocks;
  const int first = stream_k_owner(tile_lo, total, ctas);
  const int last = stream_k_owner(tile_lo + k_blocks - 1, total, ctas);
  w.unit = static_cast<int>(t);
  w.k0 = static_cast<int>(start - tile_lo);
  w.k1 = static_cast<int>(end - tile_lo);
  w.piece = cta - first;
  w.npieces = last - first + 1;
  return true;
}

// Partial slot of the piece of tile `unit` that runs on CTA c.  Only a
// CTA's first and last work items can be pieces of a shared tile (the items
// between are whole tiles), so each CTA owns two slots: 2c for its first item
// and 2c + 1 for its last.  A piece is its CTA's first item exactly when the
// CTA's share starts inside the tile.  The tile's arrival counters sit with
// the slot of its piece 0.
FGEMM_HD inline long long stream_k_slot(int tiles, int k_blocks, int ctas, int unit, int c) {
  const long long total = static_cast<long long>(tiles) * k_blocks;
  const long long tile_lo = static_cast<long long>(unit) * k_blocks;
  const long long lo = static_cast<long long>(c) * total / ctas;
  return static_cast<long long>(c) * 2 + (lo >= tile_lo ? 0 : 1);
}

struct KernelParams {
  CUtensorMap tmap_a;  // A: inner dim K, outer M, box {64, 128}, 128B swizzle
  CUtensorMap tmap_b;  // B: inner dim N, outer K, box {64, 64},  128B swizzle
  CUtensorMap tmap_c;  // C (CTA-pair classical kernel): inner n_out, outer M, box {32, 32}, 64B swizzle
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* C;
  const uint16_t* bias;   // N entries (virtual column index) or nullptr
  float* workspace;       // Strassen partial tiles, 4^depth * 128 * BN floats per CTA
  unsigned int* err;      // device error word (0 = ok)
  long long lda, ldb, ldc;
  unsigned long long spin_ns;  // bound of every mbarrier wait
  int M, N, K;            // virtual GEMM: A is M x K, B is K x N
  int n_out;              // columns of C (N, or N/2 for SwiGLU)
  int sub_m, sub_n, sub_k;  // block sizes of one product (M, N, K >> depth)
  int tiles_m, tiles_n;   // output tile grid of one product (256-row tiles on CTA pairs)
  int num_units;          // tiles_m * tiles_n
  int k_blocks;           // ceil(sub_k / 64)
  int epi;                // EpiKind
  int is_bf16;
  int raster_group;       // tile rows per rasterisation group
  uint32_t idesc;         // tcgen05 instruction descriptor
  float alpha;
  int num_products;
  // K split of the last partial wave (CTA-pair classical kernel only)
  int split_tiles;          // tiles split along K (0: none), units [0, split_tiles)
  int split_pieces;         // pieces per split tile (>= 2 when split_tiles > 0)
  unsigned int split_gen;   // launch generation tagging the counters, 1 .. 2^24 - 1
  unsigned int* split_ctr;  // per (split tile, CTA rank, epilogue warp): gen << 8 | arrivals
  float* split_ws;          // per (split tile, piece, CTA rank): 128 x BN fp32, [col/4][row][4]
  // RMSNorm statistics (classical one-CTA and CTA-pair kernels, no K split)
  float* sumsq_out;         // [ceil(n_out / 64)][M]: sums of squares of stored outputs, or null
  const float* sumsq_in;    // [sumsq_parts][M] from an earlier product, or null
  int sumsq_parts;
  float rms_inv_n;          // 1 / width of the normalised rows
  float rms_eps;
};

// The launch arguments of the Strassen / Winograd kernels: the common
// parameters and the scheme's table.  The classical kernels take
// KernelParams alone (a smaller parameter block is a cheaper launch).
struct StrassenParams {
  KernelParams k;
  StrassenTable tab;
};

// ---------------------------------------------------------------------------
// Low-complexity forms on CTA pairs with the summed operands streamed
// through HBM: a streaming pre-pass forms each summed operand of the scheme
// once (fp32 sum of the exact blocks, one rounding) into temporaries, then
// one persistent launch runs the block products on the classical pair
// mainloop and folds each product into the output blocks it feeds.

// Product p of a scheme as the product kernel reads it: its A operand is
// raw block a_idx of A (a_temp == 0) or temporary a_idx (a_temp == 1), the
// same for B; its accumulator is added, with the codes' signs, into output
// blocks c[0 .. nc) (codes as in StrassenTable, with kTermFirst / kTermLast
// marking the first and the last contribution to each block in product
// order).  fin: the output blocks (bit b) whose value is complete once this
// product is in, or for SwiGLU the block rows (bit r: gate block 2r, up
// block 2r + 1) complete with it.  Block indices as in StrassenTable: block
// (r, c) of the 2^depth x 2^depth split is r << depth | c.
struct LcmaProduct {
  uint8_t a_temp, a_idx, b_temp, b_idx;
  uint8_t nc;
  uint8_t c[kMaxTerms];
  uint16_t fin;
  uint16_t groups;  // output groups it feeds (bit g: block g, or for SwiGLU block row g)
};

// One matrix of the operand formation: the 4^depth `rows` x `cols` blocks
// of src (block q at block row q >> depth, block column q & (2^depth - 1))
// are combined into ntemp temporaries, temporary t = sum_q coef[t][q] *
// block_q (coef in {-1, 0, 1}), stored one after another, each rows x cols
// with pitch cols.
constexpr int kLcmaProducts = 49;   // up to two levels: 7^depth block products
constexpr int kLcmaMaxTemps = 49;   // summed operands per side (one level: Strassen 5, Winograd 4)
constexpr int kLcmaMaxBlocks = 16;  // 4^depth blocks of each matrix
struct LcmaFormJob {
  const uint16_t* src;
  long long ld;
  uint16_t* dst;
  int rows, cols;
  int ntemp;
  uint32_t block_mask;  // blocks some temporary reads
  int8_t coef[kLcmaMaxTemps][kLcmaMaxBlocks];
  // two levels: the temporary that holds product p's operand on this side
  // (-1: a raw block, read in place)
  int8_t leaf_temp[kLcmaProducts];
};

// One Strassen level's operand coefficients (side 0: A, 1: B) over the
// blocks 11, 12, 21, 22 (index i = r * 2 + c) for the products p = M1 .. M7: the two-level pre-pass forms
// product (p, q)'s operand on a side as the inner combination q of the outer
// combination p of the quarter blocks.  The host checks them against the
// scheme's two-level table before it uses that pre-pass.
FGEMM_HD constexpr int strassen_coef(int side, int p, int i) {
  constexpr int8_t a[7][4] = {{1, 0, 0, 1}, {0, 0, 1, 1}, {1, 0, 0, 0}, {0, 0, 0, 1},
                              {1, 1, 0, 0}, {-1, 0, 1, 0}, {0, 1, 0, -1}};
  constexpr int8_t b[7][4] = {{1, 0, 0, 1}, {1, 0, 0, 0}, {0, 1, 0, -1}, {-1, 0, 1, 0},
                              {0, 0, 0, 1}, {1, 1, 0, 0}, {0, 0, 1, 1}};
  return side == 0 ? a[p][i] : b[p][i];
}

struct LcmaFormParams {
  LcmaFormJob job[2];  // A and B
  int is_bf16;
};

// Rows of one matrix per formation task when the product kernel forms the
// temporaries itself.
constexpr int kFormRows = 8;
// The kernel forms them itself (automatic mode) when the scheme's leading
// products that read only blocks of A and B span at least this many waves.
constexpr long long kFusedMinWaves = 16;

struct LcmaParams {
  KernelParams k;        // tmap_a / tmap_b map A and B; k.workspace holds the partial tiles
  CUtensorMap tmap_ta;   // A temporaries: inner sub_k, outer ntemp_a * sub_m, box {64, 128}
  CUtensorMap tmap_tb;   // B temporaries: inner sub_n, outer ntemp_b * sub_k, box {64, 64}
  long long units;       // output positions * num_products (informational)
  LcmaProduct prod[kLcmaProducts];
  uint8_t group_pieces[kLcmaMaxBlocks];  // products feeding each output group
  int tail_at;              // whole-position products a pair runs before its tail units
  // Temporaries formed inside the product kernel (form_tasks[0] +
  // form_tasks[1] > 0; otherwise the pre-pass launch formed them): job j is
  // cut into form_tasks[j] bands of kFormRows rows, claimed through
  // form_ctr[0] by the CTAs' otherwise idle warps; form_ctr[1 + j] counts the
  // bands of job j that are stored.  A producer issues the first load of a
  // temporary of side j only once all of job j is stored.  The counters
  // start at zero (the host clears them before the launch).
  LcmaFormParams form;
  unsigned int* form_ctr;
  int form_tasks[2];
};

// Per-CTA partial tiles of the product kernel's whole positions: the 4^depth
// output blocks, 128 x bn fp32 each.
inline size_t lcma_slot_floats(int bn, int depth) {
  return (static_cast<size_t>(1) << (2 * depth)) * 128 * static_cast<size_t>(bn);
}

// The pre-pass over both jobs in one launch (depth 1 or 2).
cudaError_t launch_lcma_form(const LcmaFormParams& f, int depth, int num_sms, cudaStream_t stream);

// The product kernel for `depth` Strassen-like levels on `clusters` CTA pairs
// (bn = 128 or 256).  p.k.workspace holds 2 * clusters * W *
// lcma_slot_floats(bn, depth) partials (W = positions / clusters whole
// positions per pair); the T = positions mod clusters positions of the
// partial last wave run as 7^depth T separate product units, whose
// accumulators (128 x bn fp32 per unit and CTA) go to p.k.split_ws, with
// 4^depth x 2 x 4 counters per such position (output groups x CTAs x
// epilogue warps) in p.k.split_ctr tagged with p.k.split_gen.  Two levels
// take the operands from the pre-pass (no in-kernel formation) and no
// SwiGLU.
cudaError_t launch_lcma_pair(int bn, int depth, const LcmaParams& p, int clusters, cudaStream_t stream);

// How many clusters of the product kernel fit on the current device.
int lcma_pair_clusters_fit(int bn, int depth);

// Error word layout written by a kernel whose bounded wait ran out.
constexpr unsigned int kErrTimeout = 0x80000000u;
// bits [24,28): role (0 producer, 1 mma, 2 epilogue, 3 operand-sum), [0,24): block

size_t kernel_smem_bytes(int bn, int depth);
int kernel_threads(int depth);

// Launches the persistent GEMM kernel for tile width bn (64/128/256) and
// Strassen depth (0 = classical) with `grid` CTAs on `stream`; `tab` is the
// Strassen table of that depth (unused, may be null, for depth 0).
cudaError_t launch_gemm(int bn, int depth, const KernelParams& p, const StrassenTable* tab, int grid,
                        cudaStream_t stream);

// Small-M kernel: C (M <= mp rows, mp = 16, 32 or 64) computed as
// C^T = B^T A^T in tiles of 128 columns of C, K split over `grid` CTAs by
// stream_k_item.  p.tmap_a has a {64, mp} box; p.split_ws holds 2 * grid
// partial slots of 128 x mp fp32 and p.split_ctr 8 * grid counters tagged
// with p.split_gen.
cudaError_t launch_gemm_skinny(int mp, const KernelParams& p, int grid, cudaStream_t stream);

// A block-scaled 8-bit matrix X (rows x cols, fmt 0 E4M3, 1 E5M2) with E8M0
// scales S of blocks of 32 along rows (along 0) or down columns (along 1),
// and the bf16 matrix Y its values go to.
struct MxJob {
  const uint8_t* X;
  long long ldx;
  const uint8_t* S;
  long long lds;
  int fmt, along;
  long long rows, cols;
  uint16_t* Y;
  long long ldy;
};

// Converts one or two such matrices (njobs 1 or 2) in a single launch.
cudaError_t launch_mx_dequant(const MxJob* jobs, int njobs, int num_sms, cudaStream_t stream);

// One-level Winograd variant on the single-CTA kernel (bn = 128 or 256): the
// Strassen kernel with up to four source blocks per formed operand; `tab`
// must be the Winograd table.
cudaError_t launch_gemm_winograd1(int bn, const KernelParams& p, const StrassenTable& tab, int grid,
                                  cudaStream_t stream);

// Classical kernel on CTA pairs: 256 x bn tiles (bn = 128 or 256) on exactly
// `clusters` pairs, which must not exceed gemm_pair_clusters_fit(bn) and must
// equal the cluster count p's split schedule was planned for.
cudaError_t launch_gemm_pair(int bn, const KernelParams& p, int clusters, cudaStream_t stream);

// How many clusters of the classical pair kernel fit on the current device
// at once (0 on error).
int gemm_pair_clusters_fit(int bn);

// The Strassen coefficient table of `depth` levels (0: one trivial product).
const StrassenTable& strassen_table(int depth);

// The one-level Winograd-variant table (seven products, operands of up to
// four blocks, outputs fed by up to four products).
const StrassenTable& winograd_table();

// One block whose bounded wait on a never-completed mbarrier runs out.
cudaError_t launch_selftest_wait(const KernelParams& p, cudaStream_t stream);

// C[i][j] = epi(bias[j]) for K == 0 (the product is empty).
cudaError_t launch_k0_fill(const KernelParams& p, cudaStream_t stream);

}  // namespace fgemm
