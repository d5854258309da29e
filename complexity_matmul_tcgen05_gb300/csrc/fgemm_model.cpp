// fgemm_model.cpp -- the analytical decision model (host only).
//
// FalconGEMM summary, "Methodology" item 4: the runtime of each candidate
// algorithm is estimated from compute throughput, memory bandwidth and the
// extra cost that grows with the recursion depth, and the candidate with the
// smallest predicted time (with its tiling) is chosen; item 5: the choice is
// made at run time from the actual (M, N, K).  Candidates: classical, Strassen at one or
// two levels, and one level of Winograd's variant (single-CTA tiles).
//
// The estimate for one (form, tile_n) candidate:
//   tiles        = tile quantization of the output of one product:
//                  ceil(m/tile_m) * ceil(n/tile_n)  (CS336 Lecture 05 notes,
//                  "Page 43")
//   waves        = ceil(tiles / slots), slots = SMs (one tile per SM) or SM
//                  pairs (256-row tiles); a partial last wave costs a full one
//                  ("Page 48", wave quantization)
//   t_tile       = products * 2 * tile_m * tile_n * K_sub / (slot peak * eff),
//                  eff measured per form and tile
//   t_compute    = waves * t_tile + fill (the pipeline fill and the last
//                  tile's epilogue, once per launch: every other epilogue
//                  overlaps the next tile's MMAs); for the classical CTA-pair kernel whose
//                  last wave holds R <= slots / 2 tiles, those tiles may run
//                  as S = slots / R pieces of K each (S <= 4), and then
//                  t_compute = (floor(tiles / slots) + 1/S) * t_tile
//                  + (S - 1) * split_fix_us, when that is less
//   t_memory     = HBM bytes / (bandwidth * streaming efficiency * share of
//                  the SMs the launch keeps busy) (operands and result once,
//                  plus the Strassen partial tiles when they cannot stay in L2)
//   t_operands   = operand elements streamed from L2 into the SMs (tiled
//                  reads, "Page 42": tiles * (128 + tile_n) * K per source
//                  term) * 2 bytes / L2 bandwidth
//   t            = max(t_compute, t_memory, t_operands) + launch ("Page 21",
//                  the roofline: time is the largest of compute and traffic)
#include <algorithm>
#include <numeric>
#include <utility>
#include <vector>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "../../include/fgemm.h"
#include "fgemm_internal.h"

namespace {

int depth_of(fgemm_algo_t a) {
  return (a == FGEMM_ALGO_STRASSEN1 || a == FGEMM_ALGO_WINOGRAD1) ? 1
                                                                 : (a == FGEMM_ALGO_STRASSEN2 ? 2 : 0);
}

int tile_index(int tile_n) { return tile_n == 64 ? 0 : (tile_n == 128 ? 1 : 2); }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

namespace fgemm {

// Shared with the API's validation: is (algo, tile_m x tile_n) legal?
bool form_is_legal(int64_t M, int64_t N, int64_t K, int32_t epi_kind, fgemm_algo_t algo,
                   int32_t tile_m, int32_t tile_n) {
  if (tile_n != 64 && tile_n != 128 && tile_n != 256) return false;
  if (tile_m == 16 || tile_m == 32 || tile_m == 64)  // the small-M kernel
    return algo == FGEMM_ALGO_CLASSICAL && tile_n == 128 && epi_kind != FGEMM_EPI_SWIGLU &&
           M <= tile_m;
  if (tile_m != 128 && tile_m != 256) return false;
  if (epi_kind == FGEMM_EPI_SWIGLU && tile_n == 64) return false;
  const int d = depth_of(algo);
  if (tile_m == 256 && tile_n < 128) return false;
  if (tile_m == 256 && d == 2 && epi_kind == FGEMM_EPI_SWIGLU) return false;
  // (two levels on pairs: the leaf-operand pre-pass runs a block of 8 rows
  // per grid row, at most 65535 of them)
  if (tile_m == 256 && d == 2 && (M / 4 > 8 * 65535 || K / 4 > 8 * 65535)) return false;
  if (d == 0) return true;
  if (tile_n == 64) return false;
  const int64_t g = int64_t{1} << d;
  if (M <= 0 || N <= 0 || K <= 0) return false;
  return M % (g * tile_m) == 0 && N % (g * tile_n) == 0 && K % (g * kBK) == 0;
}

}  // namespace fgemm

extern "C" {

void fgemm_model_default(fgemm_device_model_t* out, int32_t num_sms, double peak_tflops,
                         double hbm_gbs) {
  if (!out) return;
  fgemm_device_model_t m{};
  m.num_sms = num_sms > 0 ? num_sms : 1;
  // The denominators: a GB300's measured dense bf16 GEMM rate (cuBLAS,
  // 8192^3, burst) and its measured streaming copy bandwidth, unless the
  // caller gives others.
  m.peak_tflops = peak_tflops > 0 ? peak_tflops : 1891.3 * m.num_sms / 152.0;
  m.hbm_gbs = hbm_gbs > 0 ? hbm_gbs : 6789.0;
  // Mainloop rates measured on GB300 by fgemm_calibrate (8192^3 bf16, every
  // form and tile), in TFLOP/s for 152 SMs; each efficiency is that rate as a
  // fraction of the peak above, so the model predicts the measured rates
  // whatever denominator it is given.  fgemm_calibrate re-measures them on
  // the device at hand.
  const double sm_scale = m.num_sms / 152.0;
  auto rate = [&](double tflops_152) { return tflops_152 * sm_scale / m.peak_tflops; };
  m.eff_classical[0] = rate(578.3);   // 128 x 64
  m.eff_classical[1] = rate(1127.3);  // 128 x 128
  m.eff_classical[2] = rate(1575.0);  // 128 x 256
  m.eff_pair[0] = rate(1122.8);       // 256 x 128
  m.eff_pair[1] = rate(1912.5);       // 256 x 256
  // Strassen on one-CTA tiles (operand sums formed on chip from registers):
  // executed-MAC rates
  m.eff_strassen[0][0] = rate(162.0);
  m.eff_strassen[0][1] = rate(184.5);
  m.eff_strassen[1][0] = rate(76.5);
  m.eff_strassen[1][1] = rate(105.8);
  // one level on CTA pairs, summed operands streamed through HBM: the rate
  // of its product kernel (executed MACs) under which the model predicts the
  // measured times (16384^3: 5.34 ms at 256 x 256 and 7.5 ms at 256 x 128,
  // against 4.80 ms classical, sustained clocks, scaled to the classical
  // rate above)
  m.eff_strassen_pair[0] = rate(1121.0);  // 256 x 128
  m.eff_strassen_pair[1] = rate(1720.0);  // 256 x 256: the product kernel at 16384^3, 4.51 ms at full clocks
  // two levels on CTA pairs: the same product kernel (its MMAs at the
  // one-level rate), each unit's fold into about three of the 16 output
  // blocks about 30 us at 256 columns (fitted to 4096 x 19456 x {4096,
  // 16384}, 16384^3 and 32768^3: 33, 45, 48 and 64 us per unit)
  m.eff_strassen2_pair[0] = rate(1121.0);  // 256 x 128
  m.eff_strassen2_pair[1] = rate(1720.0);  // 256 x 256
  m.fold2_unit_us = 30.0;
  // launch: back-to-back calls of a one-kernel product; fill: the first
  // MMA about 1.5 us after the start, the last 256 x 256 tile's epilogue
  // about 5 us after the last MMA (timestamps of an instrumented build)
  m.launch_us = 4.0;
  m.tile_fill_us = 6.5;
  m.l2_bytes = 126.0 * 1024 * 1024;
  m.l2_gbs = 40000.0;
  m.split_fix_us = 4.0;
  m.eff_winograd[0] = rate(146.3);  // 128 x 128 (below Strassen's: 14 + 14 source terms, not 12 + 12)
  m.eff_winograd[1] = rate(166.5);  // 128 x 256
  // small-M tiles: an N = tile_m MMA runs at most tile_m / 256 of the full
  // rate.  These are lower bounds from streams that stayed memory-bound:
  // 16 x 16384^2 at 6.4 TB/s, and tile_m 64 only 5 % slower than tile_m 16
  m.eff_small_m[0] = rate(157.5);   // tile_m 16
  m.eff_small_m[1] = rate(315.0);   // tile_m 32
  m.eff_small_m[2] = rate(607.5);   // tile_m 64
  // streaming rates, as fractions of the copy bandwidth above (fitted as
  // 7110, 5925 and 7663 GB/s)
  m.hbm_stream_eff = 7110.0 / m.hbm_gbs;
  m.small_m_stream_eff = 5925.0 / m.hbm_gbs;  // 16 x 16384^2: 537 MB in ~101-106 us inside the kernel
  m.small_m_fix_us = 4.0;
  // 16 x 16384^2 on 128 CTAs of one whole tile each: 537 MB in 83.7 us, and
  // 16 x 8192^2 on 128 CTAs of half a tile: 32.7 us (CUDA events)
  m.small_m_aligned_eff = 7663.0 / m.hbm_gbs;
  // Winograd's operands formed by the pair kernel's two idle warps per CTA
  // beside its first products: 2.05 GB in about 1.9 ms at 16384^3, while the
  // products of that time ran about 6 % slower
  m.form_in_kernel_eff = 1080.0 / m.hbm_gbs;
  m.form_in_kernel_drag = 0.063;
  // the low-complexity forms round their operand sums: AUTO takes one only
  // for a clear predicted gain, larger than the model's own error
  m.lcma_margin = 0.03;
  // operand panels re-read from DRAM once a wave's panels outgrow the L2
  // (fitted to the classical pair kernel's full-clock times at 16384^3 and
  // 24576^3)
  m.dram_miss_slope = 1.0;
  m.dram_exposed = 0.065 * m.hbm_gbs / 6789.0;  // 0.065 of that time at the measured copy rate
  *out = m;
}

int64_t fgemm_model_tiles(int64_t M, int64_t N, int32_t tile_m, int32_t tile_n) {
  if (M <= 0 || N <= 0 || tile_m <= 0 || tile_n <= 0) return 0;
  return ceil_div(M, tile_m) * ceil_div(N, tile_n);
}

int64_t fgemm_model_waves(int64_t tiles, int32_t slots, double* tail_util) {
  if (tiles <= 0 || slots <= 0) {
    if (tail_util) *tail_util = 0.0;
    return 0;
  }
  const int64_t waves = ceil_div(tiles, slots);
  if (tail_util) {
    const int64_t rem = tiles % slots;
    *tail_util = rem == 0 ? 1.0 : static_cast<double>(rem) / slots;
  }
  return waves;
}

double fgemm_model_tiled_reads(int64_t M, int64_t N, int64_t K, int32_t tile_m, int32_t tile_n) {
  if (K <= 0) return 0.0;
  return static_cast<double>(fgemm_model_tiles(M, N, tile_m, tile_n)) * (tile_m + tile_n) *
         static_cast<double>(K);
}

double fgemm_model_roofline(double flops, double bytes, double peak_flops, double bandwidth) {
  if (bytes <= 0) return peak_flops;
  return std::min(peak_flops, flops / bytes * bandwidth);
}

int32_t fgemm_model_split_tail(const fgemm_device_model_t* dev, int64_t tiles, int32_t clusters,
                               int32_t k_blocks, int32_t tile_n, int32_t mode, int32_t* pieces) {
  if (pieces) *pieces = 1;
  if (mode <= 0 || tiles <= 0 || clusters < 2 || clusters > 255 || k_blocks <= 0) return 0;
  const int64_t rem = tiles % clusters;
  if (rem == 0 || 2 * rem > clusters) return 0;
  const int32_t s = static_cast<int32_t>(
      std::min<int64_t>(std::min<int64_t>(clusters / rem, k_blocks), fgemm::kMaxSplitPieces));
  if (s < 2) return 0;
  if (mode == 1) {
    // auto: split when the part of a tile time it saves, (1 - 1/S) * t_tile,
    // outweighs its cost, split_fix_us per other piece each last piece reads;
    // and only with at least one wave of whole tiles, whose MMAs hide the
    // pieces' partial stores and sums (with none, they are all exposed)
    if (!dev || dev->num_sms <= 0 || tiles < clusters) return 0;
    const double eff = std::max(dev->eff_pair[tile_n == 128 ? 0 : 1], 1e-3);
    const double pair_flop_per_us = dev->peak_tflops * 1e6 / dev->num_sms * 2.0;
    const double t_tile = 2.0 * 256.0 * tile_n * fgemm::kBK * k_blocks / (pair_flop_per_us * eff);
    if ((1.0 - 1.0 / s) * t_tile <= dev->split_fix_us * (s - 1)) return 0;
  }
  if (pieces) *pieces = s;
  return static_cast<int32_t>(rem);
}

int32_t fgemm_split_work_item(int64_t tiles, int32_t split_tiles, int32_t split_pieces,
                              int32_t clusters, int32_t k_blocks, int32_t cluster, int32_t n,
                              int32_t* out5) {
  if (tiles <= 0 || tiles > (1ll << 31) - 1 || clusters <= 0 || k_blocks <= 0 || cluster < 0 ||
      cluster >= clusters || n < 0 || split_tiles < 0 || split_tiles > tiles || !out5)
    return 0;
  if (split_tiles > 0 && (split_pieces < 2 || split_pieces > k_blocks ||
                          static_cast<int64_t>(split_tiles) * split_pieces > clusters))
    return 0;
  fgemm::WorkItem w;
  if (!fgemm::work_item(static_cast<int>(tiles), split_tiles, split_pieces, clusters, k_blocks,
                        cluster, n, w))
    return 0;
  out5[0] = w.unit;
  out5[1] = w.k0;
  out5[2] = w.k1;
  out5[3] = w.piece;
  out5[4] = w.npieces;
  return 1;
}

int32_t fgemm_stream_k_work_item(int64_t tiles, int32_t k_blocks, int32_t ctas, int32_t cta,
                                 int32_t n, int64_t* out6) {
  if (tiles <= 0 || tiles > (1ll << 30) || k_blocks <= 0 || ctas <= 0 || cta < 0 || cta >= ctas ||
      n < 0 || !out6 || static_cast<long long>(ctas) > tiles * k_blocks)
    return 0;
  fgemm::WorkItem w;
  if (!fgemm::stream_k_item(static_cast<int>(tiles), k_blocks, ctas, cta, n, w)) return 0;
  out6[0] = w.unit;
  out6[1] = w.k0;
  out6[2] = w.k1;
  out6[3] = w.piece;
  out6[4] = w.npieces;
  out6[5] = fgemm::stream_k_slot(static_cast<int>(tiles), k_blocks, ctas, w.unit, cta);
  return 1;
}

int32_t fgemm_small_m_grid(int64_t tiles, int32_t k_blocks, int32_t num_sms, int32_t* phases_out) {
  if (tiles <= 0 || tiles > (1ll << 30) || k_blocks <= 0 || num_sms <= 0) return 0;
  const int64_t iters = tiles * k_blocks;
  const int64_t most = std::max<int64_t>(1, std::min<int64_t>(num_sms, ceil_div(iters, 8)));
  const int64_t least = std::max<int64_t>(1, ceil_div(most * 3, 4));
  int64_t best = most, best_phases = most;
  for (int64_t c = most; c >= least; --c) {
    if (iters % c) continue;
    const int64_t share = iters / c;
    const int64_t phases = std::min<int64_t>(c, k_blocks / std::gcd<int64_t>(share, k_blocks));
    if (phases < best_phases) {
      best = c;
      best_phases = phases;
    }
  }
  if (best_phases > 4) {
    best = most;
    best_phases = most;
  }
  if (phases_out) *phases_out = static_cast<int32_t>(best_phases);
  return static_cast<int32_t>(best);
}

namespace {

// Time the operand panels' DRAM re-reads add to a persistent GEMM launch
// (microseconds).  The tiles of one wave (rows x cols of the tile grid in
// flight, rasterised in groups of 8 tile rows) share the A panels of their
// rows and the B panels of their columns, each K long.  Once those panels
// outgrow the L2, the part beyond it is re-read from DRAM by the tiles that
// share it: a share min(1, dram_miss_slope * (panels / L2 - 1)) of the tiled
// reads, of whose DRAM time a part (dram_exposed) is not hidden behind the
// MMAs.  Fitted to the classical pair kernel's full-clock times (16384^3:
// panels 1.09 L2, no visible cost; 24576^3: 1.63 L2, about 1.4 ms of 17).
// `products`: launches of that shape in sequence (the block products of a
// Strassen-like level, each with its own half-size panels).
double operand_dram_us(const fgemm_device_model_t* dev, int64_t tiles_m, int64_t tiles_n, int32_t tile_m,
                       int32_t tile_n, double k, int32_t slots, double products) {
  if (dev->dram_exposed <= 0.0 || dev->dram_miss_slope <= 0.0 || dev->l2_bytes <= 0.0) return 0.0;
  const int64_t rows = std::min<int64_t>(tiles_m, 8);
  const int64_t cols = std::min<int64_t>(tiles_n, ceil_div(slots, std::max<int64_t>(rows, 1)));
  const double panels = (static_cast<double>(rows) * tile_m + static_cast<double>(cols) * tile_n) * k * 2.0;
  const double tiled = static_cast<double>(tiles_m) * tiles_n * (tile_m + tile_n) * k * 2.0 * products;
  const double miss = std::min(1.0, dev->dram_miss_slope * std::max(0.0, panels / dev->l2_bytes - 1.0));
  return dev->dram_exposed * tiled * miss / (dev->hbm_gbs * 1e3);
}

}  // namespace

extern "C++" {
namespace fgemm {

fgemm_status_t model_search(const fgemm_device_model_t* dev, int64_t M, int64_t N, int64_t K,
                            int32_t epi_kind, fgemm_algo_t algo, int32_t tile_m, int32_t tile_n,
                            int32_t min_tile_m, fgemm_algo_t* algo_out, int32_t* tm_out, int32_t* tn_out,
                            double* us_out) {
  if (!dev) return FGEMM_ERR_INVALID_ARG;
  const fgemm_algo_t forms[4] = {FGEMM_ALGO_CLASSICAL, FGEMM_ALGO_STRASSEN1, FGEMM_ALGO_STRASSEN2,
                                 FGEMM_ALGO_WINOGRAD1};
  // the classical forms first; under AUTO a low-complexity form must then
  // beat the best of them by the margin
  const double margin = std::min(std::max(dev->lcma_margin, 0.0), 0.9);
  double best = INFINITY, best_us = INFINITY;
  fgemm_algo_t best_algo = FGEMM_ALGO_CLASSICAL;
  int32_t best_m = 0, best_n = 0;
  for (fgemm_algo_t a : forms) {
    if (algo != FGEMM_ALGO_AUTO && a != algo) continue;
    const double scale = (algo == FGEMM_ALGO_AUTO && a != FGEMM_ALGO_CLASSICAL) ? 1.0 / (1.0 - margin) : 1.0;
    for (int32_t tm : {16, 32, 64, 128, 256}) {
      if ((tile_m != 0 && tm != tile_m) || tm < min_tile_m) continue;
      for (int32_t tn : {64, 128, 256}) {
        if (tile_n != 0 && tn != tile_n) continue;
        double us = 0;
        if (fgemm_model_predict(dev, M, N, K, epi_kind, a, tm, tn, &us) != FGEMM_OK) continue;
        if (us * scale < best) {
          best = us * scale;
          best_us = us;
          best_algo = a;
          best_m = tm;
          best_n = tn;
        }
      }
    }
  }
  if (best_n == 0) return FGEMM_ERR_UNSUPPORTED;
  if (algo_out) *algo_out = best_algo;
  if (tm_out) *tm_out = best_m;
  if (tn_out) *tn_out = best_n;
  if (us_out) *us_out = best_us;
  return FGEMM_OK;
}

}  // namespace fgemm
}  // extern "C++"

int64_t fgemm_lcma_pair_clusters(int64_t positions, int32_t depth, int32_t fit) {
  if (positions <= 0 || fit <= 0) return 0;
  const int64_t units = positions * (depth == 2 ? 49 : 7);
  if (depth != 2) return std::min<int64_t>(fit, units);
  // Two levels: each position of a partial last wave becomes 49 product
  // units whose combinations the helper warps run.  With fewer positions
  // than pairs, one pair per position; with more than 24 such units per pair
  // (8192 x 16384^2 at 256 x 256: 34 per pair, 14.6 ms against 4.6 at
  // 256 x 128), the most pairs, down to half of them, that divide the
  // positions into whole waves.
  if (positions < fit) return positions;
  const int64_t tail = positions % fit;
  if ((tail * 49 + fit - 1) / fit <= 24) return fit;
  for (int64_t c = fit; 2 * c >= fit; --c)
    if (positions % c == 0) return c;
  return fit;
}

fgemm_status_t fgemm_model_predict(const fgemm_device_model_t* dev, int64_t M, int64_t N,
                                   int64_t K, int32_t epi_kind, fgemm_algo_t algo, int32_t tile_m,
                                   int32_t tile_n, double* predicted_us) {
  if (!dev || M < 0 || N < 0 || K < 0) return FGEMM_ERR_INVALID_ARG;
  if (algo == FGEMM_ALGO_AUTO) return FGEMM_ERR_INVALID_ARG;
  if (!fgemm::form_is_legal(M, N, K, epi_kind, algo, tile_m, tile_n)) return FGEMM_ERR_UNSUPPORTED;
  if (tile_m < 128) {
    // small-M kernel: every CTA of the grid fgemm_small_m_grid picks streams
    // an equal share of the K blocks of all 128-column tiles; bound by B from
    // HBM or by the narrow MMAs
    const int64_t tiles = ceil_div(N, 128), kb = ceil_div(K, fgemm::kBK);
    const int64_t iters = tiles * kb;
    int32_t phases = 0;
    const int64_t ctas = std::max(1, fgemm_small_m_grid(tiles, static_cast<int32_t>(kb), dev->num_sms, &phases));
    const bool aligned = phases <= 4;
    const double eff = std::max(dev->eff_small_m[tile_m == 16 ? 0 : (tile_m == 32 ? 1 : 2)], 1e-3);
    const double sm_flop_per_us = dev->peak_tflops * 1e6 / dev->num_sms;
    const double t_kb = 2.0 * 128.0 * tile_m * fgemm::kBK / (sm_flop_per_us * eff);
    // (its pipeline fill and last sum are in small_m_fix_us)
    const double t_compute = static_cast<double>(ceil_div(iters, ctas)) * t_kb;
    const double bytes = 2.0 * (static_cast<double>(M) * K + static_cast<double>(K) * N +
                                static_cast<double>(M) * N);
    // CTAs reading B in step stream at the full rate from 3/4 of the SMs on;
    // otherwise the rate scales with the SMs in use
    const double sm_share = std::min(
        1.0, static_cast<double>(ctas) / std::max(1.0, (aligned ? 0.75 : 1.0) * dev->num_sms));
    const double stream_eff = aligned ? dev->small_m_aligned_eff : dev->small_m_stream_eff;
    const double t_memory = bytes / (dev->hbm_gbs * 1e3 * std::max(stream_eff, 1e-3) * sm_share);
    if (predicted_us)
      *predicted_us = std::max(t_compute, t_memory) + dev->small_m_fix_us + dev->launch_us;
    return FGEMM_OK;
  }
  const int d = depth_of(algo);
  const bool swiglu = epi_kind == FGEMM_EPI_SWIGLU;
  const bool pair = tile_m == 256;
  if (pair && d >= 1) {
    // One or two levels on CTA pairs with the summed operands streamed
    // through HBM: a pre-pass reads A and B once and writes each summed
    // operand once (one level: Strassen 5 + 5 of the 4 + 4 blocks, Winograd
    // 4 + 4; two levels: 45 + 45 of the 16 + 16), then the 7^d block
    // products run on the classical pair mainloop: whole positions in waves
    // over the pairs, the partial last wave's positions as separate product
    // units shared out evenly, whose combination costs about one more fill.
    const bool wino = algo == FGEMM_ALGO_WINOGRAD1;
    const int64_t sub_m = M >> d, sub_n = N >> d, sub_k = K >> d;
    const int64_t np = d == 1 ? 7 : 49;
    const double temps = d == 2 ? 45.0 : (wino ? 4.0 : 5.0);
    const double pre_bytes = 2.0 * (static_cast<double>(M) * K + static_cast<double>(K) * N +
                                    temps * (static_cast<double>(sub_m) * sub_k +
                                             static_cast<double>(sub_k) * sub_n));
    double t_pre = pre_bytes / (dev->hbm_gbs * 1e3 * std::max(dev->hbm_stream_eff, 1e-3)) +
                   dev->launch_us;
    const int64_t positions = fgemm_model_tiles(sub_m, sub_n, 256, tile_n);
    const int32_t pairs = std::max(1, dev->num_sms / 2);
    const int64_t used = fgemm_lcma_pair_clusters(positions, d, pairs);
    const int64_t whole = positions / used;
    const int64_t tail_units = (positions % used) * np;
    const double eff = std::max(d == 2 ? dev->eff_strassen2_pair[tile_n == 128 ? 0 : 1]
                                       : dev->eff_strassen_pair[tile_n == 128 ? 0 : 1],
                                1e-3);
    const double pair_flop_per_us = dev->peak_tflops * 1e6 / dev->num_sms * 2.0;
    const double k_pad = static_cast<double>(ceil_div(sub_k, fgemm::kBK) * fgemm::kBK);
    double t_unit = 2.0 * 256.0 * tile_n * k_pad / (pair_flop_per_us * eff);
    if (d == 2) {
      // the fold of a unit into its output blocks (fp32 reductions at the
      // L2) overlaps its MMAs only in part: the longer of the two, plus a
      // share kFoldOverlap of the shorter
      constexpr double kFoldOverlap = 0.55;
      const double fold = std::max(dev->fold2_unit_us, 0.0) * tile_n / 256.0;
      t_unit = std::max(t_unit, fold) + kFoldOverlap * std::min(t_unit, fold);
    }
    // The product kernel forms sums itself while the products that do not
    // read them run first: Winograd's two sum-free products (A11 B11, A12 B21)
    // cover both sides' sums, formed A's then B's; Strassen's M2 and M5 read
    // no sum of B, so B's sums are formed in the kernel and A's by a pre-pass
    // half the size.  With at least kFusedMinWaves waves of those products
    // this is done; what shows is the products' drag during the formation,
    // and any part of it still running when the first product that reads
    // the last side formed starts.
    const int64_t lead = 2;
    if (d == 1 && lead * whole >= fgemm::kFusedMinWaves && sub_m % fgemm::kFormRows == 0 &&
        sub_k % fgemm::kFormRows == 0) {
      const double a_bytes = 2.0 * (static_cast<double>(M) * K + temps * static_cast<double>(sub_m) * sub_k);
      const double b_bytes = 2.0 * (static_cast<double>(K) * N + temps * static_cast<double>(sub_k) * sub_n);
      const double in_kernel = wino ? a_bytes + b_bytes : b_bytes;
      const double t_form = in_kernel / (dev->hbm_gbs * 1e3 * std::max(dev->form_in_kernel_eff, 1e-3));
      const double drag = std::max(dev->form_in_kernel_drag, 0.0);
      const double w = static_cast<double>(whole) * t_unit;
      // the first product that needs the in-kernel side's (last) sums
      const double needed_at = static_cast<double>(wino ? lead + 1 : lead) * w;
      t_pre = drag * t_form + std::max(0.0, t_form - (1.0 + drag) * needed_at);
      if (!wino)  // A's sums by the pre-pass
        t_pre += a_bytes / (dev->hbm_gbs * 1e3 * std::max(dev->hbm_stream_eff, 1e-3)) + dev->launch_us;
    }
    const double per_pair = static_cast<double>(whole * np + ceil_div(tail_units, used));
    const double t_compute = per_pair * t_unit + dev->tile_fill_us * (tail_units > 0 ? 2.0 : 1.0) +
                             operand_dram_us(dev, ceil_div(sub_m, 256), ceil_div(sub_n, tile_n), 256, tile_n,
                                             k_pad, pairs, static_cast<double>(np));
    if (predicted_us) *predicted_us = t_pre + t_compute + dev->launch_us;
    return FGEMM_OK;
  }
  const int64_t n_out = swiglu ? N / 2 : N;
  const int64_t sub_m = M >> d, sub_n = N >> d, sub_k = K >> d;
  const int64_t products = d == 0 ? 1 : (d == 1 ? 7 : 49);
  int64_t tiles;
  if (d == 0 && swiglu)
    tiles = fgemm_model_tiles(sub_m, n_out, tile_m, tile_n / 2);
  else
    tiles = fgemm_model_tiles(sub_m, sub_n, tile_m, tile_n);
  // a pair of SMs works on one 256-row tile
  const int32_t slots = pair ? std::max(1, dev->num_sms / 2) : dev->num_sms;
  const int64_t waves = fgemm_model_waves(tiles, slots, nullptr);
  const bool wino = algo == FGEMM_ALGO_WINOGRAD1;
  double eff;
  if (wino)
    eff = dev->eff_winograd[tile_n == 128 ? 0 : 1];
  else if (d > 0 && pair)
    eff = dev->eff_strassen_pair[tile_n == 128 ? 0 : 1];
  else if (d > 0)
    eff = dev->eff_strassen[d - 1][tile_n == 128 ? 0 : 1];
  else if (pair)
    eff = dev->eff_pair[tile_n == 128 ? 0 : 1];
  else
    eff = dev->eff_classical[tile_index(tile_n)];
  const double slot_flop_per_us = dev->peak_tflops * 1e6 / dev->num_sms * (pair ? 2.0 : 1.0);
  const double k_pad = static_cast<double>(ceil_div(sub_k, fgemm::kBK) * fgemm::kBK);
  // a tile's (or a Strassen position's) MMA time; the epilogue of one tile
  // overlaps the next tile's MMAs, so the pipeline fill and the last
  // epilogue are paid once per launch
  const double t_tile =
      products * (2.0 * tile_m * tile_n * k_pad / (slot_flop_per_us * std::max(eff, 1e-3)));
  double t_compute = static_cast<double>(waves) * t_tile;
  if (pair && d == 0) {
    // the tiles of the last partial wave may be split along K into S pieces
    const int32_t kb = static_cast<int32_t>(std::min<int64_t>(ceil_div(sub_k, fgemm::kBK), 1 << 30));
    int32_t s = 1;
    if (fgemm_model_split_tail(dev, tiles, slots, kb, tile_n, 1, &s) > 0)
      t_compute = (static_cast<double>(tiles / slots) + 1.0 / s) * t_tile + dev->split_fix_us * (s - 1);
  }
  t_compute += dev->tile_fill_us;
  {
    const int32_t tn_eff = (d == 0 && swiglu) ? tile_n / 2 : tile_n;
    const int64_t cols = d == 0 && swiglu ? n_out : sub_n;
    t_compute += operand_dram_us(dev, ceil_div(sub_m, tile_m), ceil_div(cols, tn_eff), tile_m, tile_n, k_pad,
                                 slots, static_cast<double>(products));
  }
  double bytes = 2.0 * (static_cast<double>(M) * K + static_cast<double>(K) * N +
                        static_cast<double>(M) * n_out);
  if (d > 0) {
    const double slot_bytes = 4.0 * fgemm::kBM * tile_n;
    const double nslots = std::pow(4.0, d);
    const double live = std::min<double>(static_cast<double>(tiles), dev->num_sms) * nslots * slot_bytes;
    if (live > dev->l2_bytes) {
      // nonzeros of the output combination: 12 per Strassen level, 14 for Winograd
      const double contributions = wino ? 14.0 : std::pow(12.0, d);
      bytes += static_cast<double>(tiles) * (2.0 * contributions) * slot_bytes;
    }
  }
  // a launch that keeps s SMs busy streams at most s / num_sms of the device
  // bandwidth (each SM has a bounded number of copies in flight)
  const double busy_sms = static_cast<double>(std::min<int64_t>(tiles, slots)) * (pair ? 2.0 : 1.0);
  const double sm_share = std::min(1.0, busy_sms / std::max(1, dev->num_sms));
  const double t_memory =
      bytes / (dev->hbm_gbs * 1e3 * std::max(dev->hbm_stream_eff, 1e-3) * std::max(sm_share, 1e-3));
  // Operand tiles streamed from L2 into the SMs (tiled reads): every product
  // re-reads its source blocks; the scheme's term counts are 12 + 12 at depth
  // 1 and 144 + 144 at depth 2 (against 8 + 8 for the four classical blocks).
  double op_elems = static_cast<double>(tiles) * (tile_m + tile_n) * k_pad;
  if (d == 1) op_elems *= wino ? 14.0 : 12.0;
  if (d == 2) op_elems *= 144.0;
  const double t_operands = 2.0 * op_elems / (dev->l2_gbs * 1e3);
  if (predicted_us)
    *predicted_us = std::max(std::max(t_compute, t_memory), t_operands) + dev->launch_us;
  return FGEMM_OK;
}

fgemm_status_t fgemm_model_plan(const fgemm_device_model_t* dev, int64_t M, int64_t N, int64_t K,
                                int32_t epi_kind, fgemm_algo_t* algo_out, int32_t* tile_m,
                                int32_t* tile_n, double* predicted_us) {
  return fgemm::model_search(dev, M, N, K, epi_kind, FGEMM_ALGO_AUTO, 0, 0, 0, algo_out, tile_m, tile_n,
                             predicted_us);
}

}  // extern "C"

// ------------------------------------------------ device model as JSON

namespace {

// Every field of the model that a calibration file carries (key, member).
std::vector<std::pair<const char*, double*>> model_fields(fgemm_device_model_t& m) {
  return {
      {"peak_tflops", &m.peak_tflops},
      {"hbm_gbs", &m.hbm_gbs},
      {"eff_classical_64", &m.eff_classical[0]},
      {"eff_classical_128", &m.eff_classical[1]},
      {"eff_classical_256", &m.eff_classical[2]},
      {"eff_pair_128", &m.eff_pair[0]},
      {"eff_pair_256", &m.eff_pair[1]},
      {"eff_strassen1_128", &m.eff_strassen[0][0]},
      {"eff_strassen1_256", &m.eff_strassen[0][1]},
      {"eff_strassen2_128", &m.eff_strassen[1][0]},
      {"eff_strassen2_256", &m.eff_strassen[1][1]},
      {"eff_strassen1_pair_128", &m.eff_strassen_pair[0]},
      {"eff_strassen1_pair_256", &m.eff_strassen_pair[1]},
      {"eff_strassen2_pair_128", &m.eff_strassen2_pair[0]},
      {"eff_strassen2_pair_256", &m.eff_strassen2_pair[1]},
      {"fold2_unit_us", &m.fold2_unit_us},
      {"launch_us", &m.launch_us},
      {"tile_fill_us", &m.tile_fill_us},
      {"l2_bytes", &m.l2_bytes},
      {"l2_gbs", &m.l2_gbs},
      {"split_fix_us", &m.split_fix_us},
      {"eff_winograd1_128", &m.eff_winograd[0]},
      {"eff_winograd1_256", &m.eff_winograd[1]},
      {"eff_small_m_16", &m.eff_small_m[0]},
      {"eff_small_m_32", &m.eff_small_m[1]},
      {"eff_small_m_64", &m.eff_small_m[2]},
      {"hbm_stream_eff", &m.hbm_stream_eff},
      {"small_m_stream_eff", &m.small_m_stream_eff},
      {"small_m_fix_us", &m.small_m_fix_us},
      {"small_m_aligned_eff", &m.small_m_aligned_eff},
      {"form_in_kernel_eff", &m.form_in_kernel_eff},
      {"form_in_kernel_drag", &m.form_in_kernel_drag},
      {"lcma_margin", &m.lcma_margin},
      {"dram_miss_slope", &m.dram_miss_slope},
      {"dram_exposed", &m.dram_exposed},
  };
}

// The number after "key": in a flat JSON object (false if absent or not a
// number).
bool json_number(const std::string& text, const char* key, double* out) {
  const std::string pat = std::string("\"") + key + "\"";
  size_t p = text.find(pat);
  if (p == std::string::npos) return false;
  p = text.find_first_not_of(" \t\r\n", p + pat.size());
  if (p == std::string::npos || text[p] != ':') return false;
  const char* s = text.c_str() + p + 1;
  char* end = nullptr;
  const double d = std::strtod(s, &end);
  if (end == s || !std::isfinite(d)) return false;
  *out = d;
  return true;
}

}  // namespace

extern "C" fgemm_status_t fgemm_model_load_json(const char* path, fgemm_device_model_t* model) {
  if (!path || !model) return FGEMM_ERR_INVALID_ARG;
  FILE* f = std::fopen(path, "rb");
  if (!f) return FGEMM_ERR_CALIBRATION;
  std::string text;
  char buf[4096];
  size_t n;
  while ((n = std::fread(buf, 1, sizeof(buf), f)) > 0 && text.size() < (1u << 20)) text.append(buf, n);
  std::fclose(f);
  fgemm_device_model_t m = *model;
  const double old_peak = m.peak_tflops, old_bw = m.hbm_gbs;
  double v = 0, tf = 0;
  // A file of measured peaks (a dense bf16 GEMM rate "bf16_tflops" and a
  // copy bandwidth "hbm_gbs", without the model's own "peak_tflops"): the
  // denominators change and every efficiency is rescaled, so that the rates
  // the model predicts stay the ones it was fitted to.
  const bool peaks_file = !json_number(text, "peak_tflops", &v) && json_number(text, "bf16_tflops", &tf);
  int found = 0;
  for (auto& fd : model_fields(m)) found += json_number(text, fd.first, fd.second) ? 1 : 0;
  if (json_number(text, "num_sms", &v) && v >= 1 && v <= 4096) {
    m.num_sms = static_cast<int32_t>(v);
    ++found;
  }
  if (peaks_file) {
    if (!(tf > 0) || !(m.hbm_gbs > 0)) return FGEMM_ERR_CALIBRATION;
    const double r = old_peak / tf;
    for (double* e : {&m.eff_classical[0], &m.eff_classical[1], &m.eff_classical[2], &m.eff_pair[0],
                      &m.eff_pair[1], &m.eff_strassen[0][0], &m.eff_strassen[0][1],
                      &m.eff_strassen[1][0], &m.eff_strassen[1][1], &m.eff_strassen_pair[0],
                      &m.eff_strassen_pair[1], &m.eff_strassen2_pair[0], &m.eff_strassen2_pair[1],
                      &m.eff_winograd[0], &m.eff_winograd[1],
                      &m.eff_small_m[0], &m.eff_small_m[1], &m.eff_small_m[2]})
      *e *= r;
    const double rb = old_bw / m.hbm_gbs;
    for (double* e : {&m.hbm_stream_eff, &m.small_m_stream_eff, &m.small_m_aligned_eff, &m.form_in_kernel_eff})
      *e *= rb;
    m.dram_exposed /= rb;  // a share of bytes / hbm_gbs: the same time
    m.peak_tflops = tf;
    ++found;
  }
  if (!found) return FGEMM_ERR_CALIBRATION;
  if (!(m.peak_tflops > 0) || !(m.hbm_gbs > 0) || !(m.launch_us >= 0) || !(m.tile_fill_us >= 0))
    return FGEMM_ERR_CALIBRATION;
  *model = m;
  return FGEMM_OK;
}

extern "C" fgemm_status_t fgemm_model_save_json(const fgemm_device_model_t* model, const char* path) {
  if (!path || !model) return FGEMM_ERR_INVALID_ARG;
  FILE* f = std::fopen(path, "w");
  if (!f) return FGEMM_ERR_CALIBRATION;
  fgemm_device_model_t m = *model;
  std::fprintf(f, "{\n  \"num_sms\": %d", m.num_sms);
  for (auto& fd : model_fields(m)) std::fprintf(f, ",\n  \"%s\": %.9g", fd.first, *fd.second);
  std::fprintf(f, "\n}\n");
  const bool ok = std::fclose(f) == 0;
  return ok ? FGEMM_OK : FGEMM_ERR_CALIBRATION;
}
