// fgemm_tables.cpp -- coefficient tables of the low-complexity schemes
// (host code).  The kernels read them as StrassenTable: per product, the
// signed source blocks summed into each operand and the output blocks the
// product is added into.
//
// FalconGEMM names Strassen-like schemes without printing their formulas;
// these are the textbook one-level Strassen scheme, its Kronecker square for
// two levels, and Winograd's variant with its shared partial sums expanded.
#include <cstdint>
#include <cstring>

#include "fgemm_internal.h"

using fgemm::StrassenTable;

namespace {

// One-level Strassen scheme (textbook form): for product k, the A blocks and
// signs summed into its left operand, the B blocks into its right operand,
// and the output blocks it is added into.  Block (r, c) of a 2 x 2 split.
struct Term1 {
  int r, c, sign;
};
struct Product1 {
  int na;
  Term1 a[2];
  int nb;
  Term1 b[2];
  int nc;
  Term1 c[2];
};
const Product1 kStrassen1[7] = {
    // M1 = (A11 + A22)(B11 + B22) -> C11 +, C22 +
    {2, {{0, 0, 1}, {1, 1, 1}}, 2, {{0, 0, 1}, {1, 1, 1}}, 2, {{0, 0, 1}, {1, 1, 1}}},
    // M2 = (A21 + A22) B11 -> C21 +, C22 -
    {2, {{1, 0, 1}, {1, 1, 1}}, 1, {{0, 0, 1}, {0, 0, 0}}, 2, {{1, 0, 1}, {1, 1, -1}}},
    // M3 = A11 (B12 - B22) -> C12 +, C22 +
    {1, {{0, 0, 1}, {0, 0, 0}}, 2, {{0, 1, 1}, {1, 1, -1}}, 2, {{0, 1, 1}, {1, 1, 1}}},
    // M4 = A22 (B21 - B11) -> C11 +, C21 +
    {1, {{1, 1, 1}, {0, 0, 0}}, 2, {{1, 0, 1}, {0, 0, -1}}, 2, {{0, 0, 1}, {1, 0, 1}}},
    // M5 = (A11 + A12) B22 -> C11 -, C12 +
    {2, {{0, 0, 1}, {0, 1, 1}}, 1, {{1, 1, 1}, {0, 0, 0}}, 2, {{0, 0, -1}, {0, 1, 1}}},
    // M6 = (A21 - A11)(B11 + B12) -> C22 +
    {2, {{1, 0, 1}, {0, 0, -1}}, 2, {{0, 0, 1}, {0, 1, 1}}, 1, {{1, 1, 1}, {0, 0, 0}}},
    // M7 = (A12 - A22)(B21 + B22) -> C11 +
    {2, {{0, 1, 1}, {1, 1, -1}}, 2, {{1, 0, 1}, {1, 1, 1}}, 1, {{0, 0, 1}, {0, 0, 0}}},
};

uint8_t term_code(int r, int c, int sign, int depth) {
  const int idx = (r << depth) | c;
  return static_cast<uint8_t>(idx | (sign < 0 ? fgemm::kTermNeg : 0));
}

// Table for `depth` levels: the depth-2 scheme applies the one-level scheme
// to each of the seven products' half-size operands (outer product p, inner
// product q), so block indices and signs multiply.
StrassenTable build_table(int depth) {
  StrassenTable t;
  std::memset(&t, 0, sizeof(t));
  if (depth == 0) {
    t.na[0] = t.nb[0] = t.nc[0] = 1;
    t.a[0][0] = t.b[0][0] = 0;
    t.c[0][0] = fgemm::kTermFirst;
    return t;
  }
  int np = 0;
  if (depth == 1) {
    for (int p = 0; p < 7; ++p, ++np) {
      const Product1& P = kStrassen1[p];
      t.na[np] = static_cast<uint8_t>(P.na);
      t.nb[np] = static_cast<uint8_t>(P.nb);
      t.nc[np] = static_cast<uint8_t>(P.nc);
      for (int i = 0; i < P.na; ++i) t.a[np][i] = term_code(P.a[i].r, P.a[i].c, P.a[i].sign, 1);
      for (int i = 0; i < P.nb; ++i) t.b[np][i] = term_code(P.b[i].r, P.b[i].c, P.b[i].sign, 1);
      for (int i = 0; i < P.nc; ++i) t.c[np][i] = term_code(P.c[i].r, P.c[i].c, P.c[i].sign, 1);
    }
  } else {
    for (int p = 0; p < 7; ++p) {
      for (int q = 0; q < 7; ++q, ++np) {
        const Product1& O = kStrassen1[p];
        const Product1& I = kStrassen1[q];
        int n = 0;
        for (int i = 0; i < O.na; ++i)
          for (int j = 0; j < I.na; ++j)
            t.a[np][n++] = term_code(O.a[i].r * 2 + I.a[j].r, O.a[i].c * 2 + I.a[j].c,
                                     O.a[i].sign * I.a[j].sign, 2);
        t.na[np] = static_cast<uint8_t>(n);
        n = 0;
        for (int i = 0; i < O.nb; ++i)
          for (int j = 0; j < I.nb; ++j)
            t.b[np][n++] = term_code(O.b[i].r * 2 + I.b[j].r, O.b[i].c * 2 + I.b[j].c,
                                     O.b[i].sign * I.b[j].sign, 2);
        t.nb[np] = static_cast<uint8_t>(n);
        n = 0;
        for (int i = 0; i < O.nc; ++i)
          for (int j = 0; j < I.nc; ++j)
            t.c[np][n++] = term_code(O.c[i].r * 2 + I.c[j].r, O.c[i].c * 2 + I.c[j].c,
                                     O.c[i].sign * I.c[j].sign, 2);
        t.nc[np] = static_cast<uint8_t>(n);
      }
    }
  }
  // Mark the first contribution to each output block (it stores instead of
  // adding), in product order.
  bool seen[16] = {false};
  for (int p = 0; p < np; ++p) {
    for (int i = 0; i < t.nc[p]; ++i) {
      const int idx = t.c[p][i] & fgemm::kTermIndexMask;
      if (!seen[idx]) {
        seen[idx] = true;
        t.c[p][i] |= fgemm::kTermFirst;
      }
    }
  }
  return t;
}

const StrassenTable& table_for(int depth) {
  static const StrassenTable t0 = build_table(0);
  static const StrassenTable t1 = build_table(1);
  static const StrassenTable t2 = build_table(2);
  return depth == 0 ? t0 : (depth == 1 ? t1 : t2);
}

// One level of Winograd's variant, its shared partial sums expanded into
// signed sums of source blocks (the kernel forms every operand from the
// blocks themselves, in fp32, rounded once):
//   S1 = A21 + A22, S2 = S1 - A11, S3 = A11 - A21, S4 = A12 - S2
//   T1 = B12 - B11, T2 = B22 - T1, T3 = B22 - B12, T4 = T2 - B21
//   P1 = A11 B11, P2 = A12 B21, P3 = S4 B22, P4 = A22 T4,
//   P5 = S1 T1, P6 = S2 T2, P7 = S3 T3
//   C11 = P1 + P2, C12 = P1 + P6 + P5 + P3, C21 = P1 + P6 + P7 - P4,
//   C22 = P1 + P6 + P7 + P5
struct TermW {
  int r, c, sign;
};
struct ProductW {
  int na;
  TermW a[4];
  int nb;
  TermW b[4];
  int nc;
  TermW c[4];
};
const ProductW kWinograd1[7] = {
    // P1 = A11 B11 -> every output block
    {1, {{0, 0, 1}}, 1, {{0, 0, 1}}, 4, {{0, 0, 1}, {0, 1, 1}, {1, 0, 1}, {1, 1, 1}}},
    // P2 = A12 B21 -> C11
    {1, {{0, 1, 1}}, 1, {{1, 0, 1}}, 1, {{0, 0, 1}}},
    // P3 = (A11 + A12 - A21 - A22) B22 -> C12
    {4, {{0, 0, 1}, {0, 1, 1}, {1, 0, -1}, {1, 1, -1}}, 1, {{1, 1, 1}}, 1, {{0, 1, 1}}},
    // P4 = A22 (B11 - B12 - B21 + B22) -> C21 -
    {1, {{1, 1, 1}}, 4, {{0, 0, 1}, {0, 1, -1}, {1, 0, -1}, {1, 1, 1}}, 1, {{1, 0, -1}}},
    // P5 = (A21 + A22)(B12 - B11) -> C12, C22
    {2, {{1, 0, 1}, {1, 1, 1}}, 2, {{0, 1, 1}, {0, 0, -1}}, 2, {{0, 1, 1}, {1, 1, 1}}},
    // P6 = (A21 + A22 - A11)(B22 - B12 + B11) -> C12, C21, C22
    {3, {{1, 0, 1}, {1, 1, 1}, {0, 0, -1}}, 3, {{1, 1, 1}, {0, 1, -1}, {0, 0, 1}}, 3,
     {{0, 1, 1}, {1, 0, 1}, {1, 1, 1}}},
    // P7 = (A11 - A21)(B22 - B12) -> C21, C22
    {2, {{0, 0, 1}, {1, 0, -1}}, 2, {{1, 1, 1}, {0, 1, -1}}, 2, {{1, 0, 1}, {1, 1, 1}}},
};

StrassenTable build_winograd_table() {
  StrassenTable t;
  std::memset(&t, 0, sizeof(t));
  bool seen[4] = {false};
  for (int p = 0; p < 7; ++p) {
    const ProductW& P = kWinograd1[p];
    t.na[p] = static_cast<uint8_t>(P.na);
    t.nb[p] = static_cast<uint8_t>(P.nb);
    t.nc[p] = static_cast<uint8_t>(P.nc);
    for (int i = 0; i < P.na; ++i) t.a[p][i] = term_code(P.a[i].r, P.a[i].c, P.a[i].sign, 1);
    for (int i = 0; i < P.nb; ++i) t.b[p][i] = term_code(P.b[i].r, P.b[i].c, P.b[i].sign, 1);
    for (int i = 0; i < P.nc; ++i) {
      t.c[p][i] = term_code(P.c[i].r, P.c[i].c, P.c[i].sign, 1);
      const int idx = t.c[p][i] & fgemm::kTermIndexMask;
      if (!seen[idx]) {  // the first contribution to a block stores
        seen[idx] = true;
        t.c[p][i] |= fgemm::kTermFirst;
      }
    }
  }
  return t;
}

const StrassenTable& winograd_table_ref() {
  static const StrassenTable t = build_winograd_table();
  return t;
}

}  // namespace

namespace fgemm {

const StrassenTable& strassen_table(int depth) { return table_for(depth); }

const StrassenTable& winograd_table() { return winograd_table_ref(); }

}  // namespace fgemm
