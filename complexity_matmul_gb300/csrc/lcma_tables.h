// LCMA coefficient tables (U, V, W) for one- and two-level Strassen, built at
// compile time.
//
// FalconGEMM write-up (hyper.ai news 54396, section "从 Strassen 出发"): an
// LCMA algorithm is described by which sub-blocks of A and B are combined
// before the products, how many products run and how the products recombine
// into C.  The one-level table is the textbook Strassen (1969) scheme
// (7 products instead of 8); two levels apply it inside every product, i.e.
// the Kronecker product of the one-level tables (49 products over a 4x4 block
// grid instead of 64).
//
// Conventions: A block (R, C) is block row R (along M), block column C (along
// K); B block (R, C) is block row R (along K), block column C (along N); C
// block (R, C) is block row R (along M), block column C (along N).  With L
// levels the grid is G x G, G = 2^L, and product index p = 7*p_outer + p_inner,
// block row = 2*r_outer + r_inner (likewise for columns).
#pragma once

#include <cstdint>

namespace lcg {

// one-level tables, block index 2*r + c (11, 12, 21, 22)
constexpr int8_t kU1[7][4] = {
    {1, 0, 0, 1},   // M1: A11 + A22
    {0, 0, 1, 1},   // M2: A21 + A22
    {1, 0, 0, 0},   // M3: A11
    {0, 0, 0, 1},   // M4: A22
    {1, 1, 0, 0},   // M5: A11 + A12
    {-1, 0, 1, 0},  // M6: A21 - A11
    {0, 1, 0, -1},  // M7: A12 - A22
};
constexpr int8_t kV1[7][4] = {
    {1, 0, 0, 1},   // M1: B11 + B22
    {1, 0, 0, 0},   // M2: B11
    {0, 1, 0, -1},  // M3: B12 - B22
    {-1, 0, 1, 0},  // M4: B21 - B11
    {0, 0, 0, 1},   // M5: B22
    {1, 1, 0, 0},   // M6: B11 + B12
    {0, 0, 1, 1},   // M7: B21 + B22
};
constexpr int8_t kW1[4][7] = {
    {1, 0, 0, 1, -1, 0, 1},   // C11 = M1 + M4 - M5 + M7
    {0, 0, 1, 0, 1, 0, 0},    // C12 = M3 + M5
    {0, 1, 0, 1, 0, 0, 0},    // C21 = M2 + M4
    {1, -1, 1, 0, 0, 1, 0},   // C22 = M1 - M2 + M3 + M6
};

constexpr int ipow(int b, int e) { return e == 0 ? 1 : b * ipow(b, e - 1); }

// Coefficient of operand block (R, C) in product p for L levels.
// `which`: 0 = U (A side), 1 = V (B side).
constexpr int coef(int which, int L, int p, int R, int C) {
  int c = 1;
  for (int l = L - 1; l >= 0; --l) {   // l = 0 is the innermost level
    const int pl = (p / ipow(7, l)) % 7;
    const int rl = (R >> l) & 1, cl = (C >> l) & 1;
    c *= (which == 0 ? kU1[pl][2 * rl + cl] : kV1[pl][2 * rl + cl]);
  }
  return c;
}

// Coefficient of product p in C block (R, C) for L levels.
constexpr int wcoef(int L, int R, int C, int p) {
  int c = 1;
  for (int l = L - 1; l >= 0; --l) {
    const int pl = (p / ipow(7, l)) % 7;
    const int rl = (R >> l) & 1, cl = (C >> l) & 1;
    c *= kW1[2 * rl + cl][pl];
  }
  return c;
}

// Per-level summary used by the kernels: for every product and side, either
// an alias of one raw block (single +1 term) or a slot in the workspace of
// summed operands, with its terms listed in ascending (R, C) block order.
template <int L>
struct LcmaPlan {
  static constexpr int G = 1 << L;
  static constexpr int R = ipow(7, L);
  static constexpr int kMaxTerms = ipow(2, L);   // at most 2 terms per level

  struct Side {
    int nslots = 0;
    int slot[R] = {};           // workspace slot of product p, or -1 for an alias
    int alias_r[R] = {};        // alias: raw block row
    int alias_c[R] = {};        // alias: raw block column
    int nterm[R] = {};
    int term_r[R][kMaxTerms] = {};
    int term_c[R][kMaxTerms] = {};
    int term_s[R][kMaxTerms] = {};
  };
  Side side[2] = {};

  constexpr LcmaPlan() {
    for (int w = 0; w < 2; ++w) {
      Side& s = side[w];
      for (int p = 0; p < R; ++p) {
        int n = 0;
        for (int r = 0; r < G; ++r)
          for (int c = 0; c < G; ++c) {
            const int v = coef(w, L, p, r, c);
            if (v != 0) {
              s.term_r[p][n] = r;
              s.term_c[p][n] = c;
              s.term_s[p][n] = v;
              ++n;
            }
          }
        s.nterm[p] = n;
        if (n == 1 && s.term_s[p][0] == 1) {
          s.slot[p] = -1;
          s.alias_r[p] = s.term_r[p][0];
          s.alias_c[p] = s.term_c[p][0];
        } else {
          s.slot[p] = s.nslots++;
        }
      }
    }
  }
};

// W as a dense compile-time table: w[R][C][p].
template <int L>
struct WTable {
  static constexpr int G = 1 << L;
  static constexpr int R = ipow(7, L);
  int w[G][G][R] = {};
  constexpr WTable() {
    for (int r = 0; r < G; ++r)
      for (int c = 0; c < G; ++c)
        for (int p = 0; p < R; ++p) w[r][c][p] = wcoef(L, r, c, p);
  }
};
}  // namespace lcg
