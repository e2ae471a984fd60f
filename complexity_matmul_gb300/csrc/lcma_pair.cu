// Fused one-level LCMA kernel on CTA pairs (cta_group::2) with 256 x 256
// Group tiles.
//
// A Group is the 7 product tiles of one 256 x 256 coordinate of the quadrant
// grid (FalconGEMM write-up, section "从 LCMA 到 FalconGEMM": the same-position
// tiles of the 7 batched products run together on one unit and are combined
// into C there, with no product written to HBM and no atomics).  Each product
// is one 256 x 256 MMA stream (M = 256 over the pair, N = 256): the same
// operand footprint per flop as the plain CTA-pair kernel, half the shared-
// memory traffic of 128-wide product tiles, which is what limits those.
//
// Tensor memory holds two 256-column accumulators (all 512 columns); the MMA
// writes them alternately, so product p+1 runs while the epilogue consumes
// product p.  Two products go straight onto the accumulator two steps back
// instead of into a fresh one: M7 (negated through the instruction's negate-A
// bit) onto M5 and M6 onto M3, so the accumulator already holds the sum that a
// C quadrant needs.  What is left of the quadrant sums lives in FP32 in a
// per-CTA scratch of two slots that stays in L2:
//
//   step  MMA                 epilogue (P = the accumulator, FP32)   slots after it
//   0     M5         -> X     s0  = P                               s0=C12
//   1     M3         -> Y     C12 = s0 + P (cast, stored)
//   2     X += -M7  (M5-M7)   s0  = -P                              s0=C11
//   3     Y += M6   (M3+M6)   s1  = P                               s1=C22
//   4     M1         -> X     s0 += P ;  s1 += P
//   5     M4         -> Y     C11 = s0 + P (stored) ;  s0 = P       s0=C21
//   6     M2         -> X     C21 = s0 + P (stored) ;  C22 = s1 - P (stored)
//
// Twelve slot accesses per Group and CTA (six writes, six reads of 128 KB)
// where a fresh accumulator per product needs sixteen and three slots, so the
// scratch takes less of the L2 that the operand panels of a wave share.  Every
// quadrant is accumulated in FP32 and cast once (numerics paragraphs of the
// write-up's "从缓存重排到 Cost Model" section).  Each epilogue thread owns one
// accumulator row and 128 columns; the scratch is laid out column-major per
// slot so that a warp's 32 rows of one column are one 128-byte line.  Final
// quadrant values are cast into 32 x 32 shared-memory boxes (two per warp) and
// leave through tensor stores of per-quadrant maps of C.
//
// Cross-CTA synchronisation (as in the plain CTA-pair kernel):
//   full[s]   leader's; armed with both CTAs' bytes; both CTAs' copies complete on it
//   empty[s]  per CTA; the leader's MMA commit arrives on both
//   pfull[b]  per CTA; the leader's MMA commit arrives on both when accumulator b is done
//   pempty[b] leader's; all 16 epilogue warps of the pair arrive when b is consumed
#include "lcma_program.cuh"

namespace lcg {

namespace {

constexpr int kRows = 128;                       // accumulator rows per CTA (256 per pair)
constexpr int kTileN = 256;                      // Group tile width
constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kEpiWarps = 8;                     // two per TMEM lane quarter, 128 columns each
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kABytes = kRows * kBK * 2;         // 16 KB
constexpr int kBBytes = (kTileN / 2) * kBK * 2;  // 16 KB (this CTA's half of B)
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTxBytes = 2 * kStageBytes;
constexpr int kTmemCols = 2 * kTileN;
constexpr int kCBoxBytes = 32 * 32 * 2;                 // one 32 x 32 chunk of C on its way to a tensor store
constexpr int kCStageBytes = kEpiWarps * 2 * kCBoxBytes;  // two boxes per epilogue warp
constexpr int kSmemBytes = kStages * kStageBytes + kCStageBytes + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr int kSlots = 2;
constexpr int kSlotFloats = kRows * kTileN;      // one slot: 128 rows x 256 columns
constexpr int kSteps1 = 7;

// Epilogue work per product step: up to two targets.
//   kTgtInit   slot  = sign * P          kTgtAcc    slot += sign * P
//   kTgtFinal  C     = slot + sign * P   kTgtFinalPX C    = sign * P + partner
//   kTgtFinalSX C    = slot + partner
// where "partner" is the same slot of the CTA that ran the other half of a
// split Group.
enum : int { kTgtNone = 0, kTgtInit = 1, kTgtAcc = 2, kTgtFinal = 3, kTgtFinalPX = 4, kTgtFinalSX = 5 };
struct Target {
  int kind, slot, sign, quad;
};
// One product step: the product, whether its MMA accumulates onto the
// accumulator of two steps before (same buffer: the MMA alternates between the
// two) instead of starting it afresh, whether it negates A, and the epilogue.
struct StepOps {
  int product, onto, negate;
  Target t[2];
};

// Work item types: a whole Group, or one of the two halves of a split Group
// (FalconGEMM write-up, "从 LCMA 到 FalconGEMM": a Group may be split over two
// units; scheduling stays per Group, execution per tile).
// kItemFullMixed is a whole Group in another product order; with Group
// ordering off, odd pairs run it, so that every wave mixes two product types
// (the effect the write-up's reordering removes).
enum : int { kItemFull = 0, kItemFirst = 1, kItemSecond = 2, kItemFullMixed = 3 };
constexpr int kItemTypes = 4;
constexpr int kItemSteps[kItemTypes] = {7, 4, 3, 7};

#define LCG_NONE {kTgtNone, 0, 0, 0}
#define LCG_L2_PROGRAMS                                                                                     \
  {                                                                                                         \
    {/* whole Group */                                                                                      \
     {4, 0, 0, {{kTgtInit, 0, 1, 1}, LCG_NONE}},                  /* M5: s0 = M5 (C12) */                   \
     {2, 0, 0, {{kTgtFinal, 0, 1, 1}, LCG_NONE}},                 /* M3: C12 = s0 + M3 */                   \
     {6, 1, 1, {{kTgtInit, 0, -1, 0}, LCG_NONE}},                 /* M5 - M7: s0 = M7 - M5 (C11) */         \
     {5, 1, 0, {{kTgtInit, 1, 1, 3}, LCG_NONE}},                  /* M3 + M6: s1 = M3 + M6 (C22) */         \
     {0, 0, 0, {{kTgtAcc, 0, 1, 0}, {kTgtAcc, 1, 1, 3}}},         /* M1: s0 += M1, s1 += M1 */              \
     {3, 0, 0, {{kTgtFinal, 0, 1, 0}, {kTgtInit, 0, 1, 2}}},      /* M4: C11 = s0 + M4; s0 = M4 (C21) */    \
     {1, 0, 0, {{kTgtFinal, 0, 1, 2}, {kTgtFinal, 1, -1, 3}}}},   /* M2: C21 = s0 + M2; C22 = s1 - M2 */    \
    {/* first half: M5 M3 M7 M6; finishes C12, and C11, C22 with the second half's partials */            \
     {4, 0, 0, {{kTgtInit, 0, 1, 1}, LCG_NONE}},                                                            \
     {2, 0, 0, {{kTgtFinal, 0, 1, 1}, LCG_NONE}},                                                           \
     {6, 1, 1, {{kTgtInit, 0, -1, 0}, LCG_NONE}},                                                           \
     {5, 1, 0, {{kTgtFinalPX, 1, 1, 3}, {kTgtFinalSX, 0, 1, 0}}}, /* C22 = M3+M6 + p1, C11 = s0 + p0 */     \
     {0, 0, 0, {LCG_NONE, LCG_NONE}},                                                                       \
     {0, 0, 0, {LCG_NONE, LCG_NONE}},                                                                       \
     {0, 0, 0, {LCG_NONE, LCG_NONE}}},                                                                      \
    {/* second half: M4 M2 M1; finishes C21, publishes p0 = M4 + M1 (C11) and p1 = M1 - M2 (C22) */        \
     {3, 0, 0, {{kTgtInit, 0, 1, 0}, {kTgtInit, 1, 1, 2}}},                                                 \
     {1, 0, 0, {{kTgtFinal, 1, 1, 2}, {kTgtInit, 1, -1, 3}}},                                               \
     {0, 0, 0, {{kTgtAcc, 0, 1, 0}, {kTgtAcc, 1, 1, 3}}},                                                   \
     {0, 0, 0, {LCG_NONE, LCG_NONE}},                                                                       \
     {0, 0, 0, {LCG_NONE, LCG_NONE}},                                                                       \
     {0, 0, 0, {LCG_NONE, LCG_NONE}},                                                                       \
     {0, 0, 0, {LCG_NONE, LCG_NONE}}},                                                                      \
    {/* whole Group, product order M3 M5 M6 M7 M1 M4 M2 */                                                 \
     {2, 0, 0, {{kTgtInit, 0, 1, 1}, LCG_NONE}},                  /* M3: s0 = M3 (C12) */                   \
     {4, 0, 0, {{kTgtFinal, 0, 1, 1}, LCG_NONE}},                 /* M5: C12 = s0 + M5 */                   \
     {5, 1, 0, {{kTgtInit, 0, 1, 3}, LCG_NONE}},                  /* M3 + M6: s0 = M3 + M6 (C22) */         \
     {6, 1, 1, {{kTgtInit, 1, -1, 0}, LCG_NONE}},                 /* M5 - M7: s1 = M7 - M5 (C11) */         \
     {0, 0, 0, {{kTgtAcc, 0, 1, 3}, {kTgtAcc, 1, 1, 0}}},         /* M1: s0 += M1, s1 += M1 */              \
     {3, 0, 0, {{kTgtFinal, 1, 1, 0}, {kTgtInit, 1, 1, 2}}},      /* M4: C11 = s1 + M4; s1 = M4 (C21) */    \
     {1, 0, 0, {{kTgtFinal, 1, 1, 2}, {kTgtFinal, 0, -1, 3}}}},   /* M2: C21 = s1 + M2; C22 = s0 - M2 */    \
  }
constexpr StepOps kL2Programs[kItemTypes][kSteps1] = LCG_L2_PROGRAMS;

// Symbolic run of the programs at compile time (coefficients over M1..M7):
// every item type stores each of its quadrants once, an accumulator is only
// continued within the item that started it, a slot is only read after this
// item wrote it, and together the two halves of a split Group produce exactly
// C_q = sum_p W[q,p] M_p for all four quadrants.
struct L2ProgramCheck {
  bool ok = true;
  constexpr void run(int type, int (&slot)[kSlots][7], int (&stored)[4][7], bool (&done)[4],
                     const int (&partner)[kSlots][7]) {
    int acc[2][7] = {};
    bool written[kSlots] = {};
    for (int s = 0; s < kItemSteps[type]; ++s) {
      const StepOps& st = kL2Programs[type][s];
      int* P = acc[s & 1];
      if (st.onto && s < 2) ok = false;                 // continues an accumulator of another item
      if (!st.onto)
        for (int j = 0; j < 7; ++j) P[j] = 0;
      P[st.product] += st.negate ? -1 : 1;
      for (int i = 0; i < 2; ++i) {
        const Target t = st.t[i];
        const bool reads_slot = t.kind == kTgtAcc || t.kind == kTgtFinal || t.kind == kTgtFinalSX;
        if (t.kind != kTgtNone && (t.slot < 0 || t.slot >= kSlots)) {
          ok = false;
          continue;
        }
        if (reads_slot && !written[t.slot]) ok = false;
        if (t.kind == kTgtInit) {
          for (int j = 0; j < 7; ++j) slot[t.slot][j] = t.sign * P[j];
          written[t.slot] = true;
        } else if (t.kind == kTgtAcc) {
          for (int j = 0; j < 7; ++j) slot[t.slot][j] += t.sign * P[j];
        } else if (t.kind >= kTgtFinal) {
          for (int j = 0; j < 7; ++j) {
            const int from_slot = (t.kind == kTgtFinal || t.kind == kTgtFinalSX) ? slot[t.slot][j] : 0;
            const int from_p = (t.kind == kTgtFinalSX) ? 0 : t.sign * P[j];
            const int from_partner = (t.kind == kTgtFinalPX || t.kind == kTgtFinalSX) ? partner[t.slot][j] : 0;
            stored[t.quad][j] = from_slot + from_p + from_partner;
          }
          if (done[t.quad]) ok = false;
          done[t.quad] = true;
        }
      }
      // a step's two targets run chunk by chunk (target 0, then target 1): an Init
      // must not precede a read of the same slot in the same step
      if (st.t[0].kind == kTgtInit && st.t[1].kind != kTgtNone && st.t[1].kind != kTgtInit &&
          st.t[1].kind != kTgtFinalPX && st.t[0].slot == st.t[1].slot)
        ok = false;
    }
  }
  constexpr L2ProgramCheck() {
    const int none[kSlots][7] = {};
    {
      int slot[kSlots][7] = {};
      int stored[4][7] = {};
      bool done[4] = {false, false, false, false};
      run(kItemFull, slot, stored, done, none);
      for (int q = 0; q < 4; ++q) {
        if (!done[q]) ok = false;
        for (int j = 0; j < 7; ++j)
          if (stored[q][j] != kW1[q][j]) ok = false;
      }
    }
    {
      int slot[kSlots][7] = {};
      int stored[4][7] = {};
      bool done[4] = {false, false, false, false};
      run(kItemFullMixed, slot, stored, done, none);
      for (int q = 0; q < 4; ++q) {
        if (!done[q]) ok = false;
        for (int j = 0; j < 7; ++j)
          if (stored[q][j] != kW1[q][j]) ok = false;
      }
    }
    {
      int slot2[kSlots][7] = {};
      int stored[4][7] = {};
      bool done[4] = {false, false, false, false};
      run(kItemSecond, slot2, stored, done, none);      // publishes slot2[0], slot2[1]
      int slot1[kSlots][7] = {};
      run(kItemFirst, slot1, stored, done, slot2);
      for (int q = 0; q < 4; ++q) {
        if (!done[q]) ok = false;
        for (int j = 0; j < 7; ++j)
          if (stored[q][j] != kW1[q][j]) ok = false;
      }
    }
  }
};
static_assert(L2ProgramCheck{}.ok, "the L2-accumulating programs must compute C_q = sum_p W[q,p] M_p");

__constant__ StepOps d_l2_programs[kItemTypes][kSteps1] = LCG_L2_PROGRAMS;
__constant__ int d_item_steps[kItemTypes] = {7, 4, 3, 7};

// Work item w of this launch -> Group index and item type.
// With Group ordering on, every pair walks its whole Groups in one product
// order, so the pairs of a wave stream one product's operand panels at a time;
// off, the odd pairs (w % num_pairs) take the other order.
__device__ __forceinline__ void item_of(int w, const LcmaArgs& a, int num_pairs, int& group, int& type) {
  if (w < a.split_first) {
    group = w;
    type = (!a.group_order && ((w % num_pairs) & 1)) ? kItemFullMixed : kItemFull;
  } else {
    const int i = (w - a.split_first) >> 1;
    group = a.split_first + i;
    type = ((w - a.split_first) & 1) ? kItemSecond : kItemFirst;
  }
}

// Operand tiles through 2-D maps (cheaper for the copy engine than 3-D / 4-D
// boxes): summed operands as one (slots * rows_b) x kb matrix, and raw blocks
// as the whole operand when raw2d is set (the block width kb is a multiple of
// the 64-deep slab, so a slab never reaches into the next block); otherwise raw
// blocks through the exact 4-D block map.  Rows past a block's end belong to
// output rows outside C and are never stored.
__device__ __forceinline__ void load_operand_pair(void* dst, const CUtensorMap* sum_map, const CUtensorMap* raw_map,
                                                  const LcmaOperand& src, uint32_t bar, int k0, int row0, int rows_b,
                                                  int kb, bool raw2d) {
  if (src.slot >= 0)
    tma_load_2d_pair(dst, sum_map, bar, k0, src.slot * rows_b + row0);
  else if (raw2d)
    tma_load_2d_pair(dst, raw_map, bar, src.c * kb + k0, src.r * rows_b + row0);
  else
    tma_load_4d_pair(dst, raw_map, bar, k0, src.c, row0, src.r);
}

__device__ __forceinline__ void tile_coords_l2(int t, const LcmaArgs& a, int& mb, int& nb) {
  const int group_tiles = a.group_m * a.tiles_n;
  const int g = t / group_tiles;
  const int first_m = g * a.group_m;
  const int rows = min(a.tiles_m - first_m, a.group_m);
  const int local = t - g * group_tiles;
  mb = first_m + local % rows;
  nb = local / rows;
}

// The quadrant scratch is read back within a few products: its stores and loads
// carry an L2 evict-last policy so that the operand panels streaming through L2
// push it out last; lines of a slot that is dead until the next Group rewrites
// it are dropped without a write-back (discard), by lane 0 of the warp that owns
// them, between two __syncwarp barriers (the warp's loads of them are complete
// before, and its later stores to them come after).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_keep(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ float ld_keep(const float* p, uint64_t pol) {
  float v;
  asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol) : "memory");
  return v;
}
__device__ __forceinline__ void discard_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Two levels: 32 FP32 values (one row, columns qcol .. qcol+31) of inner
// quadrant `iq` of this launch's outer product P go to the outer level: into an
// outer slot (Init / Acc), or, with the slot's sum, into outer quadrant q of C
// (Final: epilogue, one cast).  Row rloc < mbp and column qcol < nbp always lie
// inside the padded slots; only C's stores are bounded by its extents.
template <bool BF16>
__device__ __forceinline__ void apply_outer(const float (&v)[32], int iq, int rloc, int qcol, const LcmaArgs& a) {
  const int ri = iq >> 1, ci = iq & 1;
  const int pr = ri * a.mbp + rloc;                      // row of P (and of every outer slot)
  const int pc = ci * a.nbp + qcol;
  const int64_t slot_floats = static_cast<int64_t>(2 * a.mbp) * (2 * a.nbp);
  const int64_t off = (static_cast<int64_t>(pr >> 7) * (2 * a.nbp) + pc) * 128 + (pr & 127);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const LcmaOuterTarget t = a.otgt[i];
    if (t.kind == kOuterNone) continue;
    float* sp = a.oslot + t.slot * slot_floats + off;
    const float sg = static_cast<float>(t.sign);
    if (t.kind == kOuterInit) {
#pragma unroll
      for (int j = 0; j < 32; ++j) sp[j * 128] = sg * v[j];
    } else if (t.kind == kOuterAcc) {
      float w[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = sp[j * 128];
#pragma unroll
      for (int j = 0; j < 32; ++j) sp[j * 128] = w[j] + sg * v[j];
    } else {
      float w[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = sp[j * 128] + sg * v[j];
      const int qr = t.quad >> 1, qc = t.quad & 1;
      const int64_t row = static_cast<int64_t>(qr) * 2 * a.mb + static_cast<int64_t>(ri) * a.mb + rloc;
      const int64_t col = static_cast<int64_t>(qc) * 2 * a.nb + static_cast<int64_t>(ci) * a.nb + qcol;
      if (rloc < a.mb && qcol < a.nb && row < a.M && col < a.N)
        store_run<BF16, 32>(static_cast<uint16_t*>(a.C) + row * a.ldc + col, row, col,
                            min(min(32, a.nb - qcol), static_cast<int>(a.N - col)), w, a.ep);
    }
  }
}

// Consume one product held in TMEM (this thread: one row, 128 columns) into
// the scratch slots / C according to the step's targets.
// `col0`: first of this thread's 128 columns inside the tile; `tile_col0`: the
// tile's first column inside the quadrant; `rloc`: this thread's quadrant row.
// Final values: with `a.c_tma`, cast into one of the warp's two shared-memory
// boxes (`sbox`, taken in turn by `nbox`) and written by a tensor store of
// quadrant map t.quad at (column, `row0q` = the warp's first quadrant row), so
// that a warp's store moves whole lines instead of one 16-byte piece of 32 rows.
template <bool BF16>
__device__ __forceinline__ void consume_product(uint32_t tsrc, const StepOps& st, float* scratch, int row,
                                                const LcmaArgs& a, int rloc, int col0, int tile_col0,
                                                const float* partner, bool last_step, const QuadMaps* tmC,
                                                uint32_t sbox, uint32_t& nbox, int row0q) {
  uint16_t* Cp = static_cast<uint16_t*>(a.C);
  const uint64_t pol = l2_policy_evict_last();
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tsrc + c * 32, r);
    tmem_wait_ld();
    const int col = col0 + c * 32;   // column inside the 256-wide tile
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const Target t = st.t[i];
      if (t.kind == kTgtNone) continue;
      float* sp = scratch + (static_cast<int64_t>(t.slot) * kTileN + col) * kRows + row;
      const float sg = static_cast<float>(t.sign);
      if (t.kind == kTgtInit) {
#pragma unroll
        for (int j = 0; j < 32; ++j) st_keep(sp + j * kRows, sg * __uint_as_float(r[j]), pol);
      } else if (t.kind == kTgtAcc) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = ld_keep(sp + j * kRows, pol);
#pragma unroll
        for (int j = 0; j < 32; ++j) st_keep(sp + j * kRows, v[j] + sg * __uint_as_float(r[j]), pol);
      } else {
        float v[32];
        if (t.kind == kTgtFinalPX) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = sg * __uint_as_float(r[j]);
        } else if (t.kind == kTgtFinalSX) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = ld_keep(sp + j * kRows, pol);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = ld_keep(sp + j * kRows, pol) + sg * __uint_as_float(r[j]);
        }
        if (t.kind == kTgtFinalPX || t.kind == kTgtFinalSX) {
          const float* pp = partner + (static_cast<int64_t>(t.slot) * kTileN + col) * kRows + row;
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += __ldcg(pp + j * kRows);
        }
        if (last_step && t.kind != kTgtFinalPX) {
          // the slot is dead until the next Group writes it again
          __syncwarp();
          if ((threadIdx.x & 31) == 0) {
            const float* line = sp - (row & 31);     // this warp's 32 rows of column col
#pragma unroll 4
            for (int j = 0; j < 32; ++j) discard_line(line + j * kRows);
          }
          __syncwarp();
        }
        const int qcol = tile_col0 + col;              // column inside the quadrant
        if (a.outer) {
          apply_outer<BF16>(v, t.quad, rloc, qcol, a);
        } else {
          // epilogue, cast once and store into quadrant t.quad of C
          const int qr = t.quad >> 1, qc = t.quad & 1;
          const int64_t crow_i = static_cast<int64_t>(qr) * a.mb + rloc;
          uint16_t* crow = Cp + crow_i * a.ldc + static_cast<int64_t>(qc) * a.nb;
          const int64_t gcol = static_cast<int64_t>(qc) * a.nb + qcol;
          const bool inside = rloc < a.mb && qcol < a.nb && crow_i < a.M && gcol < a.N;
          const int n = min(min(32, a.nb - qcol), static_cast<int>(a.N - gcol));
          if (a.c_tma) {
            if (inside) apply_epilogue<BF16, 32>(crow_i, gcol, n, v, a.ep);
            const int lane = threadIdx.x & 31;
            const uint32_t box = sbox + (nbox++ & 1u) * kCBoxBytes;
            if (lane == 0) bulk_wait_read<1>();   // the store that read this box two chunks ago is done with it
            __syncwarp();
            stage_chunk<BF16>(box, lane, v);
            fence_proxy_async_shared();
            __syncwarp();
            // the map clips rows past the quadrant's part of C and ends at its last whole
            // 16-byte unit of a row; the columns after it are stored from registers
            const int qcols = min(a.nb, a.N - qc * a.nb), qcols8 = qcols & ~7;
            if (lane == 0) {
              if (row0q < min(a.mb, a.M - qr * a.mb) && qcol < qcols8) tma_store_2d(&tmC->q[t.quad], box, qcol, row0q);
              bulk_commit();
            }
            if (qcol + 32 > qcols8 && qcol < qcols && rloc < a.mb && crow_i < a.M)
              store_cols<BF16>(crow + qcol, v, max(qcols8 - qcol, 0), min(qcols - qcol, 32));
          } else if (inside) {
            store_run<BF16, 32>(crow + qcol, crow_i, gcol, n, v, a.ep);
          }
        }
      }
    }
  }
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lcma1_l2_kernel(const __grid_constant__ CUtensorMap tmA_sum, const __grid_constant__ CUtensorMap tmA_raw,
                    const __grid_constant__ CUtensorMap tmB_sum, const __grid_constant__ CUtensorMap tmB_raw,
                    const __grid_constant__ QuadMaps tmC, const LcmaArgs args_in) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sC = sB + kStages * kBBytes;      // 1024-byte aligned: the stages are whole KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sC + kCStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* pfull = bars + 2 * kStages;
  uint64_t* pempty = pfull + 2;
  uint64_t* drain = pempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA_sum);
    prefetch_tensormap(&tmA_raw);
    prefetch_tensormap(&tmB_sum);
    prefetch_tensormap(&tmB_raw);
    if (args_in.c_tma)
      for (int q = 0; q < 4; ++q) prefetch_tensormap(&tmC.q[q]);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, args_in.err, args_in.timeout_ns};
  const int num_kb = (args_in.kb + kBK - 1) / kBK;
  const int pair = blockIdx.x / 2;
  const int num_pairs = gridDim.x / 2;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      griddep_wait();   // the summed operands come from the pre-pass kernel before this one
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int w = pair; ok && w < args_in.num_items; w += num_pairs) {
        int grp, type;
        item_of(w, args_in, num_pairs, grp, type);
        int mb, nb;
        tile_coords_l2(grp, args_in, mb, nb);
        const int nsteps = d_item_steps[type];
        for (int s = 0; ok && s < nsteps; ++s) {
          const int p = d_l2_programs[type][s].product;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&full[stage], kTxBytes);
            const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
            load_operand_pair(sA + stage * kABytes, &tmA_sum, &tmA_raw, args_in.a_src[p], bar, kb * kBK,
                              mb * 2 * kRows + static_cast<int>(rank) * kRows, args_in.mb, args_in.kb, args_in.raw2d);
            load_operand_pair(sB + stage * kBBytes, &tmB_sum, &tmB_raw, args_in.b_src[p], bar, kb * kBK,
                              nb * kTileN + static_cast<int>(rank) * (kTileN / 2), args_in.nb, args_in.kb, args_in.raw2d);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (!ok) {
        if (leader)
          for (int s = 0; s < kStages; ++s)
            if (armed >> s & 1u) mbar_wait(&full[s], (armed_par >> s) & 1u, wc, false);
        settle_ns(1000000);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc_pos = idesc_f16(BF16, 2 * kRows, kTileN);
      constexpr uint32_t idesc_neg = idesc_f16(BF16, 2 * kRows, kTileN, /*negate_a=*/true);
      const uint64_t a_desc0 = sdesc_k128(smem_u32(sA));
      const uint64_t b_desc0 = sdesc_k128(smem_u32(sB));
      uint32_t stage = 0, phase = 0, buf = 0, buf_phase = 0;
      bool ok = true, issued = false;
      for (int w = pair; ok && w < args_in.num_items; w += num_pairs) {
        int grp, type;
        item_of(w, args_in, num_pairs, grp, type);
        const int nsteps = d_item_steps[type];
        for (int s = 0; ok && s < nsteps; ++s) {
          if (!mbar_wait(&pempty[buf], buf_phase ^ 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kTileN;
          // continuing the accumulator of two steps before (same buffer), or starting it afresh
          const uint32_t onto = d_l2_programs[type][s].onto;
          const uint32_t idesc = d_l2_programs[type][s].negate ? idesc_neg : idesc_pos;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&full[stage], phase, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * kABytes) >> 4);
            const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * kBBytes) >> 4);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) mma_f16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, onto | ((kb | k) != 0));
            mma_commit_pair(&empty[stage]);
            issued = true;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          mma_commit_pair(&pfull[buf]);
          buf ^= 1;
          if (buf == 0) buf_phase ^= 1;
        }
      }
      if (!ok && issued) {
        mma_commit_pair(drain);
        mbar_wait(drain, 0, wc, false);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs, 8 warps)
    if (args_in.outer) griddep_wait();   // the outer slots come from the launch before this one
    const int ew = warp - 2;
    const int q = warp & 3;                 // TMEM lane quarter
    const int half = ew >> 2;               // which 128 of the 256 columns
    const int row = q * 32 + lane;          // accumulator row inside this CTA's 128
    float* scratch = args_in.scratch + static_cast<int64_t>(blockIdx.x) * kSlots * kSlotFloats;
    const uint32_t sbox = smem_u32(sC) + ew * 2 * kCBoxBytes;   // this warp's two boxes
    uint32_t nbox = 0;
    uint32_t buf = 0, buf_phase = 0;
    bool ok = true;
    for (int w = pair; ok && w < args_in.num_items; w += num_pairs) {
      int grp, type;
      item_of(w, args_in, num_pairs, grp, type);
      int mb, nb;
      tile_coords_l2(grp, args_in, mb, nb);
      const int rloc = mb * 2 * kRows + static_cast<int>(rank) * kRows + row;   // row inside the quadrant
      const int nsteps = d_item_steps[type];
      // split Groups: the halves meet through the second half's scratch and a counter
      const int split_idx = (w - args_in.split_first) >> 1;
      int* flag = type == kItemFull ? nullptr : args_in.flags + 2 * split_idx + static_cast<int>(rank);
      const float* partner = nullptr;
      if (type == kItemFirst) {
        const int partner_pair = (args_in.split_first + 2 * split_idx + 1) % num_pairs;
        partner = args_in.scratch + static_cast<int64_t>(2 * partner_pair + static_cast<int>(rank)) * kSlots * kSlotFloats;
      }
      for (int s = 0; s < nsteps; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(&pfull[buf], buf_phase, wc));
        if (!ok) break;
        tc_fence_after();
        if (type == kItemFirst && s == nsteps - 1) {
          // all 8 epilogue warps of the partner CTA with this rank have published (bounded wait)
          ok = __all_sync(0xffffffffu, wait_flag(flag, kEpiWarps, wc));
          if (!ok) break;
        }
        const uint32_t tsrc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kTileN + half * 128;
        // at the last step of a whole Group, the slots it reads are dead until the next Group
        consume_product<BF16>(tsrc, d_l2_programs[type][s], scratch, row, args_in, rloc, half * 128, nb * kTileN,
                              partner, s == nsteps - 1 && (type == kItemFull || type == kItemFullMixed), &tmC, sbox,
                              nbox, rloc - lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&pempty[buf]), 0));
        buf ^= 1;
        if (buf == 0) buf_phase ^= 1;
      }
      if (ok && type == kItemSecond) {
        // publish this warp's partial sums (slots 0 and 1) to the first half
        __threadfence();
        __syncwarp();
        if (lane == 0 && !args_in.debug_drop) red_release_gpu_add(flag, 1);
      }
    }
    if (lane == 0) bulk_wait_all();   // the tensor stores have read their boxes and written C
  }

  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <bool BF16>
cudaError_t launch_impl(const LcmaLaunch& L, cudaStream_t st) {
  auto kern = lcma1_l2_kernel<BF16>;
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return launch_maybe_pdl(kern, L.grid, kThreads, kSmemBytes, st, L.pdl, L.tmA_sum, L.tmA_raw, L.tmB_sum, L.tmB_raw,
                          L.tmC, L.args);
}

}  // namespace

size_t lcma_pair_scratch_bytes(int grid) { return static_cast<size_t>(grid) * kSlots * kSlotFloats * sizeof(float); }

cudaError_t launch_lcma_pair(const LcmaLaunch& L, cudaStream_t st) {
  if (L.levels != (L.args.outer ? 2 : 1) || L.grid % 2 || !L.args.scratch) return cudaErrorInvalidValue;
  if (L.args.outer && !L.args.oslot) return cudaErrorInvalidValue;
  return L.bf16 ? launch_impl<true>(L, st) : launch_impl<false>(L, st);
}

}  // namespace lcg
