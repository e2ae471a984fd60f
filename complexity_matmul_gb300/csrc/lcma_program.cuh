// The one-level fused LCMA program (product order, TMEM buffer use, epilogue
// ops) and the device helpers shared by the single-CTA and the CTA-pair fused
// kernels.  See lcma_fused.cu for the schedule and its rationale.
#pragma once

#include "epilogue.cuh"
#include "kernels.h"
#include "lcma_tables.h"
#include "ptx.cuh"

namespace lcg {
namespace {

constexpr int kBufCols = 128;   // TMEM columns per buffer = output tile width

// ---------------------------------------------------------------- the one-level program

constexpr int kSteps = 7;
#define LCG_STEP_PRODUCT {4, 2, 6, 0, 3, 1, 5} /* M5 M3 M7 M1 M4 M2 M6 (0-based) */
#define LCG_STEP_BUF {0, 1, 2, 3, 0, 3, 2}
#define LCG_STEP_FRESH {1, 1, 0, 1, 1, 1, 1}
constexpr int kStepProduct[kSteps] = LCG_STEP_PRODUCT;
constexpr int kStepBuf[kSteps] = LCG_STEP_BUF;
constexpr int kStepFresh[kSteps] = LCG_STEP_FRESH;

enum : int { kOpCopy = 0, kOpAdd = 1, kOpStore = 2 };
struct Op {
  int kind, dst, src, sign, quad, after;
};
constexpr int kNumOps = 12;
#define LCG_OPS                                                                                  \
  {                                                                                              \
    {kOpCopy, 2, 0, -1, -1, 0}, {kOpAdd, 0, 1, 1, -1, 1}, {kOpStore, -1, 0, 0, 1, 1},           \
        {kOpAdd, 2, 3, 1, -1, 3}, {kOpAdd, 1, 3, 1, -1, 3}, {kOpAdd, 2, 0, 1, -1, 4},            \
        {kOpStore, -1, 2, 0, 0, 4}, {kOpAdd, 0, 3, 1, -1, 5}, {kOpStore, -1, 0, 0, 2, 5},        \
        {kOpAdd, 1, 3, -1, -1, 5}, {kOpAdd, 1, 2, 1, -1, 6}, {kOpStore, -1, 1, 0, 3, 6},         \
  }
constexpr Op kOps[kNumOps] = LCG_OPS;

constexpr bool touches(const Op& o, int b) { return o.dst == b || o.src == b; }

// Epilogue ops that must be complete before MMA step s may write its buffer,
// as a count relative to kNumOps * (Group index): the last op touching the
// buffer that precedes step s (in this Group, or else in the previous one).
constexpr int step_need(int s) {
  int need = -1000000;
  for (int i = 0; i < kNumOps; ++i)
    if (kOps[i].after < s && touches(kOps[i], kStepBuf[s])) need = i + 1;
  if (need > -1000000) return need;
  for (int i = 0; i < kNumOps; ++i)
    if (touches(kOps[i], kStepBuf[s])) need = i + 1 - kNumOps;
  return need > -1000000 ? need : 0;
}

constexpr bool step_has_ops(int s) {
  for (int i = 0; i < kNumOps; ++i)
    if (kOps[i].after == s) return true;
  return false;
}

// The program computes C_q = sum_p W[q,p] M_p: checked symbolically at compile time.
struct ProgramCheck {
  bool ok = true;
  constexpr ProgramCheck() {
    int buf[4][7] = {};
    int stored[4][7] = {};
    bool done[4] = {false, false, false, false};
    int op = 0;
    for (int s = 0; s < kSteps; ++s) {
      const int b = kStepBuf[s];
      for (int p = 0; p < 7; ++p) buf[b][p] = kStepFresh[s] ? 0 : buf[b][p];
      buf[b][kStepProduct[s]] += 1;
      for (; op < kNumOps && kOps[op].after == s; ++op) {
        const Op& o = kOps[op];
        if (o.kind == kOpCopy)
          for (int p = 0; p < 7; ++p) buf[o.dst][p] = o.sign * buf[o.src][p];
        if (o.kind == kOpAdd)
          for (int p = 0; p < 7; ++p) buf[o.dst][p] += o.sign * buf[o.src][p];
        if (o.kind == kOpStore) {
          for (int p = 0; p < 7; ++p) stored[o.quad][p] = buf[o.src][p];
          if (done[o.quad]) ok = false;
          done[o.quad] = true;
        }
      }
    }
    for (int q = 0; q < 4; ++q) {
      if (!done[q]) ok = false;
      for (int p = 0; p < 7; ++p)
        if (stored[q][p] != kW1[q][p]) ok = false;
    }
    if (op != kNumOps) ok = false;
  }
};
static_assert(ProgramCheck{}.ok, "the fused one-level program must compute C_q = sum_p W[q,p] M_p");

// Device copies of the program (read uniformly by the role threads).
__constant__ int d_step_product[kSteps] = LCG_STEP_PRODUCT;
__constant__ int d_step_buf[kSteps] = LCG_STEP_BUF;
__constant__ int d_step_fresh[kSteps] = LCG_STEP_FRESH;
__constant__ int d_step_need[kSteps] = {step_need(0), step_need(1), step_need(2), step_need(3),
                                        step_need(4), step_need(5), step_need(6)};
__constant__ int d_step_has_ops[kSteps] = {step_has_ops(0), step_has_ops(1), step_has_ops(2), step_has_ops(3),
                                           step_has_ops(4), step_has_ops(5), step_has_ops(6)};
__constant__ Op d_ops[kNumOps] = LCG_OPS;

__device__ __forceinline__ void tile_coords(int t, const LcmaArgs& a, int& mb, int& nb) {
  const int group_tiles = a.group_m * a.tiles_n;
  const int g = t / group_tiles;
  const int first_m = g * a.group_m;
  const int rows = min(a.tiles_m - first_m, a.group_m);
  const int local = t - g * group_tiles;
  mb = first_m + local % rows;
  nb = local / rows;
}

__device__ __forceinline__ void load_operand(void* dst, const CUtensorMap* sum_map, const CUtensorMap* raw_map,
                                             const LcmaOperand& src, uint64_t* bar, int k0, int row0) {
  if (src.slot >= 0)
    tma_load_3d(dst, sum_map, bar, k0, row0, src.slot);
  else
    tma_load_4d(dst, raw_map, bar, k0, src.c, row0, src.r);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// The four epilogue warps advance independently (a warp with no rows inside C
// skips its stores and runs ahead), so each keeps its own count of finished
// ops; an op is complete once every warp's count has passed it.
__device__ __forceinline__ bool counters_reached(const uint32_t* ctr, uint32_t target) {
  return ld_acquire_u32(ctr) >= target && ld_acquire_u32(ctr + 1) >= target && ld_acquire_u32(ctr + 2) >= target &&
         ld_acquire_u32(ctr + 3) >= target;
}

// Bounded wait until all four counters ctr[0..3] >= target.
__device__ __forceinline__ bool wait_counter(const uint32_t* ctr, uint32_t target, const WaitCtl& w) {
  if (counters_reached(ctr, target)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (counters_reached(ctr, target)) return true;
    if ((i & 31u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        record_error(w, kErrWaitTimeout);
        return false;
      }
    }
  }
}

// Epilogue, cast and store of one warp's 32 rows x 128 columns of a TMEM
// buffer into quadrant `quad` of C.  `rloc`: this thread's row inside the
// quadrant; `col0`: the tile's first column inside the quadrant.
template <bool BF16>
__device__ __forceinline__ void store_quadrant(uint32_t tsrc, const LcmaArgs& a, int quad, int rloc, int col0) {
  const int qr = quad >> 1, qc = quad & 1;
  uint16_t* Cp = static_cast<uint16_t*>(a.C);
  const int64_t row = static_cast<int64_t>(qr) * a.mb + rloc;
  uint16_t* crow = Cp + row * a.ldc + static_cast<int64_t>(qc) * a.nb;
#pragma unroll 1
  for (int c = 0; c < kBufCols / 32; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tsrc + c * 32, r);
    tmem_wait_ld();
    const int col = col0 + c * 32;
    const int64_t gcol = static_cast<int64_t>(qc) * a.nb + col;
    if (rloc < a.mb && col < a.nb && row < a.M && gcol < a.N) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
      const int n = min(min(32, a.nb - col), static_cast<int>(a.N - gcol));
      store_run<BF16, 32>(crow + col, row, gcol, n, v, a.ep);
    }
  }
}

// dst (+)= sign * src over one warp's 32 lanes x 128 columns.
__device__ __forceinline__ void combine_buffers(uint32_t tdst, uint32_t tsrc, float sign, bool add) {
#pragma unroll 1
  for (int c = 0; c < kBufCols / 32; ++c) {
    uint32_t s[32], d[32];
    tmem_ld_32x32b_x32(tsrc + c * 32, s);
    if (add) tmem_ld_32x32b_x32(tdst + c * 32, d);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float v = sign * __uint_as_float(s[e]);
      d[e] = __float_as_uint(add ? __uint_as_float(d[e]) + v : v);
    }
    tmem_st_32x32b_x32(tdst + c * 32, d);
  }
  tmem_wait_st();
}

}  // namespace
}  // namespace lcg
