// Fused LCMA kernel (one-level Strassen): the 7 product tiles of one output
// coordinate run as one Group on one CTA and are recombined into the four
// quadrants of C in tensor memory, with a single cast on the way out.
//
// FalconGEMM write-up (hyper.ai news 54396, section "从 LCMA 到 FalconGEMM"):
// grouping the product tiles that share an output coordinate onto one SM lets
// a Group add its products into C on chip -- no intermediate products in
// global memory, no atomics between SMs (parallelising over products would
// need them) and no recomputation (parallelising over C blocks would repeat
// products).  The kernel is persistent so that the order of Groups and of the
// products inside them is under the kernel's control (same section, persistent
// kernel paragraph); every CTA walks its Groups' products in the same order,
// so a wave of CTAs works on one product type at a time and shares its
// operand panels in L2 (cache-reordering paragraph).  Numerics: products are
// accumulated in FP32 and the four quadrants are combined in FP32, then cast
// once (numerics paragraph).
//
// Tensor memory holds four 128 x 128 FP32 buffers (all 512 columns).  The
// product order M5, M3, M7, M1, M4, M2, M6 retires C12 after the second
// product and keeps at most three quadrants live, so one buffer is always
// free for the next product and the tensor core never waits for the
// epilogue once K is large enough:
//
//   step  product -> buffer     epilogue work after the product completes
//   0     M5 -> b0 (fresh)      b2 = -b0
//   1     M3 -> b1 (fresh)      b0 += b1; store b0 as C12
//   2     M7 -> b2 (accumulate)
//   3     M1 -> b3 (fresh)      b2 += b3; b1 += b3
//   4     M4 -> b0 (fresh)      b2 += b0; store b2 as C11
//   5     M2 -> b3 (fresh)      b0 += b3; store b0 as C21; b1 -= b3
//   6     M6 -> b2 (fresh)      b1 += b2; store b1 as C22
//
// Warp roles as in the plain kernel: warp 0 TMA producer, warp 1 TMEM owner
// and MMA issuer, warps 2..5 epilogue (TMEM read-modify-write and stores).
// The MMA issuer waits on per-warp epilogue progress counters before reusing
// a buffer; the epilogue waits on one mbarrier per product step.
#include "kernels.h"
#include "lcma_tables.h"
#include "ptx.cuh"

namespace lcg {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kTileBytes = kBM * kBK * 2;             // A and B tiles are both 128 x 64
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kTmemCols = 512;
constexpr int kSmemBytes = kStages * kStageBytes + 512 + 1024;

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

template <bool BF16>
__device__ __forceinline__ void store_quadrant(uint32_t tsrc, const LcmaArgs& a, int quad, int mb, int nb, int q,
                                               int lane) {
  const int qr = quad >> 1, qc = quad & 1;
  const int rloc = mb * kBM + q * 32 + lane;      // row inside the quadrant
  uint16_t* Cp = static_cast<uint16_t*>(a.C);
  uint16_t* crow = Cp + (static_cast<int64_t>(qr) * a.mb + rloc) * a.ldc + static_cast<int64_t>(qc) * a.nb;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tsrc + c * 32, r);
    tmem_wait_ld();
    const int col = nb * kBN + c * 32;
    if (rloc < a.mb && col < a.nb) {
      const bool vec = (col + 32 <= a.nb) && ((reinterpret_cast<uintptr_t>(crow + col) & 15u) == 0);
      if (vec) {
        uint4* dst = reinterpret_cast<uint4*>(crow + col);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 o;
          o.x = pack2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]), BF16);
          o.y = pack2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]), BF16);
          o.z = pack2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]), BF16);
          o.w = pack2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]), BF16);
          dst[v] = o;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const uint32_t p = pack2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), BF16);
          if (col + j < a.nb) crow[col + j] = static_cast<uint16_t>(p & 0xffffu);
          if (col + j + 1 < a.nb) crow[col + j + 1] = static_cast<uint16_t>(p >> 16);
        }
      }
    }
  }
}

// dst (+)= sign * src over one warp's 32 lanes x 128 columns.
__device__ __forceinline__ void combine_buffers(uint32_t tdst, uint32_t tsrc, float sign, bool add) {
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
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

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    lcma1_fused_kernel(const __grid_constant__ CUtensorMap tmA_sum, const __grid_constant__ CUtensorMap tmA_raw,
                       const __grid_constant__ CUtensorMap tmB_sum, const __grid_constant__ CUtensorMap tmB_raw,
                       const LcmaArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kTileBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* mdone = bars + 2 * kStages;          // one per program step
  uint64_t* drain = mdone + kSteps;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* progress = tmem_slot + 1;            // [4]: epilogue ops completed, per epilogue warp
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 5);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kSteps; ++s) mbar_init(&mdone[s], 1);
    mbar_init(drain, 1);
    for (int w = 0; w < 4; ++w) progress[w] = 0;
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA_sum);
    prefetch_tensormap(&tmA_raw);
    prefetch_tensormap(&tmB_sum);
    prefetch_tensormap(&tmB_raw);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, args.err, args.timeout_ns};
  const int num_kb = (args.kb + kBK - 1) / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < args.num_groups; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, args, mb, nb);
        for (int s = 0; ok && s < kSteps; ++s) {
          const int p = d_step_product[s];
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            load_operand(sA + stage * kTileBytes, &tmA_sum, &tmA_raw, args.a_src[p], &full[stage], kb * kBK,
                         mb * kBM);
            load_operand(sB + stage * kTileBytes, &tmB_sum, &tmB_raw, args.b_src[p], &full[stage], kb * kBK,
                         nb * kBN);
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
        for (int s = 0; s < kStages; ++s)
          if (armed >> s & 1u) mbar_wait(&full[s], (armed_par >> s) & 1u, wc, false);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BF16, kBM, kBN);
      uint32_t stage = 0, phase = 0, g = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; ok && t < args.num_groups; t += gridDim.x, ++g) {
        for (int s = 0; ok && s < kSteps; ++s) {
          const int need = static_cast<int>(g) * kNumOps + d_step_need[s];
          if (need > 0 && !wait_counter(progress, static_cast<uint32_t>(need), wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + d_step_buf[s] * kBN;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&full[stage], phase, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + stage * kTileBytes);
            const uint32_t b0 = smem_u32(sB + stage * kTileBytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_f16(d_tmem, sdesc_k128(a0 + k * 32), sdesc_k128(b0 + k * 32), idesc,
                      (d_step_fresh[s] && kb == 0 && k == 0) ? 0u : 1u);
            mma_commit(&empty[stage]);
            issued = true;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (ok && d_step_has_ops[s]) mma_commit(&mdone[s]);
        }
      }
      if (!ok && issued) {
        mma_commit(drain);
        mbar_wait(drain, 0, wc, false);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t g = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < args.num_groups; t += gridDim.x, ++g) {
      int mb, nb;
      tile_coords(t, args, mb, nb);
      int waited = -1;
      for (int i = 0; i < kNumOps; ++i) {
        const Op o = d_ops[i];
        if (o.after != waited) {
          ok = __all_sync(0xffffffffu, mbar_wait(&mdone[o.after], g & 1u, wc));
          if (!ok) break;
          tc_fence_after();
          waited = o.after;
        }
        if (o.kind == kOpStore) {
          store_quadrant<BF16>(lane_base + o.src * kBN, args, o.quad, mb, nb, q, lane);
        } else {
          combine_buffers(lane_base + o.dst * kBN, lane_base + o.src * kBN, static_cast<float>(o.sign),
                          o.kind == kOpAdd);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) red_release_add(progress + q, 1u);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- unfused products (ablation)
//
// The basic pipeline's middle step: every product P_p = A~_p . B~_p is a
// separate GEMM tile stream whose FP32 result goes to HBM; a recombination
// kernel forms C afterwards.  Work unit = (product, 128 x 128 tile); two TMEM
// accumulators let the FP32 store of one unit overlap the next unit's K loop.
__global__ void __launch_bounds__(kThreads, 1)
    lcma_products_kernel(const __grid_constant__ CUtensorMap tmA_sum, const __grid_constant__ CUtensorMap tmA_raw,
                         const __grid_constant__ CUtensorMap tmB_sum, const __grid_constant__ CUtensorMap tmB_raw,
                         const LcmaArgs args, const bool bf16) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kTileBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int units_per_p = args.tiles_m * args.tiles_n;
  const int num_units = units_per_p * args.num_products;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, args.err, args.timeout_ns};
  const int num_kb = (args.kb + kBK - 1) / kBK;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const int p = u / units_per_p;
        int mb, nb;
        tile_coords(u - p * units_per_p, args, mb, nb);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          load_operand(sA + stage * kTileBytes, &tmA_sum, &tmA_raw, args.a_src[p], &full[stage], kb * kBK, mb * kBM);
          load_operand(sB + stage * kTileBytes, &tmB_sum, &tmB_raw, args.b_src[p], &full[stage], kb * kBK, nb * kBN);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < kStages; ++s)
          if (armed >> s & 1u) mbar_wait(&full[s], (armed_par >> s) & 1u, wc, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(bf16, kBM, kBN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kTileBytes);
          const uint32_t b0 = smem_u32(sB + stage * kTileBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_f16(d_tmem, sdesc_k128(a0 + k * 32), sdesc_k128(b0 + k * 32), idesc, (kb | k) != 0);
          mma_commit(&empty[stage]);
          issued = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok && issued) {
        mma_commit(drain);
        mbar_wait(drain, 0, wc, false);
      }
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const int p = u / units_per_p;
      int mb, nb;
      tile_coords(u - p * units_per_p, args, mb, nb);
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, wc))) break;
      tc_fence_after();
      const int row = mb * kBM + q * 32 + lane;
      float* prow = args.prod + (static_cast<int64_t>(p) * args.mb + row) * args.ldp;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + c * 32, r);
        tmem_wait_ld();
        const int col = nb * kBN + c * 32;
        if (row < args.mb && col < args.nb) {
          if (col + 32 <= args.nb) {
            uint4* dst = reinterpret_cast<uint4*>(prow + col);
#pragma unroll
            for (int v = 0; v < 8; ++v) dst[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col + j < args.nb) prow[col + j] = __uint_as_float(r[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

template <bool BF16>
cudaError_t launch_impl(const LcmaLaunch& L, cudaStream_t st) {
  auto kern = lcma1_fused_kernel<BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<L.grid, kThreads, kSmemBytes, st>>>(L.tmA_sum, L.tmA_raw, L.tmB_sum, L.tmB_raw, L.args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lcma_fused(const LcmaLaunch& L, cudaStream_t st) {
  if (L.levels != 1) return cudaErrorInvalidValue;
  return L.bf16 ? launch_impl<true>(L, st) : launch_impl<false>(L, st);
}

cudaError_t launch_lcma_products(const LcmaLaunch& L, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(lcma_products_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  lcma_products_kernel<<<L.grid, kThreads, kSmemBytes, st>>>(L.tmA_sum, L.tmA_raw, L.tmB_sum, L.tmB_raw, L.args,
                                                              L.bf16);
  return cudaGetLastError();
}

}  // namespace lcg
