// Skinny GEMM for sm_103a (M <= 256: LLM decode and small-batch layers, where
// the weights B stream from HBM and the GEMM is bandwidth bound):
// C = A . B with every element of B read from HBM once.
//
// Orientation: the kernel computes D = B . A^T (N x M).  Each tcgen05.mma
// takes 128 rows of B as its M = 128 operand and all of A, its rows padded to
// MP by the TMA's zero fill, as its N = MP operand; one block's accumulator is
// 128 TMEM lanes (n) x MP columns (m).
//
// Work split (stream-K): the nblk x num_kb (128-row block of B, 64-deep K
// slab) iterations are cut into `grid` equal contiguous ranges, one per CTA,
// so every SM streams the same number of B bytes.  A CTA walks its range as
// segments of consecutive slabs of one block.  A segment that covers its whole
// block is stored directly; otherwise its FP32 partial goes to the workspace
// and, per block and 32-row quarter, the last CTA to arrive sums the block's
// partials in K order, applies the epilogue and stores.  Nobody waits for
// anybody; the arrival counters carry the launch's epoch in their high word,
// so they never need a reset.
//
// Warp roles as in the plain kernels: warp 0 TMA producer, warp 1 TMEM
// allocator and MMA issuer, warps 2..5 epilogue (warp w reads TMEM lanes
// 32 (w % 4) .. 32 (w % 4) + 31).
#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace lcg {

namespace {

constexpr int kRowsB = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;

// One pipeline stage holds SUB consecutive 64-deep K boxes of B and of A, so
// each row of B is fetched in runs of SUB x 128 contiguous bytes.
template <int MP, int SUB>
struct SkCfg {
  static constexpr int kBBox = kRowsB * kBK * 2;                   // 16 KB
  static constexpr int kABox = MP * kBK * 2;                       // 2 .. 32 KB
  static constexpr int kBBytes = SUB * kBBox;
  static constexpr int kABytes = SUB * kABox;
  static constexpr int kStageBytes = kBBytes + kABytes;
  static constexpr int kFit = 200 * 1024 / kStageBytes;
  static constexpr int kStages = kFit < 8 ? kFit : 8;
  static constexpr int kTmemCols = 2 * MP < 32 ? 32 : 2 * MP;      // two accumulators
  static constexpr int kCols = MP < 32 ? MP : 32;                  // columns per TMEM load
  static constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(MP % 16 == 0 && MP >= 16 && MP <= 256, "MMA N for M = 128");
};

__device__ __forceinline__ int64_t range_begin(int64_t c, int64_t total, int grid) { return c * total / grid; }

// The CTA whose range holds iteration i.
__device__ __forceinline__ int cta_of(int64_t i, int64_t total, int grid) {
  int64_t c = i * grid / total;
  while (c + 1 < grid && range_begin(c + 1, total, grid) <= i) ++c;
  while (c > 0 && range_begin(c, total, grid) > i) --c;
  return static_cast<int>(c);
}

__device__ __forceinline__ unsigned long long atom_cas_acq_rel(unsigned long long* p, unsigned long long cmp,
                                                               unsigned long long val) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;" : "=l"(old) : "l"(p), "l"(cmp), "l"(val) : "memory");
  return old;
}

// Counts one arrival on a counter tagged with `epoch` (a stale epoch counts as
// zero arrivals).  Returns the arrival number, or 0 if the bounded
// compare-and-swap loop gave up.
__device__ __forceinline__ unsigned int epoch_arrive(unsigned long long* p, unsigned int epoch) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(p);
  for (int tries = 0; tries < 4096; ++tries) {
    const unsigned long long base =
        static_cast<unsigned int>(old >> 32) == epoch ? old : static_cast<unsigned long long>(epoch) << 32;
    const unsigned long long want = base + 1;
    const unsigned long long seen = atom_cas_acq_rel(p, old, want);
    if (seen == old) return static_cast<unsigned int>(want & 0xffffffffu);
    old = seen;
  }
  return 0;
}

template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[W]) {
  if constexpr (W == 16) tmem_ld_32x32b_x16(taddr, r);
  else tmem_ld_32x32b_x32(taddr, r);
}

// Final values of C[m0 .. m0 + W) at column n from their FP32 sums (entries
// past M ignored): epilogue (bias_n already decoded), one rounding, store.
// The residual words are loaded for the whole run before the first store, so
// their latencies overlap.  ACT is the activation, fixed per call site.
template <bool BF16, int ACT, int W>
__device__ __forceinline__ void finish_run(const SkinnyArgs& a, int m0, int n, float (&v)[W], float bias_n) {
  float res[W];
  if (a.ep.residual) {
#pragma unroll
    for (int i = 0; i < W; ++i)
      res[i] = m0 + i < a.M ? unpack1<BF16>(a.ep.residual[static_cast<int64_t>(m0 + i) * a.ep.ldr + n]) : 0.f;
  }
  uint16_t* Cp = static_cast<uint16_t*>(a.C) + n;
#pragma unroll
  for (int i = 0; i < W; ++i) {
    if (m0 + i >= a.M) break;
    float x = a.ep.bias ? v[i] + bias_n : v[i];
    if constexpr (ACT != kActNone) x = activate(x, ACT);
    if (a.ep.residual) x += res[i];
    Cp[static_cast<int64_t>(m0 + i) * a.ldc] = static_cast<uint16_t>(pack2(x, 0.f, BF16) & 0xffffu);
  }
}

// A whole block's accumulator -> C (thread = one n, MP columns = m).
template <int MP, bool BF16, int ACT>
__device__ __forceinline__ void store_block(const SkinnyArgs& a, uint32_t taddr, int n, float bias_n) {
  constexpr int W = 16;
#pragma unroll 1
  for (int j = 0; j < MP / W; ++j) {
    uint32_t r[W];
    tmem_ld_cols<W>(taddr + j * W, r);
    tmem_wait_ld();
    if (n < a.N && j * W < a.M) {
      float v[W];
#pragma unroll
      for (int i = 0; i < W; ++i) v[i] = __uint_as_float(r[i]);
      finish_run<BF16, ACT, W>(a, j * W, n, v, bias_n);
    }
  }
}

// Sum of the block's partials (quarter q, this thread's n) in K order -> C.
// Runs of 8 m values; the contributor loop is unrolled so that the loads of
// several partials are in flight before their (in-order) sums.
template <int MP, bool BF16, int ACT>
__device__ __forceinline__ void fixup_block(const SkinnyArgs& a, int blk, int q, int lane, int c_lo, int c_hi, int n,
                                            float bias_n, int grid) {
  constexpr int W = 8;
  if (n >= a.N) return;
  // the block is the first of every contributor's range except possibly c_lo's
  const int slot_lo = range_begin(c_lo, a.total, grid) == int64_t(blk) * a.num_kb ? 0 : 1;
#pragma unroll 1
  for (int m0 = 0; m0 < a.M; m0 += W) {
    float v[W];
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = 0.f;
#pragma unroll 4
    for (int c = c_lo; c <= c_hi; ++c) {
      const int slot = c == c_lo ? slot_lo : 0;
      const float* p = a.partial + ((static_cast<int64_t>(c) * 2 + slot) * MP + m0) * kRowsB + q * 32 + lane;
      float x[W];
#pragma unroll
      for (int i = 0; i < W; ++i) x[i] = m0 + i < a.M ? __ldcg(p + i * kRowsB) : 0.f;
#pragma unroll
      for (int i = 0; i < W; ++i) v[i] += x[i];
    }
    finish_run<BF16, ACT, W>(a, m0, n, v, bias_n);
  }
}

template <int MP, int SUB, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const SkinnyArgs args) {
  using C = SkCfg<MP, SUB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sB = smem;
  uint8_t* sA = smem + C::kStages * C::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + C::kStages * C::kABytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* tfull = bars + 2 * C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int grid = gridDim.x;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
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
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Programmatic dependent launch: the next kernel in the stream may start its
  // prologue now, and no global memory is touched before the kernel before this
  // one has completed (its writes, e.g. to A, B or C, are then visible).
  griddep_launch_dependents();
  griddep_wait();
  const WaitCtl wc{abort_flag, args.err, args.timeout_ns};
  const int64_t it_begin = range_begin(cta, args.total, grid);
  const int64_t it_end = range_begin(cta + 1, args.total, grid);
  const int S = args.num_kb;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      const uint64_t b_policy = l2_policy_evict_first();   // every B byte is read once
      bool ok = true;
      for (int64_t it = it_begin; ok && it < it_end;) {
        const int blk = static_cast<int>(it / S);
        const int s0 = static_cast<int>(it - int64_t(blk) * S);
        const int s1 = (it_end - it) < int64_t(S - s0) ? s0 + static_cast<int>(it_end - it) : S;
        for (int s = s0; s < s1; ++s) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
#pragma unroll
          for (int j = 0; j < SUB; ++j) {
            const int x = (s * SUB + j) * kBK;   // boxes past K read zeros
            tma_load_2d_hint(sB + stage * C::kBBytes + j * C::kBBox, &tmB, &full[stage], x, blk * kRowsB, b_policy);
            tma_load_2d(sA + stage * C::kABytes + j * C::kABox, &tmA, &full[stage], x, 0);
          }
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        it += s1 - s0;
      }
      if (!ok) {
        // The CTA is aborting: let every copy this thread started land first.
        drain_armed(full, C::kStages, armed, armed_par, wc);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BF16, kRowsB, MP);
      const uint64_t a_desc0 = sdesc_k128(smem_u32(sB));   // B rows are the MMA's M side
      const uint64_t b_desc0 = sdesc_k128(smem_u32(sA));   // A rows are its N side
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int64_t it = it_begin; ok && it < it_end;) {
        const int blk = static_cast<int>(it / S);
        const int s0 = static_cast<int>(it - int64_t(blk) * S);
        const int s1 = (it_end - it) < int64_t(S - s0) ? s0 + static_cast<int>(it_end - it) : S;
        it += s1 - s0;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * MP;
        for (int s = s0; s < s1; ++s) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * C::kBBytes) >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * C::kABytes) >> 4);
#pragma unroll
          for (int j = 0; j < SUB; ++j)
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_f16(d_tmem, ad + ((j * C::kBBox) >> 4) + 2 * k, bd + ((j * C::kABox) >> 4) + 2 * k, idesc,
                      (s != s0 || j != 0 || k != 0) ? 1u : 0u);
          mma_commit(&empty[stage]);
          issued = true;
          if (++stage == C::kStages) {
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
        // Aborting: the tensor core must be done with TMEM before it is freed.
        mma_commit(drain);
        mbar_wait(drain, 0, wc, false);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    const int act = args.ep.act;
    for (int64_t it = it_begin; it < it_end;) {
      const int blk = static_cast<int>(it / S);
      const int s0 = static_cast<int>(it - int64_t(blk) * S);
      const int s1 = (it_end - it) < int64_t(S - s0) ? s0 + static_cast<int>(it_end - it) : S;
      const bool first_segment = it == it_begin;
      it += s1 - s0;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, wc))) break;
      tc_fence_after();
      const int n = blk * kRowsB + q * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * MP;
      const float bias_n = (args.ep.bias && n < args.N) ? unpack1<BF16>(args.ep.bias[n]) : 0.f;
      if (s0 == 0 && s1 == S) {
        if (act == kActRelu) store_block<MP, BF16, kActRelu>(args, taddr, n, bias_n);
        else if (act == kActGelu) store_block<MP, BF16, kActGelu>(args, taddr, n, bias_n);
        else if (act == kActGeluTanh) store_block<MP, BF16, kActGeluTanh>(args, taddr, n, bias_n);
        else store_block<MP, BF16, kActNone>(args, taddr, n, bias_n);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      } else {
        // publish this segment's FP32 partial ([m][128] per slot: lanes write consecutive floats)
        const int slot = first_segment ? 0 : 1;
        float* mine = args.partial + (static_cast<int64_t>(cta) * 2 + slot) * MP * kRowsB + q * 32 + lane;
#pragma unroll 1
        for (int j = 0; j < MP / C::kCols; ++j) {
          uint32_t r[C::kCols];
          tmem_ld_cols<C::kCols>(taddr + j * C::kCols, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < C::kCols; ++i) {
            const int m = j * C::kCols + i;
            if (m < args.M) mine[static_cast<int64_t>(m) * kRowsB] = __uint_as_float(r[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        __threadfence();
        __syncwarp();
        const int c_lo = cta_of(int64_t(blk) * S, args.total, grid);
        const int c_hi = cta_of(int64_t(blk) * S + S - 1, args.total, grid);
        unsigned int arrived = 0;
        if (lane == 0) {
          arrived = epoch_arrive(args.counters + blk * 4 + q, args.epoch);
          if (arrived == 0) record_error(wc, kErrFixupTimeout);
        }
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        if (arrived == static_cast<unsigned int>(c_hi - c_lo + 1)) {
          __threadfence();
          if (act == kActRelu) fixup_block<MP, BF16, kActRelu>(args, blk, q, lane, c_lo, c_hi, n, bias_n, grid);
          else if (act == kActGelu) fixup_block<MP, BF16, kActGelu>(args, blk, q, lane, c_lo, c_hi, n, bias_n, grid);
          else if (act == kActGeluTanh)
            fixup_block<MP, BF16, kActGeluTanh>(args, blk, q, lane, c_lo, c_hi, n, bias_n, grid);
          else fixup_block<MP, BF16, kActNone>(args, blk, q, lane, c_lo, c_hi, n, bias_n, grid);
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int MP, int SUB, bool BF16>
cudaError_t launch_impl(const SkinnyLaunch& L, cudaStream_t stream) {
  using C = SkCfg<MP, SUB>;
  if constexpr (C::kStages < 2) {
    return cudaErrorInvalidValue;   // the host never picks a stage that leaves no double buffering
  } else {
  auto kern = skinny_kernel<MP, SUB, BF16>;
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return launch_maybe_pdl(kern, L.grid, kThreads, C::kSmemBytes, stream, L.pdl, L.tmA, L.tmB, L.args);
  }
}

// One stage depth per padded width (the host's skinny_sub): 4 K boxes up to 64
// rows of A, 2 above (the ring keeps at least two stages).
template <bool BF16>
cudaError_t launch_mp(const SkinnyLaunch& L, cudaStream_t stream) {
  switch (L.mp) {
    case 16: return L.sub == 4 ? launch_impl<16, 4, BF16>(L, stream) : cudaErrorInvalidValue;
    case 32: return L.sub == 4 ? launch_impl<32, 4, BF16>(L, stream) : cudaErrorInvalidValue;
    case 64: return L.sub == 4 ? launch_impl<64, 4, BF16>(L, stream) : cudaErrorInvalidValue;
    case 128: return L.sub == 2 ? launch_impl<128, 2, BF16>(L, stream) : cudaErrorInvalidValue;
    case 256: return L.sub == 2 ? launch_impl<256, 2, BF16>(L, stream) : cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_skinny(const SkinnyLaunch& L, cudaStream_t stream) {
  return L.bf16 ? launch_mp<true>(L, stream) : launch_mp<false>(L, stream);
}

}  // namespace lcg
