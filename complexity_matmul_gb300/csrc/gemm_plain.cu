// Persistent plain GEMM for sm_103a: C = A . B, FP16/BF16 in, FP32 accumulate
// in tensor memory, one round-to-nearest-even cast on the way out.
//
// One CTA per SM walks a grouped raster of 128 x BN output tiles.  Warp roles:
//   warp 0      TMA producer: A (128 x 64) and B (BN x 64) K-slabs into a
//               STAGES-deep shared-memory ring (full/empty mbarriers)
//   warp 1      TMEM allocator and MMA issuer: 4 tcgen05.mma (K = 16 each)
//               per slab into one of two TMEM accumulators
//   warps 2..5  epilogue: tcgen05.ld -> cvt.rn -> global stores, overlapped
//               with the next tile's main loop through the second accumulator
//
// Few tiles and a long K: the launcher cuts each tile's K range into chunks
// (split-K) on consecutive work items; a chunk's FP32 partial goes to a
// column-major slot of the workspace, and two or three chunks are summed by
// the last to arrive, more by splitk_reduce_kernel.  When C has one tile row,
// every B tile is read once and its loads carry an L2 evict-first policy.
//
// Prior art for the tiling, the multi-stage prefetch and the block swizzle:
// CUDA-L2 summary (gist.science 2512.02551), "discovered techniques" list
// (double-buffering, multi-step prefetch, block swizzling for L2 hit rate).
#include "kernels.h"
#include "plain_common.cuh"
#include "ptx.cuh"

namespace lcg {

namespace {

constexpr int kBM = kPlainBM;
constexpr int kBK = kPlainBK;
constexpr int kThreads = 192;
static_assert(kSeparateReduceSplits == 4, "the last arriver's sum is instantiated for 2 and 3 chunks");

template <int BN, int STAGES>
struct Cfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kAccCols = BN <= 128 ? 128 : 256;       // accumulator stride (128-column aligned)
  static constexpr int kTmemCols = 2 * kAccCols;                // two accumulators, a power of two
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = STAGES * kStageBytes + kBarBytes + 1024;
  static_assert(2 * BN <= kTmemCols && BN % 32 == 0, "accumulator columns");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int BN, int STAGES, bool BF16, bool EPI>
__global__ void __launch_bounds__(kThreads, 1)
    plain_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const PlainArgs args) {
  using C = Cfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * C::kBBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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
  const int num_kb = (args.K + kBK - 1) / kBK;
  const int num_work = args.num_tiles * args.splits;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      const uint64_t b_policy = l2_policy_evict_first();
      bool ok = true;
      for (int w = blockIdx.x; ok && w < num_work; w += gridDim.x) {
        const int tile = w / args.splits, split = w - tile * args.splits;
        int mb, nb;
        tile_coords(tile, args, mb, nb);
        const int kb0 = split * args.kb_per_split, kb1 = min(num_kb, kb0 + args.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(args.a_rows * kBK * 2 + C::kBBytes));
          tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], kb * kBK, mb * kBM);
          if (args.b_read_once)
            tma_load_2d_hint(sB + stage * C::kBBytes, &tmB, &full[stage], kb * kBK, nb * BN, b_policy);
          else
            tma_load_2d(sB + stage * C::kBBytes, &tmB, &full[stage], kb * kBK, nb * BN);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // The CTA is aborting: let every copy this thread started land first.
        drain_armed(full, STAGES, armed, armed_par, wc);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BF16, kBM, BN);
      // descriptors of stage 0; a stage / K-step offset is added to the start-address field
      const uint64_t a_desc0 = sdesc_k128(smem_u32(sA));
      const uint64_t b_desc0 = sdesc_k128(smem_u32(sB));
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int w = blockIdx.x; ok && w < num_work; w += gridDim.x) {
        const int split = w % args.splits;
        const int kb0 = split * args.kb_per_split, kb1 = min(num_kb, kb0 + args.kb_per_split);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::kAccCols;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * C::kABytes) >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * C::kBBytes) >> 4);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          mma_commit(&empty[stage]);
          issued = true;
          if (++stage == STAGES) {
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
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t acc = 0, acc_phase = 0;
    uint16_t* Cp = static_cast<uint16_t*>(args.C);
    for (int w = blockIdx.x; w < num_work; w += gridDim.x) {
      const int tile = w / args.splits, split = w - tile * args.splits;
      int mb, nb;
      tile_coords(tile, args, mb, nb);
      const int row = mb * kBM + q * 32 + lane;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, wc));
      if (!ok) break;
      tc_fence_after();
      uint16_t* crow = Cp + static_cast<int64_t>(row) * args.ldc;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
      if (args.splits == 1) {
        if constexpr (EPI) {
          // the next chunk's bias / residual loads are in flight while this chunk is finished
          EpiLoads<32> pre;
          load_chunk(row, nb * BN, args, pre);
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + c * 32, r);
            const EpiLoads<32> cur = pre;
            if (c + 1 < BN / 32) load_chunk(row, nb * BN + (c + 1) * 32, args, pre);
            tmem_wait_ld();
            store_chunk<BF16, true>(crow, row, nb * BN + c * 32, r, args, &cur);
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + c * 32, r);
            tmem_wait_ld();
            store_chunk<BF16, false>(crow, row, nb * BN + c * 32, r, args);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      } else {
        // split-K: publish this chunk's FP32 partial (rows and column chunks inside C
        // only; column-major slot, one cache line per warp store), free TMEM
        const int64_t slot = int64_t(kBM) * BN;
        const int chunks = min(BN / 32, (args.N - nb * BN + 31) / 32);
        float* mine = args.partial + (static_cast<int64_t>(tile) * args.splits + split) * slot + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < chunks; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + c * 32, r);
          tmem_wait_ld();
          if (row < args.M) publish_partial(mine + c * 32 * kBM, kBM, r);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        if (args.reduce_separately) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
          continue;
        }
        // The last chunk to arrive (per tile and lane quarter: no cross-warp
        // barrier, no waiting) sums all chunks' partials in chunk order.
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atom_add_acq_rel(args.counters + tile * 4 + q, 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == args.splits - 1) {
          if (lane == 0) args.counters[tile * 4 + q] = 0;   // ready for the next launch
          __threadfence();
          const float* first = args.partial + static_cast<int64_t>(tile) * args.splits * slot + q * 32 + lane;
          if (row < args.M) {
#pragma unroll 1
            for (int c = 0; c < chunks; ++c) {
              EpiLoads<32> pre;
              if constexpr (EPI) load_chunk(row, nb * BN + c * 32, args, pre);
              uint32_t r[32];
              if (args.splits == 2) sum_partials<2>(first + c * 32 * kBM, kBM, slot, r);
              else sum_partials<3>(first + c * 32 * kBM, kBM, slot, r);
              store_chunk<BF16, EPI>(crow, row, nb * BN + c * 32, r, args, &pre);
            }
          }
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

// Split-K reduction: one block per (tile, 32-column chunk).  The chunk's
// valid rows x 32 columns are dealt to the threads column-major (consecutive
// threads on consecutive rows of a column: each load instruction reads
// contiguous bytes of a column-major slot), so a skinny tile keeps every thread
// busy.  Each thread sums its elements over the K chunks in chunk order, four
// chunks' loads in flight at a time; the block transposes the sums through
// shared memory and each thread then finishes 8-column runs of a row:
// epilogue, one rounding, 16-byte stores.
constexpr int kReduceThreads = 256;
constexpr int kReducePer = 32 * kBM / kReduceThreads;   // elements per thread (full tile)

template <int BN, bool BF16>
__global__ void __launch_bounds__(kReduceThreads) splitk_reduce_kernel(const PlainArgs a) {
  __shared__ float T[32][kBM + 1];
  // launched as a programmatic dependent of the GEMM that wrote the partials: its blocks
  // are resident when that grid ends and read nothing before it has completed
  griddep_launch_dependents();
  griddep_wait();
  constexpr int kChunks = BN / 32;
  const int tile = blockIdx.x / kChunks;
  const int c32 = (blockIdx.x % kChunks) * 32;
  int mb, nb;
  tile_coords(tile, a, mb, nb);
  const int64_t row0 = int64_t(mb) * kBM;
  const int64_t col0 = int64_t(nb) * BN + c32;
  if (col0 >= a.N) return;                      // the whole block: no barrier skipped by part of it
  const int rows = static_cast<int>(a.M - row0 < kBM ? a.M - row0 : kBM);
  const int64_t slot = int64_t(kBM) * BN;
  const float* base = a.partial + int64_t(tile) * a.splits * slot + int64_t(c32) * kBM;
  int off[kReducePer];
  bool on[kReducePer];
  float s[kReducePer];
#pragma unroll
  for (int k = 0; k < kReducePer; ++k) {
    const int e = threadIdx.x + k * kReduceThreads;
    const int j = e / rows;
    on[k] = j < 32;
    off[k] = j * kBM + (e - j * rows);
    s[k] = 0.f;
  }
#pragma unroll 1
  for (int sp0 = 0; sp0 < a.splits; sp0 += 4) {
    const int n = a.splits - sp0 < 4 ? a.splits - sp0 : 4;
    float x[4][kReducePer];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < kReducePer; ++k)
        x[i][k] = (i < n && on[k]) ? __ldcg(base + (sp0 + i) * slot + off[k]) : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < kReducePer; ++k)
        if (i < n) s[k] += x[i][k];
  }
#pragma unroll
  for (int k = 0; k < kReducePer; ++k)
    if (on[k]) T[off[k] / kBM][off[k] % kBM] = s[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int u = threadIdx.x + k * kReduceThreads;     // 128 rows x 4 runs of 8 columns
    const int rr = u / 4, c8 = (u % 4) * 8;
    const int64_t row = row0 + rr, col = col0 + c8;
    if (rr >= rows || col >= a.N) continue;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = T[c8 + i][rr];
    const int n = static_cast<int>(a.N - col < 8 ? a.N - col : 8);
    uint16_t* C = static_cast<uint16_t*>(a.C) + row * a.ldc + col;
    if (a.ep.on) store_run<BF16, 8>(C, row, col, n, v, a.ep);
    else cast_store<BF16, 8>(C, n, v);
  }
}

template <int BN, int STAGES, bool BF16, bool EPI>
cudaError_t launch_impl(const PlainLaunch& L, cudaStream_t stream) {
  using C = Cfg<BN, STAGES>;
  auto kern = plain_gemm_kernel<BN, STAGES, BF16, EPI>;
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return launch_maybe_pdl(kern, L.grid, kThreads, C::kSmemBytes, stream, L.pdl, L.tmA, L.tmB, L.args);
}

template <int BN, bool BF16>
cudaError_t launch_reduce_impl(const PlainLaunch& L, cudaStream_t stream) {
  const int64_t blocks = int64_t(L.args.num_tiles) * (BN / 32);
  return launch_maybe_pdl(splitk_reduce_kernel<BN, BF16>, static_cast<int>(blocks), kReduceThreads, 0, stream, L.pdl,
                          L.args);
}

}  // namespace

cudaError_t launch_splitk_reduce(const PlainLaunch& L, cudaStream_t stream) {
  if (L.bn == 256) return L.bf16 ? launch_reduce_impl<256, true>(L, stream)
                                 : launch_reduce_impl<256, false>(L, stream);
  if (L.bn == 96) return L.bf16 ? launch_reduce_impl<96, true>(L, stream)
                                : launch_reduce_impl<96, false>(L, stream);
  if (L.bn == 128) return L.bf16 ? launch_reduce_impl<128, true>(L, stream)
                                 : launch_reduce_impl<128, false>(L, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_plain(const PlainLaunch& L, cudaStream_t stream) {
  // the kernel without an epilogue keeps the lean store path
  if (L.args.ep.on) {
    if (L.bn == 256) return L.bf16 ? launch_impl<256, 4, true, true>(L, stream) : launch_impl<256, 4, false, true>(L, stream);
    if (L.bn == 128) return L.bf16 ? launch_impl<128, 6, true, true>(L, stream) : launch_impl<128, 6, false, true>(L, stream);
    if (L.bn == 96) return L.bf16 ? launch_impl<96, 7, true, true>(L, stream) : launch_impl<96, 7, false, true>(L, stream);
  }
  if (L.bn == 256) return L.bf16 ? launch_impl<256, 4, true, false>(L, stream) : launch_impl<256, 4, false, false>(L, stream);
  if (L.bn == 128) return L.bf16 ? launch_impl<128, 6, true, false>(L, stream) : launch_impl<128, 6, false, false>(L, stream);
  if (L.bn == 96) return L.bf16 ? launch_impl<96, 7, true, false>(L, stream) : launch_impl<96, 7, false, false>(L, stream);
  return cudaErrorInvalidValue;
}

}  // namespace lcg
