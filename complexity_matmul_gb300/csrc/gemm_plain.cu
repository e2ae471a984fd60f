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
// the last to arrive, more by splitk_reduce_kernel.  With KC > 1 the KC chunks
// of a 128-column tile run on the KC CTAs of one cluster instead: each leaves
// its FP32 partial in its own (drained) operand ring and CTA r sums columns
// 32r .. 32r + 31 of all KC partials through distributed shared memory, in
// chunk order, with no workspace, counter or second kernel.  When C has one
// tile row, every B tile is read once and its loads carry an L2 evict-first
// policy.
//
// Prior art for the tiling, the multi-stage prefetch and the block swizzle:
// CUDA-L2 summary (gist.science 2512.02551), "discovered techniques" list
// (double-buffering, multi-step prefetch, block swizzling for L2 hit rate).
#include <mutex>

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

// Row pitch (floats) of a cluster-split partial in shared memory: 16-byte rows, and
// consecutive rows 4 banks apart.
template <int BN>
constexpr int kRedPitch = BN + 4;

template <int BN, int STAGES, bool BF16, bool EPI, int KC>
__global__ void __launch_bounds__(kThreads, 1)
    plain_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const PlainArgs args) {
  using C = Cfg<BN, STAGES>;
  static_assert(KC == 1 || (BN / KC == 32 && kBM * kRedPitch<BN> * 4 <= STAGES * C::kStageBytes),
                "a cluster split gives each CTA 32 columns; the partial fits in the ring");
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
  bool epi_ok = false;   // KC > 1: this epilogue warp's partial is in shared memory

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
      if constexpr (KC > 1) {
        // one item per CTA: this chunk's FP32 partial into the drained operand ring
        // (every copy landed and every MMA finished before tfull), row-major
        float* red = reinterpret_cast<float*>(smem) + (q * 32 + lane) * kRedPitch<BN>;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + c * 32, r);
          tmem_wait_ld();
          float4* dst = reinterpret_cast<float4*>(red + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        epi_ok = true;
        break;
      } else if (args.splits == 1) {
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

  if constexpr (KC > 1) {
    // every CTA of the cluster has its partial in shared memory (or has given up)
    cluster_sync();
    if (warp >= 2 && epi_ok) {
      const int q = warp & 3;
      const uint32_t rank = cluster_ctarank();
      int mb, nb;
      tile_coords(static_cast<int>(blockIdx.x) / KC, args, mb, nb);
      const int rloc = q * 32 + lane, row = mb * kBM + rloc;
      const int col = nb * BN + static_cast<int>(rank) * 32;
      if (row < args.M && col < args.N) {
        EpiLoads<32> pre;
        if constexpr (EPI) load_chunk(row, col, args, pre);
        const uint32_t mine = smem_u32(smem) + static_cast<uint32_t>((rloc * kRedPitch<BN> + rank * 32) * 4);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
#pragma unroll 1
        for (int s = 0; s < KC; ++s) {   // chunk order
          const uint32_t src = mapa_shared(mine, static_cast<uint32_t>(s));
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 x = ld_cluster_v4(src + 16 * j);
            v[4 * j] += x.x;
            v[4 * j + 1] += x.y;
            v[4 * j + 2] += x.z;
            v[4 * j + 3] += x.w;
          }
        }
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
        store_chunk<BF16, EPI>(static_cast<uint16_t*>(args.C) + static_cast<int64_t>(row) * args.ldc, row, col, r,
                               args, &pre);
      }
    }
    // no CTA leaves while the others may still read its shared memory
    cluster_sync();
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

template <int BN, int STAGES, bool BF16, bool EPI, int KC = 1>
cudaError_t launch_impl(const PlainLaunch& L, cudaStream_t stream) {
  using C = Cfg<BN, STAGES>;
  auto kern = plain_gemm_kernel<BN, STAGES, BF16, EPI, KC>;
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  if constexpr (KC == 1) {
    return launch_maybe_pdl(kern, L.grid, kThreads, C::kSmemBytes, stream, L.pdl, L.tmA, L.tmB, L.args);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = KC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.args);
  }
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
  if (L.cluster_k == kPlainClusterK) {
    if (L.bn != 128 || L.args.splits != kPlainClusterK || L.grid != L.args.num_tiles * kPlainClusterK)
      return cudaErrorInvalidValue;
    if (L.args.ep.on)
      return L.bf16 ? launch_impl<128, 6, true, true, kPlainClusterK>(L, stream)
                    : launch_impl<128, 6, false, true, kPlainClusterK>(L, stream);
    return L.bf16 ? launch_impl<128, 6, true, false, kPlainClusterK>(L, stream)
                  : launch_impl<128, 6, false, false, kPlainClusterK>(L, stream);
  }
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

int plain_cluster_capacity() {
  // per device, once: the occupancy query needs the kernel's shared-memory opt-in
  static std::mutex mu;
  static int cached[64];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cached[dev];
  using C = Cfg<128, 6>;
  auto kern = plain_gemm_kernel<128, 6, true, false, kPlainClusterK>;
  int n = 0;
  if (set_smem_limit(reinterpret_cast<const void*>(kern), C::kSmemBytes) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kPlainClusterK);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPlainClusterK;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();   // the failed query's error, not a launch's
    }
  }
  cached[dev] = n;
  done[dev] = true;
  return n;
}

}  // namespace lcg
