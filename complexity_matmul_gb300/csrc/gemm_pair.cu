// Plain GEMM on CTA pairs (cta_group::2): 256 x 256 or 256 x 512 output tiles per pair.
//
// Same pipeline as the single-CTA kernel (TMA producer, MMA issuer, four
// epilogue warps, accumulators in tensor memory), but each tcgen05.mma covers
// M = 256 rows: the even CTA of a cluster of two issues it, each CTA stages 128
// rows of A and its half of the tile's B rows in its own shared memory, and
// each CTA keeps its 128 accumulator rows in its own tensor memory.  Per SM
// and 256 x 256 x 64 step the tensor core reads 16 KB of A and 16 KB of B
// instead of 16 KB + 32 KB, which halves the shared-memory and L2 traffic per
// flop; 512-column tiles let two such steps share the A slab.
//
// Epilogue: each warp casts 32 x 32 chunks of its 32 accumulator rows into two
// alternating shared-memory boxes and writes each with one tensor store, so C
// leaves in whole cache lines (a direct store of the row-per-lane layout
// touches 32 lines per warp instruction, ~2 us per 256 x 256 tile).
//
// Tail split (static order only): when the tiles of the partial last wave fit
// twice over into the pairs, each runs as two K halves on two pairs.  Each half
// publishes the FP32 partial of the half of the tile's columns that the other
// half finishes, raises its flag, waits (bounded) for the other's flag, and
// finishes its own columns as (0 + half 0) + half 1 from its accumulator and
// the other's partial.  A pair has at most one such item, its last, and publishes before it
// waits, so the two halves cannot wait on each other in a cycle.
//
// Work distribution.  Few waves: pair p runs items p, p + P, p + 2P, ... (P
// pairs).  Many waves (DYN): every pair still starts with item p, but takes
// each later item from a global counter, claimed a few slabs before its
// current item ends.  Claims then follow the order in which pairs become free,
// so the items that share an A or B panel (neighbours in the grouped raster)
// run close together in time whatever the pairs' drift, and the panel is still
// in L2 for the second reader: at 16384^3 this halves the DRAM reads of the
// static order.  The leader CTA's producer claims and publishes each item
// through a small queue in both CTAs' shared memory; the other roles read it
// from there.  The host zeroes the counter before each such launch.
//
// Synchronisation across the pair:
//   full[s]   leader's barrier; the leader arms it with both CTAs' bytes and
//             both CTAs' TMA copies complete on it
//   empty[s]  one per CTA; the leader's MMA commit arrives on both
//   tfull[b]  one per CTA; the leader's MMA commit arrives on both
//   tempty[b] leader's barrier; all 8 epilogue warps of the pair arrive
//   qfull[j]  one per CTA (DYN); the leader's producer arrives after writing
//             queue slot j of that CTA
//   qempty[j] leader's barrier (DYN); every reader of slot j arrives
#include "kernels.h"
#include "plain_common.cuh"
#include "ptx.cuh"

namespace lcg {

namespace {

constexpr int kBM = 128;           // rows per CTA (256 per pair)
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBox = 128 * kBK * 2;  // one 128-row B box: a CTA's share of one 256-column MMA
constexpr int kTmemCols = 512;

// Tile of 256 x (256 * NB) per pair: per 16-deep K step NB MMAs of N = 256 share
// the A operand.  NB = 1: six 32 KB stages and two accumulators (the epilogue of
// one tile overlaps the next tile's main loop).  NB = 2: four 48 KB stages and
// one 512-column accumulator (the epilogue does not overlap), but each A slab
// serves 512 columns: a quarter less operand traffic from L2 per flop.
template <int NB>
struct PairCfg {
  static constexpr int kBN = 256 * NB;
  static constexpr int kStages = NB == 1 ? 6 : 4;
  static constexpr int kBBytes = NB * kBBox;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTxBytes = 2 * kStageBytes;
  static constexpr int kAccs = NB == 1 ? 2 : 1;
  static_assert(kAccs * kBN == kTmemCols, "accumulators fill tensor memory");
};
constexpr int kQ = 4;              // queue slots (DYN): items published but not yet read by every role
constexpr int kQReaders = 10;      // the leader's MMA issuer, the partner's producer, 8 epilogue warps
constexpr int kClaimLead = 8;      // the next item is claimed this many slabs before the current one ends
constexpr int kCBoxBytes = 32 * 32 * 2;            // one epilogue warp's 32 x 32 chunk of C
constexpr int kCStageBytes = 4 * 2 * kCBoxBytes;     // two boxes per epilogue warp
template <int NB>
constexpr int pair_smem_bytes() {
  return PairCfg<NB>::kStages * PairCfg<NB>::kStageBytes + kCStageBytes + 512 + 1024;
}
static_assert(pair_smem_bytes<1>() <= 232448 && pair_smem_bytes<2>() <= 232448, "shared memory budget");

// Queue of claimed items (DYN).  `item`/`full` are this CTA's; `empty` is the
// leader CTA's (addressed through the cluster window from either CTA).
struct ItemQueue {
  int* item;
  uint64_t* full;
  uint64_t* empty;
  uint32_t slot, phase;

  __device__ __forceinline__ void advance() {
    if (++slot == kQ) {
      slot = 0;
      phase ^= 1;
    }
  }
  // Leader's producer: writes item w into slot `slot` of both CTAs and signals them.
  __device__ __forceinline__ bool publish(int w, const WaitCtl& wc) {
    if (!mbar_wait_cluster(&empty[slot], phase ^ 1, wc)) return false;
    item[slot] = w;
    st_relaxed_cluster_s32(mapa_shared(smem_u32(&item[slot]), 1), w);
    mbar_arrive_cluster(mapa_shared(smem_u32(&full[slot]), 0));
    mbar_arrive_cluster(mapa_shared(smem_u32(&full[slot]), 1));
    advance();
    return true;
  }
  // Any other role: reads the next item and frees the slot.
  __device__ __forceinline__ bool pop(int& w, const WaitCtl& wc) {
    if (!mbar_wait_cluster(&full[slot], phase, wc)) return false;
    w = *reinterpret_cast<volatile int*>(&item[slot]);
    mbar_arrive_cluster(mapa_shared(smem_u32(&empty[slot]), 0));
    advance();
    return true;
  }
};

// Work item -> tile and K-slab range.  Items below tail_first are whole tiles;
// the rest are the two K halves of the tiles of the partial last wave.
__device__ __forceinline__ void pair_item(int w, const PlainArgs& a, int num_kb, int& tile, int& kb0, int& kb1,
                                          int& half) {
  if (w < a.tail_first) {
    tile = w;
    kb0 = 0;
    kb1 = num_kb;
    half = -1;
  } else {
    const int i = (w - a.tail_first) >> 1;
    half = (w - a.tail_first) & 1;
    tile = a.tail_first + i;
    const int mid = num_kb / 2;
    kb0 = half ? mid : 0;
    kb1 = half ? num_kb : mid;
  }
}

// Epilogue (EPI), cast and tensor store of one finished 32 x 32 chunk: rows
// row0 .. row0 + 31 (this lane: row), columns col .. col + 31, through `box`, one
// of the warp's two shared-memory boxes used in turn.
template <bool BF16, bool EPI>
__device__ __forceinline__ void emit_chunk(float (&v)[32], int row, int row0, int col, uint32_t box, int lane,
                                           const CUtensorMap* tmC, const PlainArgs& args, const EpiLoads<32>* cur) {
  if constexpr (EPI)
    if (row < args.M && col < args.N) apply_epilogue<BF16, 32>(row, col, min(32, args.N - col), v, args.ep, cur);
  if (lane == 0) bulk_wait_read<1>();   // the store that read this box two chunks ago is done with it
  __syncwarp();
  stage_chunk<BF16>(box, lane, v);
  fence_proxy_async_shared();
  __syncwarp();
  const int n8 = args.N & ~7;   // the map of C ends at the last whole 16-byte unit of a row
  if (lane == 0) {
    if (row0 < args.M && col < n8) tma_store_2d(tmC, box, col, row0);
    bulk_commit();
  }
  if (col + 32 > n8 && col < args.N && row < args.M)
    store_cols<BF16>(static_cast<uint16_t*>(args.C) + static_cast<int64_t>(row) * args.ldc + col, v,
                     max(n8 - col, 0), min(args.N - col, 32));
}

template <bool BF16, bool EPI, bool DYN, int NB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    plain_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const PlainArgs args) {
  using Cfg = PairCfg<NB>;
  constexpr int kBN = Cfg::kBN, kStages = Cfg::kStages, kBBytes = Cfg::kBBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sC = sB + kStages * kBBytes;   // epilogue boxes (1024-byte aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sC + kCStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* qfull = drain + 1;
  uint64_t* qempty = qfull + kQ;
  int* qitem = reinterpret_cast<int*>(qempty + kQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qitem + kQ);
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
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);
    }
    mbar_init(drain, 1);
    for (int j = 0; j < kQ; ++j) {
      mbar_init(&qfull[j], 1);
      mbar_init(&qempty[j], kQReaders);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Programmatic dependent launch: the next kernel in the stream may start its
  // prologue now, and no global memory is touched before the kernel before this
  // one has completed (its writes, e.g. to A, B or C, are then visible).
  griddep_launch_dependents();
  griddep_wait();
  const WaitCtl wc{abort_flag, args.err, args.timeout_ns};
  const int num_kb = (args.K + kBK - 1) / kBK;
  const int pair = blockIdx.x / 2;
  const int num_pairs = gridDim.x / 2;
  ItemQueue iq{qitem, qfull, qempty, 0, 0};

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      int next = pair;   // DYN leader: the item claimed for after the current one
      for (int w = pair; ok;) {
        if constexpr (DYN) {
          if (leader) {
            w = next;
            if (!iq.publish(w, wc)) {
              ok = false;
              break;
            }
          } else if (!iq.pop(w, wc)) {
            ok = false;
            break;
          }
        }
        if (w >= args.num_items) break;   // DYN: every pair's last claim lies past the end
        int tile, kb0, kb1, half;
        pair_item(w, args, num_kb, tile, kb0, kb1, half);
        int mb, nb;
        tile_coords(tile, args, mb, nb);
        const int claim_at = max(kb0, kb1 - kClaimLead);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (DYN && leader && kb == claim_at) next = num_pairs + atomicAdd(args.tile_ctr, 1);
          if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], Cfg::kTxBytes);
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          tma_load_2d_pair(sA + stage * kABytes, &tmA, bar, kb * kBK, mb * 2 * kBM + rank * kBM);
          // B: for each 256-column part of the tile, this CTA's 128 rows
#pragma unroll
          for (int j = 0; j < NB; ++j)
            tma_load_2d_pair(sB + stage * kBBytes + j * kBBox, &tmB, bar, kb * kBK, nb * kBN + j * 256 + rank * 128);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (DYN && leader && kb0 >= kb1) next = num_pairs + atomicAdd(args.tile_ctr, 1);   // (no empty items exist)
        if constexpr (!DYN) w += num_pairs;
      }
      if (!ok) {
        // Aborting: let this CTA's copies land before it leaves.
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
      constexpr uint32_t idesc = idesc_f16(BF16, 2 * kBM, 256);
      // descriptors of stage 0; a stage / K-step offset is added to the start-address field
      const uint64_t a_desc0 = sdesc_k128(smem_u32(sA));
      const uint64_t b_desc0 = sdesc_k128(smem_u32(sB));
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int w = pair; ok; w += num_pairs) {
        if constexpr (DYN) {
          if (!iq.pop(w, wc)) break;
        }
        if (w >= args.num_items) break;
        int tile, kb0, kb1, half;
        pair_item(w, args, num_kb, tile, kb0, kb1, half);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;   // NB parts of 256 columns
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * kABytes) >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * kBBytes) >> 4);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
#pragma unroll
            for (int j = 0; j < NB; ++j)
              mma_f16_pair(d_tmem + j * 256, ad + 2 * k, bd + ((j * kBBox) >> 4) + 2 * k, idesc,
                           (kb != kb0 || k != 0) ? 1u : 0u);
          mma_commit_pair(&empty[stage]);
          issued = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair(&tfull[acc]);
        if (++acc == Cfg::kAccs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok && issued) {
        mma_commit_pair(drain);
        mbar_wait(drain, 0, wc, false);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    const uint32_t sbox = smem_u32(sC) + q * 2 * kCBoxBytes;   // this warp's two boxes
    uint32_t nbox = 0;
    for (int w = pair;; w += num_pairs) {
      if constexpr (DYN) {
        int v = 0;
        const bool got = lane == 0 ? iq.pop(v, wc) : true;
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) break;
        w = __shfl_sync(0xffffffffu, v, 0);
      }
      if (w >= args.num_items) break;
      int tile, kb0, kb1, half;
      pair_item(w, args, num_kb, tile, kb0, kb1, half);
      int mb, nb;
      tile_coords(tile, args, mb, nb);
      const int row = mb * 2 * kBM + rank * kBM + q * 32 + lane;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, wc))) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
      const int row0 = row - lane;
      if (half < 0) {
        // whole tile: each 32 x 32 chunk is finished in registers, cast into one of
        // the warp's two shared-memory boxes and written by a tensor store (full
        // lines; rows past C are clipped by the tensor map, a row's last partial
        // 16-byte unit is stored from registers)
        EpiLoads<32> pre;
        if constexpr (EPI) {
          load_chunk(row, nb * kBN, args, pre);   // next chunk's bias / residual in flight
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            const int col = nb * kBN + c * 32;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + c * 32, r);
            const EpiLoads<32> cur = pre;
            if (c + 1 < kBN / 32) load_chunk(row, col + 32, args, pre);
            tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
            emit_chunk<BF16, EPI>(v, row, row0, col, sbox + ((nbox++ & 1u) * kCBoxBytes), lane, &tmC, args, &cur);
          }
        } else {
          // chunk c + 1's tensor-memory load is in flight while chunk c is cast and
          // stored (two register sets, the loop unrolled by two)
          static_assert((kBN / 32) % 2 == 0, "chunks come in pairs");
          uint32_t ra[32], rb[32];
          auto finish = [&](const uint32_t (&r)[32], int c) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
            emit_chunk<BF16, EPI>(v, row, row0, nb * kBN + c * 32, sbox + ((nbox++ & 1u) * kCBoxBytes), lane, &tmC,
                                  args, nullptr);
          };
          tmem_ld_32x32b_x32(tbase, ra);
          tmem_wait_ld(ra);
#pragma unroll 1
          for (int c = 0; c < kBN / 32; c += 2) {
            tmem_ld_32x32b_x32(tbase + (c + 1) * 32, rb);
            finish(ra, c);
            tmem_wait_ld(rb);
            if (c + 2 < kBN / 32) tmem_ld_32x32b_x32(tbase + (c + 2) * 32, ra);
            finish(rb, c + 1);
            tmem_wait_ld(ra);
          }
        }
      } else {
        // tail tile, K half `half`: the partial of the columns the other half finishes
        // goes out (column-major per half: one cache line per warp store), then this
        // half's columns are finished from its accumulator and the other's partial
        const int i = tile - args.tail_first;
        const int slot_rows = 2 * kBM;
        const int64_t slot = int64_t(slot_rows) * (kBN / 2);
        const int64_t rloc = rank * kBM + q * 32 + lane;
        const int own_c0 = half * (kBN / 2), other_c0 = (half ^ 1) * (kBN / 2);
        const int left = args.N - nb * kBN;   // columns of C from this tile's first on
        const int out_chunks = max(0, min(kBN / 64, (left - other_c0 + 31) / 32));
        float* out = args.partial + (int64_t(i) * 2 + half) * slot + rloc;
#pragma unroll 1
        for (int c = 0; c < out_chunks; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + other_c0 + c * 32, r);
          tmem_wait_ld();
          if (row < args.M) publish_partial(out + c * 32 * slot_rows, slot_rows, r);
        }
        __threadfence();
        __syncwarp();
        int* flag = args.counters + ((i * 2 + half) * 2 + static_cast<int>(rank)) * 4 + q;
        const int* peer = args.counters + ((i * 2 + (half ^ 1)) * 2 + static_cast<int>(rank)) * 4 + q;
        if (lane == 0 && !(args.debug_drop && half == 1)) red_release_gpu_add(flag, 1);
        if (__all_sync(0xffffffffu, wait_flag(peer, 1, wc))) {
          // rows past M read slot entries nobody wrote and are not stored
          const float* in = args.partial + (int64_t(i) * 2 + (half ^ 1)) * slot + rloc;
          const int own_chunks = max(0, min(kBN / 64, (left - own_c0 + 31) / 32));
          float o[32];
          if (own_chunks > 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __ldcg(in + j * slot_rows);
          }
#pragma unroll 1
          for (int c = 0; c < own_chunks; ++c) {
            const int col = nb * kBN + own_c0 + c * 32;
            EpiLoads<32> cur;
            if constexpr (EPI) load_chunk(row, col, args, cur);
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + own_c0 + c * 32, r);
            tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float mine = __uint_as_float(r[j]);
              v[j] = half == 0 ? (0.f + mine) + o[j] : (0.f + o[j]) + mine;
            }
            // the next chunk's loads go out before this one is emitted (after it with the
            // fused epilogue, whose registers they would otherwise share)
            if (!EPI && c + 1 < own_chunks) {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __ldcg(in + ((c + 1) * 32 + j) * slot_rows);
            }
            emit_chunk<BF16, EPI>(v, row, row0, col, sbox + ((nbox++ & 1u) * kCBoxBytes), lane, &tmC, args, &cur);
            if (EPI && c + 1 < own_chunks) {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __ldcg(in + ((c + 1) * 32 + j) * slot_rows);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      if (++acc == Cfg::kAccs) {
        acc = 0;
        acc_phase ^= 1;
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

template <bool BF16, bool EPI, bool DYN, int NB>
cudaError_t launch_impl(const PlainLaunch& L, cudaStream_t stream) {
  auto kern = plain_pair_kernel<BF16, EPI, DYN, NB>;
  constexpr int smem = pair_smem_bytes<NB>();
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
  }
  return launch_maybe_pdl(kern, L.grid, kThreads, smem, stream, L.pdl, L.tmA, L.tmB, L.tmC, L.args);
}

}  // namespace

namespace {

template <int NB>
cudaError_t launch_width(const PlainLaunch& L, cudaStream_t stream) {
  // the kernel without an epilogue keeps the lean store path
  if (L.args.tile_ctr) {
    if (L.args.ep.on)
      return L.bf16 ? launch_impl<true, true, true, NB>(L, stream) : launch_impl<false, true, true, NB>(L, stream);
    return L.bf16 ? launch_impl<true, false, true, NB>(L, stream) : launch_impl<false, false, true, NB>(L, stream);
  }
  if (L.args.ep.on)
    return L.bf16 ? launch_impl<true, true, false, NB>(L, stream) : launch_impl<false, true, false, NB>(L, stream);
  return L.bf16 ? launch_impl<true, false, false, NB>(L, stream) : launch_impl<false, false, false, NB>(L, stream);
}

}  // namespace

cudaError_t launch_plain_pair(const PlainLaunch& L, cudaStream_t stream) {
  if (L.grid % 2) return cudaErrorInvalidValue;
  if (L.bn == 512) return launch_width<2>(L, stream);
  if (L.bn == 256) return launch_width<1>(L, stream);
  return cudaErrorInvalidValue;
}

}  // namespace lcg
