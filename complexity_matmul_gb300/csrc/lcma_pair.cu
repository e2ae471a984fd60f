// Fused one-level LCMA kernel on CTA pairs (cta_group::2).
//
// Same Group program as the single-CTA kernel in lcma_fused.cu (product order
// M5 M3 M7 M1 M4 M2 M6, four 128-column TMEM buffers, 12 epilogue ops per
// Group), but a Group covers a 256 x 128 tile of each quadrant: the even CTA
// of a cluster of two issues tcgen05.mma.cta_group::2 with M = 256, N = 128;
// each CTA stages 128 rows of the product's A operand and 64 of its 128 B
// rows, and holds its 128 rows of every buffer in its own tensor memory.
// Per SM the tensor core then reads 16 KB of A and 8 KB of B per 64-deep K
// slab for 128 x 128 x 64 MACs (96 B/clk at the tensor peak) instead of
// 16 KB + 16 KB (128 B/clk) -- the single-CTA 128 x 128 tile is limited by
// shared-memory bandwidth, the pair tile is not.
//
// Cross-CTA synchronisation:
//   full[s]       leader's; armed with both CTAs' bytes; both CTAs' copies complete on it
//   empty[s]      per CTA; the leader's commit arrives on both
//   mdone[step]   per CTA; the leader's commit arrives on both
//   progress[4]   per CTA, one counter per epilogue warp; the leader's MMA thread
//                 reads all eight through distributed shared memory
#include "lcma_program.cuh"

namespace lcg {

namespace {

constexpr int kRows = 128;                 // rows per CTA (256 per pair)
constexpr int kBN = kBufCols;              // columns per Group tile
constexpr int kBK = 64;
constexpr int kStages = 8;
constexpr int kThreads = 192;
constexpr int kABytes = kRows * kBK * 2;   // 16 KB
constexpr int kBBytes = (kBN / 2) * kBK * 2;   // 8 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTxBytes = 2 * kStageBytes;
constexpr int kTmemCols = 512;
constexpr int kSmemBytes = kStages * kStageBytes + 512 + 1024;

__device__ __forceinline__ void load_operand_pair(void* dst, const CUtensorMap* sum_map, const CUtensorMap* raw_map,
                                                  const LcmaOperand& src, uint32_t bar, int k0, int row0) {
  if (src.slot >= 0)
    tma_load_3d_pair(dst, sum_map, bar, k0, row0, src.slot);
  else
    tma_load_4d_pair(dst, raw_map, bar, k0, src.c, row0, src.r);
}

// All eight epilogue-warp counters of the pair have reached `target`.
__device__ __forceinline__ bool pair_counters_reached(uint32_t local0, uint32_t peer0, uint32_t target) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    if (ld_acquire_cluster_u32(local0 + 4 * w) < target) return false;
    if (ld_acquire_cluster_u32(peer0 + 4 * w) < target) return false;
  }
  return true;
}

__device__ __forceinline__ bool wait_pair_counters(uint32_t local0, uint32_t peer0, uint32_t target,
                                                   const WaitCtl& w) {
  if (pair_counters_reached(local0, peer0, target)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (pair_counters_reached(local0, peer0, target)) return true;
    if ((i & 31u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        record_error(w, kErrWaitTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void red_release_cluster_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.cluster.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lcma1_pair_kernel(const __grid_constant__ CUtensorMap tmA_sum, const __grid_constant__ CUtensorMap tmA_raw,
                      const __grid_constant__ CUtensorMap tmB_sum, const __grid_constant__ CUtensorMap tmB_raw,
                      const LcmaArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* mdone = bars + 2 * kStages;
  uint64_t* drain = mdone + kSteps;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* progress = tmem_slot + 1;            // [4]: ops completed per epilogue warp of this CTA
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 5);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

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
  if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, args.err, args.timeout_ns};
  const int num_kb = (args.kb + kBK - 1) / kBK;
  const int pair = blockIdx.x / 2;
  const int num_pairs = gridDim.x / 2;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int t = pair; ok && t < args.num_groups; t += num_pairs) {
        int mb, nb;
        tile_coords(t, args, mb, nb);
        for (int s = 0; ok && s < kSteps; ++s) {
          const int p = d_step_product[s];
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, wc)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&full[stage], kTxBytes);
            const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
            load_operand_pair(sA + stage * kABytes, &tmA_sum, &tmA_raw, args.a_src[p], bar, kb * kBK,
                              mb * 2 * kRows + static_cast<int>(rank) * kRows);
            load_operand_pair(sB + stage * kBBytes, &tmB_sum, &tmB_raw, args.b_src[p], bar, kb * kBK,
                              nb * kBN + static_cast<int>(rank) * (kBN / 2));
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
      constexpr uint32_t idesc = idesc_f16(BF16, 2 * kRows, kBN);
      // descriptors of stage 0; a stage / K-step offset is added to the start-address field
      const uint64_t a_desc0 = sdesc_k128(smem_u32(sA));
      const uint64_t b_desc0 = sdesc_k128(smem_u32(sB));
      const uint32_t ctr_local = mapa_shared(smem_u32(progress), 0);
      const uint32_t ctr_peer = mapa_shared(smem_u32(progress), 1);
      uint32_t stage = 0, phase = 0, g = 0;
      bool ok = true, issued = false;
      for (int t = pair; ok && t < args.num_groups; t += num_pairs, ++g) {
        for (int s = 0; ok && s < kSteps; ++s) {
          const int need = static_cast<int>(g) * kNumOps + d_step_need[s];
          if (need > 0 && !wait_pair_counters(ctr_local, ctr_peer, static_cast<uint32_t>(need), wc)) {
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
            const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * kABytes) >> 4);
            const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * kBBytes) >> 4);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_f16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc,
                           (d_step_fresh[s] && kb == 0 && k == 0) ? 0u : 1u);
            mma_commit_pair(&empty[stage]);
            issued = true;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (ok && d_step_has_ops[s]) mma_commit_pair(&mdone[s]);
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
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t g = 0;
    bool ok = true;
    for (int t = pair; ok && t < args.num_groups; t += num_pairs, ++g) {
      int mb, nb;
      tile_coords(t, args, mb, nb);
      const int rloc = mb * 2 * kRows + static_cast<int>(rank) * kRows + q * 32 + lane;
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
          store_quadrant<BF16>(lane_base + o.src * kBN, args, o.quad, rloc, nb * kBN);
        } else {
          combine_buffers(lane_base + o.dst * kBN, lane_base + o.src * kBN, static_cast<float>(o.sign),
                          o.kind == kOpAdd);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) red_release_cluster_add(progress + q, 1u);
      }
    }
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
  auto kern = lcma1_pair_kernel<BF16>;
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

cudaError_t launch_lcma_pair(const LcmaLaunch& L, cudaStream_t st) {
  if (L.levels != 1 || L.grid % 2) return cudaErrorInvalidValue;
  return L.bf16 ? launch_impl<true>(L, st) : launch_impl<false>(L, st);
}

}  // namespace lcg
