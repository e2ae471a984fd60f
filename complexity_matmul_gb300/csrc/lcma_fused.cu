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
#include "lcma_program.cuh"

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
      griddep_wait();   // the summed operands come from the pre-pass kernel before this one
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
      if (!ok) drain_armed(full, kStages, armed, armed_par, wc);   // aborting: let this thread's copies land
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BF16, kBM, kBN);
      // descriptors of stage 0; a stage / K-step offset is added to the start-address field
      const uint64_t a_desc0 = sdesc_k128(smem_u32(sA));
      const uint64_t b_desc0 = sdesc_k128(smem_u32(sB));
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
            const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * kTileBytes) >> 4);
            const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * kTileBytes) >> 4);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc,
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
          store_quadrant<BF16>(lane_base + o.src * kBN, args, o.quad, mb * kBM + q * 32 + lane, nb * kBN);
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
      griddep_wait();   // the summed operands come from the pre-pass kernel before this one
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
      if (!ok) drain_armed(full, kStages, armed, armed_par, wc);   // aborting: let this thread's copies land
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(bf16, kBM, kBN);
      // descriptors of stage 0; a stage / K-step offset is added to the start-address field
      const uint64_t a_desc0 = sdesc_k128(smem_u32(sA));
      const uint64_t b_desc0 = sdesc_k128(smem_u32(sB));
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
          const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * kTileBytes) >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * kTileBytes) >> 4);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
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
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return launch_maybe_pdl(kern, L.grid, kThreads, kSmemBytes, st, L.pdl, L.tmA_sum, L.tmA_raw, L.tmB_sum, L.tmB_raw,
                          L.args);
}

}  // namespace

cudaError_t launch_lcma_fused(const LcmaLaunch& L, cudaStream_t st) {
  if (L.levels != 1) return cudaErrorInvalidValue;
  return L.bf16 ? launch_impl<true>(L, st) : launch_impl<false>(L, st);
}

cudaError_t launch_lcma_products(const LcmaLaunch& L, cudaStream_t st) {
  {
    const cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(lcma_products_kernel), kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return launch_maybe_pdl(lcma_products_kernel, L.grid, kThreads, kSmemBytes, st, L.pdl, L.tmA_sum, L.tmA_raw, L.tmB_sum,
                          L.tmB_raw, L.args, L.bf16);
}

}  // namespace lcg
