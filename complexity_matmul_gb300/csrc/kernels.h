// Host-side declarations shared by the C-ABI layer and the kernel launchers.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace lcg {

// Fused element-wise epilogue D = act(acc + bias[col]) + residual[row, col],
// applied in FP32 by whichever kernel finishes an output element, before the
// one rounding to the output type (epilogue.cuh).
enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2, kActGeluTanh = 3 };
struct Epilogue {
  const uint16_t* bias;      // N values of the output type, 16-byte aligned, or null
  const uint16_t* residual;  // M x N of the output type, rows ldr apart (16-byte aligned), or null
  int64_t ldr;               // elements, a multiple of 8
  int act;                   // kActNone .. kActGeluTanh
  int on;                    // any of bias, residual, act present
};

// Arguments of the persistent plain GEMM: C[M,N] = A[M,K] . B[K,N].
// A and B are read through tensor maps (K-major, 128-byte swizzled boxes of
// 64 x 128 resp. 64 x BN elements); C is written directly.
struct PlainArgs {
  void* C;
  int64_t ldc;          // elements
  int M, N, K;
  int tiles_m, tiles_n, num_tiles;
  int group_m;          // tile rows per raster group (L2 reuse)
  int* err;             // device-visible error word
  uint64_t timeout_ns;  // bound on every mbarrier wait
  // split-K (single-CTA kernel only): every tile's K range is cut into `splits`
  // chunks of `kb_per_split` 64-deep slabs on consecutive work items; each
  // chunk's FP32 partial goes to `partial`, and per tile and 32-row quarter the
  // last chunk to finish (per `counters`) sums them in chunk order and writes C.
  int splits;
  int kb_per_split;
  float* partial;       // [num_tiles][splits][BN][128]: column-major slots (row fastest)
  int* counters;        // [num_tiles][4], zero before the launch
  // tail split (CTA-pair kernel only): work items below tail_first are whole tiles,
  // the 2 * (num_tiles - tail_first) items after them are K halves of the last tiles
  // (each half's partial of the other half's 128 columns in `partial` as
  // [tile][half][128 columns][256 rows], row fastest; flags [tile][half][rank][4]).
  int tail_first;
  int num_items;
  int debug_drop;       // test hook: the second K halves never raise their flags
  // CTA-pair kernel, many waves: items after each pair's first are claimed from
  // this counter (zero at launch); null: the static order
  int* tile_ctr;
  Epilogue ep;
  // split-K with many chunks: the chunks only publish their partials and a
  // separate reduction kernel sums them (every output element in parallel)
  int reduce_separately;
  // single-CTA kernel: every B tile is read once (one tile row): its loads
  // carry an L2 evict-first policy
  int b_read_once;
  // single-CTA kernel: rows per A box (a multiple of 8, at most 128).  With one
  // tile row only the rows that exist are copied; the MMA's rows past them read
  // whatever the stage held before, into accumulator rows that are never stored
  // or published, so each stage moves A bytes for M rows instead of 128.
  int a_rows;
};

// Single-CTA plain kernel with the K chunks of a tile on the CTAs of one cluster
// (summed through distributed shared memory): chunks per tile, 128-column tiles.
constexpr int kPlainClusterK = 4;
// Clusters of kPlainClusterK single-CTA plain kernels that fit on the device at once.
int plain_cluster_capacity();

struct PlainLaunch {
  CUtensorMap tmA, tmB;
  CUtensorMap tmC;      // CTA-pair kernel: C in 32 x 32 boxes, 64-byte swizzle (tensor stores)
  PlainArgs args;
  int bn;               // single-CTA kernel: 96, 128 or 256; CTA-pair kernel: 256 or 512
  int cluster_k;        // single-CTA kernel: 1, or kPlainClusterK (args.splits chunks of each tile on
                        // the CTAs of one cluster, grid = tiles x chunks)
  bool bf16;
  int grid;
  bool pdl;             // launch as a programmatic dependent of the kernel before it
};

// Box sizes the plain kernel expects in its tensor maps.
constexpr int kPlainBM = 128;
constexpr int kPlainBK = 64;

cudaError_t launch_plain(const PlainLaunch& L, cudaStream_t stream);
// Split-K with at least this many chunks sums them in a separate kernel.
constexpr int kSeparateReduceSplits = 4;
// Split-K needs at least this many 64-deep K slabs per tile: the hand-off
// (partials out, a counter, the sum) costs about as much as 24 slabs of a
// single-CTA tile's main loop, so two chunks of 16 do not pay it back.
constexpr int kSplitKMinSlabs = 48;
// Sum of the split-K partials of launch L in chunk order, epilogue, one rounding (after launch_plain).
cudaError_t launch_splitk_reduce(const PlainLaunch& L, cudaStream_t stream);
// CTA-pair variant: 256 x 256 tiles per cluster of two; tensor maps use 128-row boxes for A and B.
// Its tail split needs at least this many 64-deep K slabs: the exchange between
// the halves (a partial of 128 columns each way through L2, flags) costs a few
// microseconds, which only long enough tiles win back.
constexpr int kTailSplitMinSlabs = 48;
// From this many waves of items on, the pair kernel claims items dynamically
// (DRAM re-reads of the static order grow with the drift between pairs).
constexpr int kPairClaimMinWaves = 16;
// Width of the pair tiles: 256 x 512 tiles (two 256-column MMAs sharing each A
// slab; a quarter less operand traffic from L2) do more work per unit of time
// than 256 x 256 ones in long main loops (~5 % in burst, 3-6 % under the power
// cap at 8192^3 to 16384^3), but their one accumulator keeps each tile's epilogue
// out of the next tile's main loop (~3 us, about 10 slabs of a 256 x 256 tile),
// and a split tail costs an exchange of about as much per 256 columns.  The
// dispatcher compares the two widths' wave-quantised times with these terms.
constexpr double kWideTileGain = 1.08;
constexpr double kWideEpilogueSlabs = 10.0;
constexpr double kSplitExchangeSlabs = 10.0;
cudaError_t launch_plain_pair(const PlainLaunch& L, cudaStream_t stream);

// Skinny GEMM (M <= 256): C^T = B . A^T with 128-row blocks of B as the MMA's
// M = 128 operand and all of A (rows padded to mp) as its N operand; the
// (block, 64-deep K slab) iteration space is split into equal contiguous
// ranges, one per CTA.  A block spread over several CTAs is finished by the
// last one to arrive (per block and 32-row quarter: a counter whose high word
// is the launch's epoch, so no reset is needed); it sums the FP32 partials of
// the block's CTAs in K order.
struct SkinnyArgs {
  void* C;
  int64_t ldc;
  int M, N, K;
  int nblk, num_kb;                // 128-row blocks of B, K slabs of 64 * sub
  int64_t total;                   // nblk * num_kb
  float* partial;                  // [grid][2][mp][128]
  unsigned long long* counters;    // [nblk][4], (epoch << 32) | arrivals
  unsigned int epoch;
  int* err;
  uint64_t timeout_ns;
  Epilogue ep;
};

struct SkinnyLaunch {
  CUtensorMap tmA, tmB;            // A: box mp x 64; B: box 128 x 64
  SkinnyArgs args;
  int mp;                          // 16, 32, 64, 128 or 256
  int sub;                         // 64-deep K boxes per pipeline stage: 4 for mp <= 64, else 2
  bool bf16;
  int grid;
  bool pdl;                        // launch as a programmatic dependent of the kernel before it
};
cudaError_t launch_skinny(const SkinnyLaunch& L, cudaStream_t stream);
constexpr int kSkinnyMaxM = 256;
constexpr int kSkinnyMinKPerCta = 1024;    // grid = min(SMs, ceil(K iterations / 1024 deep))

// GEMV-shaped products (M <= 4) on the CUDA cores (gemv.cu).
struct GemvArgs {
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  int M;
  int64_t N, K;
  Epilogue ep;
};
constexpr int kGemvMaxM = 4;
cudaError_t launch_gemv(const GemvArgs& a, bool bf16, bool pdl, cudaStream_t st);

// ---------------------------------------------------------------- LCMA pre-pass / recombination

// One operand side of the Combine-A/B pre-pass.  The raw operand is stored as
// G*rows_b rows of G*kb contiguous elements (A: M x K; B: N x K).  Summed
// operands go to dst + slot * slot_stride, rows_b rows of kb elements, dst_ld apart.
struct CombineSide {
  const uint16_t* src;
  int64_t ld;
  uint16_t* dst;
  int64_t dst_ld;
  int64_t slot_stride;
  int64_t rows_b;
  int64_t kb;      // multiple of 8
  int64_t vecs;    // rows_b * kb / 8
};
struct CombineArgs {
  CombineSide side[2];  // 0: A, 1: B
};
cudaError_t launch_combine_ab(const CombineArgs& a, int levels, bool bf16, int num_sms, cudaStream_t st);

// Zero-padded copies of A and B for Strassen on non-divisible shapes: dst is
// rows_p x kp (row stride kp, a multiple of 8), src rows x k with stride ld.
struct PadSide {
  const uint16_t* src;
  int64_t ld, rows, k;
  uint16_t* dst;
  int64_t rows_p, kp;
};
struct PadArgs {
  PadSide side[2];
  int64_t vecs[2];     // rows_p * kp / 8 per side
};
cudaError_t launch_pad_copy(const PadArgs& a, int num_sms, cudaStream_t st);

// Recombination of FP32 products [R][mb][ldp] into the G x G blocks of C.
struct CombineHArgs {
  const float* prod;
  int64_t ldp;
  uint16_t* C;
  int64_t ldc;
  int mb, nb;
  Epilogue ep;          // applied in C's coordinates
  int M, N;             // C's extents: blocks of zero-padded operands may reach past them
};
cudaError_t launch_combine_h(const CombineHArgs& a, int levels, bool bf16, int num_sms, cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- fused LCMA product kernel

// Where product p's operand tile comes from: a workspace slot of summed
// operands (3-D map: k, row, slot) or one raw block of A / B in place (4-D
// map: k, storage column block c, row, storage row block r).
struct LcmaOperand {
  int slot;   // >= 0: workspace slot; -1: raw block (r, c)
  int r, c;
};

// Two-level Strassen, hierarchical: the 7 outer products each run as one
// launch of the CTA-pair fused kernel over the inner (M/4 x N/4) block grid,
// and every inner quadrant value it finishes goes to the outer level instead
// of C: up to two targets per launch, each an FP32 outer slot (Init / Acc) or
// C itself (Final: slot + sign * value, then the epilogue and the one cast).
enum : int { kOuterNone = 0, kOuterInit = 1, kOuterAcc = 2, kOuterFinal = 3 };
struct LcmaOuterTarget {
  int kind, slot, sign, quad;     // quad: outer quadrant of C (2 * row + column)
};

struct LcmaArgs {
  void* C;
  int64_t ldc;
  int mb, nb, kb;                 // block sizes M/G, N/G, K/G
  int tiles_m, tiles_n, num_groups, group_m;
  LcmaOperand a_src[49], b_src[49];
  float* prod;                    // unfused path: FP32 products [num_products][mb][ldp]
  float* scratch;                 // CTA-pair fused path: per-CTA FP32 quadrant slots
  int num_items;                  // CTA-pair fused path: work items (whole Groups + split halves)
  int split_first;                // items >= split_first are halves of split tail Groups
  int* flags;                     // one counter per split Group and CTA rank (zeroed before launch)
  int debug_drop;                 // test hook: second halves never publish
  int raw2d;                      // CTA-pair path: raw-block maps are 2-D maps of the whole operand
  int group_order;                // CTA-pair path: 1 all pairs walk one product order; 0 odd pairs another
  int outer;                      // CTA-pair path, two levels: inner quadrant values go to `otgt`
  float* oslot;                   // outer FP32 slots: 3 x [2 * mbp / 128][2 * nbp][128] (128-row blocks,
                                  // column-major inside: a warp's 32 rows of one column are one line)
  int mbp, nbp;                   // inner block sizes rounded up to the 256 x 256 Group tile
  LcmaOuterTarget otgt[2];
  int64_t ldp;
  int num_products;
  int* err;
  uint64_t timeout_ns;
  Epilogue ep;                    // applied in C's coordinates when a value is final
  int M, N;                       // C's extents: blocks of zero-padded operands may reach past them
  int c_tma;                      // CTA-pair path, one level: final values leave through tensor stores
                                  // of the quadrant maps (else 16-byte stores from registers)
};

// Tensor maps of C's four quadrant blocks (q = 2 * block row + block column),
// each clipped to C's extents: boxes of 32 x 32 elements, 64-byte swizzle.
struct QuadMaps {
  CUtensorMap q[4];
};

struct LcmaLaunch {
  CUtensorMap tmA_sum, tmA_raw, tmB_sum, tmB_raw;
  QuadMaps tmC;
  LcmaArgs args;
  int levels;
  bool bf16;
  int grid;
  bool pdl;   // launch as a programmatic dependent of the preceding pre-pass kernel
};

// Opts kernel `kern` into `bytes` of dynamic shared memory on the current
// device, once per (kernel, device).  The attribute belongs to each device's
// copy of the function, so a process that drives several devices sets it on
// each; callers on several host threads are serialised.
cudaError_t set_smem_limit(const void* kern, int bytes);

// Launches kern<<<grid, block, smem, st>>>(args...), as a programmatic dependent
// of the previous kernel in `st` when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t st, bool pdl,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
cudaError_t launch_lcma_fused(const LcmaLaunch& L, cudaStream_t st);
cudaError_t launch_lcma_products(const LcmaLaunch& L, cudaStream_t st);
// CTA-pair fused one-level kernel: Groups of 256 x 256 quadrant tiles; A and B maps use 128-row
// boxes; quadrant sums in a per-CTA FP32 scratch of lcma_pair_scratch_bytes(grid) bytes.
cudaError_t launch_lcma_pair(const LcmaLaunch& L, cudaStream_t st);
size_t lcma_pair_scratch_bytes(int grid);

// K = 0 with an epilogue: C = act(bias) + residual (the product is empty).
cudaError_t launch_epilogue_only(void* C, int64_t ldc, int M, int N, const Epilogue& ep, bool bf16, int num_sms,
                                 cudaStream_t st);

}  // namespace lcg
