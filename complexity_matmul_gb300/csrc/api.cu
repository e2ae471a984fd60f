// C ABI of lcgemm: handle, argument checks, tensor-map encoding, algorithm
// dispatch and the host-buffer entry point.  See include/lcgemm.h for the
// contract of every entry point.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "kernels.h"
#include "lcgemm.h"
#include "runtime.h"

using namespace lcg;

namespace lcg {

// ---------------------------------------------------------------- tensor maps

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_map(CUtensorMap* m, bool bf16, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5];
  cuuint32_t e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// K-major 2-D operand: `rows` rows of `k` contiguous elements, `ld` apart,
// read in boxes of 64 (K) x box_rows.
bool encode_kmajor(CUtensorMap* m, bool bf16, const void* base, int64_t rows, int64_t k, int64_t ld,
                   int box_rows) {
  const uint64_t dims[2] = {static_cast<uint64_t>(k), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(ld) * 2};
  const uint32_t box[2] = {64u, static_cast<uint32_t>(box_rows)};
  return encode_map(m, bf16, base, 2, dims, strides, box);
}

cudaError_t set_smem_limit(const void* kern, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;   // (kernel, device) pairs already opted in
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& d : done)
    if (d.first == kern && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(kern, dev);
  return e;
}

}  // namespace lcg

// ---------------------------------------------------------------- helpers

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

int check_shape(int64_t M, int64_t N, int64_t K, int dtype, int algo) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return LCGEMM_ERR_ARG;
  if (dtype != LCGEMM_F16 && dtype != LCGEMM_BF16) return LCGEMM_ERR_ARG;
  if (algo < LCGEMM_PLAIN || algo > LCGEMM_STRASSEN1_UNFUSED) return LCGEMM_ERR_ARG;
  return LCGEMM_OK;
}

int check_device_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                      const void* C, int64_t ldc) {
  if (!C || ldc < N) return LCGEMM_ERR_ARG;
  if (K > 0 && (!A || !B || lda < K || ldb < K)) return LCGEMM_ERR_ARG;
  if (ldc > (int64_t(1) << 36) || lda > (int64_t(1) << 36) || ldb > (int64_t(1) << 36)) return LCGEMM_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(C) & 15u) || (ldc & 7)) return LCGEMM_ERR_ALIGN;
  if (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
                (lda & 7) || (ldb & 7)))
    return LCGEMM_ERR_ALIGN;
  const int64_t c_bytes = ((M - 1) * ldc + N) * 2;
  if (K > 0) {
    if (overlaps(C, c_bytes, A, ((M - 1) * lda + K) * 2)) return LCGEMM_ERR_ALIAS;
    if (overlaps(C, c_bytes, B, ((N - 1) * ldb + K) * 2)) return LCGEMM_ERR_ALIAS;
  }
  return LCGEMM_OK;
}

// Checks the caller's epilogue against C and converts it for the kernels.
int make_epilogue(const lcgemm_epilogue* in, int64_t M, int64_t N, const void* C, int64_t ldc, lcg::Epilogue* out) {
  *out = lcg::Epilogue{};
  if (!in) return LCGEMM_OK;
  if (in->act < LCGEMM_ACT_NONE || in->act > LCGEMM_ACT_GELU_TANH) return LCGEMM_ERR_ARG;
  const int64_t c_bytes = ((M - 1) * ldc + N) * 2;
  if (in->bias) {
    if (reinterpret_cast<uintptr_t>(in->bias) & 15u) return LCGEMM_ERR_ALIGN;
    if (overlaps(C, c_bytes, in->bias, N * 2)) return LCGEMM_ERR_ALIAS;
  }
  if (in->residual) {
    if (in->ldr < N || in->ldr > (int64_t(1) << 36)) return LCGEMM_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(in->residual) & 15u) || (in->ldr & 7)) return LCGEMM_ERR_ALIGN;
    const bool in_place = in->residual == C && in->ldr == ldc;
    if (!in_place && overlaps(C, c_bytes, in->residual, ((M - 1) * in->ldr + N) * 2)) return LCGEMM_ERR_ALIAS;
  }
  out->bias = static_cast<const uint16_t*>(in->bias);
  out->residual = static_cast<const uint16_t*>(in->residual);
  out->ldr = in->residual ? in->ldr : 0;
  out->act = in->act;
  out->on = (in->bias || in->residual || in->act != LCGEMM_ACT_NONE) ? 1 : 0;
  return LCGEMM_OK;
}

int take_error(lcgemm_ctx* h) {
  volatile int* e = h->err_host;
  const int v = *e;
  if (v) *e = 0;
  return v ? LCGEMM_ERR_TIMEOUT : LCGEMM_OK;
}

}  // namespace

// ---------------------------------------------------------------- plain path

namespace lcg {

int grid_cap(const lcgemm_ctx* h) {
  return h->max_ctas > 0 ? std::min(h->max_ctas, h->num_sms) : h->num_sms;
}

double pair_waves(int64_t M, int64_t N, int64_t K, int bn, int pairs, bool split) {
  if (pairs <= 0) return 0.0;
  const int64_t tiles = ((M + 255) / 256) * ((N + bn - 1) / bn);
  const double kb = static_cast<double>((K + kPlainBK - 1) / kPlainBK);
  const bool claimed = tiles >= int64_t(kPairClaimMinWaves) * pairs;
  const int64_t full = tiles / pairs, rem = tiles - full * pairs;
  const bool halves = rem > 0 && split && !claimed && 2 * rem <= pairs && kb >= kTailSplitMinSlabs;
  const double waves = static_cast<double>(full) + (rem == 0 ? 0.0 : halves ? 0.5 : 1.0);
  double t = waves * (bn / 256);
  if (bn == 512) t += static_cast<double>(full + (rem > 0 ? 1 : 0)) * kWideEpilogueSlabs / kb;
  if (halves) t += kSplitExchangeSlabs * (bn / 256) / kb;
  return t;
}

int pair_tile_bn(int64_t M, int64_t N, int64_t K, int pairs, bool split) {
  return pair_waves(M, N, K, 512, pairs, split) < kWideTileGain * pair_waves(M, N, K, 256, pairs, split) ? 512 : 256;
}

// Single-CTA 128 x 256 tiles (1), CTA-pair 256 x 256 (2) or 256 x 512 (5) tiles
// (gemm_pair.cu), the weight-streaming skinny kernel (3, gemm_skinny.cu) or the GEMV (4).
int plain_variant(const lcgemm_ctx* h, int64_t M, int64_t N, int64_t K) {
  const bool skinny_ok = M <= kSkinnyMaxM && (N + 127) / 128 <= (int64_t(1) << 20);
  if (h->plain_kernel == 4 && M <= kGemvMaxM) return 4;
  if (h->plain_kernel == 3 && skinny_ok) return 3;
  if (h->plain_kernel == 1) return 1;
  if (h->plain_kernel == 2) return grid_cap(h) < 2 ? 1 : 2;
  if (h->plain_kernel == 5) return grid_cap(h) < 2 ? 1 : 5;
  // measured choices: one or two rows stream B best on the CUDA cores (at four
  // the FMA work makes the tiled split-K kernel faster); CTA pairs once their
  // 256 x 256 tiles fill a quarter of the pairs' slots; otherwise the single-CTA
  // tiles, whose split-K spreads a few tiles over the machine.  (The stream-K
  // skinny kernel measured at best level with split-K since the latter's deep
  // splits are summed by a separate kernel; it stays available as an option.)
  if (M <= 2) return 4;
  if (grid_cap(h) < 2) return 1;
  const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
  if (!(M > 128 && N > 128 && pair_tiles >= grid_cap(h) / 4)) return 1;
  return pair_tile_bn(M, N, K, grid_cap(h) / 2, h->split != 0) == 512 ? 5 : 2;
}

// Tile width of the single-CTA kernel: 256 columns, 128 for narrow C, and 96
// when C has one tile row whose 96-column tiles about fill the SMs (N = 14336
// on 152 SMs: 150 tiles), so that every SM streams its own slice of B once and
// no split-K hand-off is needed.
int plain_single_bn(int64_t M, int64_t N, int sms) {
  if (M <= kPlainBM) {
    const int64_t t96 = (N + 95) / 96;
    if (t96 <= sms && t96 * 100 >= int64_t(85) * sms) return 96;
  }
  return N <= 128 ? 128 : 256;
}

int run_gemv(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
             int64_t ldc, bool bf16, const Epilogue& ep, bool pdl, cudaStream_t st) {
  GemvArgs a{};
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = N;
  a.K = K;
  a.ep = ep;
  return launch_gemv(a, bf16, pdl, st) == cudaSuccess ? LCGEMM_OK : LCGEMM_ERR_CUDA;
}

int skinny_sub(int mp, int64_t /*K*/) { return mp <= 64 ? 4 : 2; }

int run_skinny(lcgemm_ctx* h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
               int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep, cudaStream_t st) {
  SkinnyLaunch L{};
  L.bf16 = bf16;
  L.pdl = h->pdl != 0;
  L.mp = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  if (!encode_kmajor(&L.tmA, bf16, A, M, K, lda, L.mp)) return LCGEMM_ERR_CUDA;
  if (!encode_kmajor(&L.tmB, bf16, B, N, K, ldb, 128)) return LCGEMM_ERR_CUDA;
  SkinnyArgs& a = L.args;
  a.C = C;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  // K boxes per stage: longer contiguous runs of each B row per fetch, while the
  // ring keeps at least two stages
  L.sub = skinny_sub(L.mp, K);
  a.nblk = static_cast<int>((N + 127) / 128);
  a.num_kb = static_cast<int>((K + 64 * L.sub - 1) / (64 * L.sub));
  a.total = int64_t(a.nblk) * a.num_kb;
  const int per_cta = std::max(1, kSkinnyMinKPerCta / (64 * L.sub));
  const int64_t want = (a.total + per_cta - 1) / per_cta;
  L.grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(grid_cap(h), want)));
  int rc = ensure_workspace(h, static_cast<size_t>(L.grid) * 2 * L.mp * 128 * sizeof(float), st);
  if (rc) return rc;
  a.partial = static_cast<float*>(h->ws);
  // arrival counters: zeroed once when (re)allocated; the epoch tag retires old arrivals
  const size_t nctr = static_cast<size_t>(a.nblk) * 4;
  const bool in_graph = capturing(st);
  if (nctr > h->skinny_ctr_n) {
    if (in_graph) return LCGEMM_ERR_CAPTURE;
    if (h->skinny_ctr) {
      cudaStreamSynchronize(st);
      cudaFree(h->skinny_ctr);
      h->skinny_ctr = nullptr;
      h->skinny_ctr_n = 0;
    }
    if (cudaMalloc(&h->skinny_ctr, nctr * sizeof(unsigned long long)) != cudaSuccess) {
      h->skinny_ctr = nullptr;
      cudaGetLastError();
      return LCGEMM_ERR_NOMEM;
    }
    if (cudaMemsetAsync(h->skinny_ctr, 0, nctr * sizeof(unsigned long long), st) != cudaSuccess)
      return LCGEMM_ERR_CUDA;
    h->skinny_ctr_n = nctr;
    h->epoch = 0;
  }
  if (in_graph) {
    // a graph replays this launch with the same epoch: reset the block counters in the graph too
    if (cudaMemsetAsync(h->skinny_ctr, 0, nctr * sizeof(unsigned long long), st) != cudaSuccess)
      return LCGEMM_ERR_CUDA;
    a.epoch = 1;
  } else {
    if (++h->epoch == 0) {   // 2^32 launches: start the tags over from zeroed counters
      if (cudaMemsetAsync(h->skinny_ctr, 0, h->skinny_ctr_n * sizeof(unsigned long long), st) != cudaSuccess)
        return LCGEMM_ERR_CUDA;
      h->epoch = 1;
    }
    a.epoch = h->epoch;
  }
  a.counters = h->skinny_ctr;
  a.err = h->err_dev;
  a.timeout_ns = h->timeout_ns;
  a.ep = ep;
  return launch_skinny(L, st) == cudaSuccess ? LCGEMM_OK : LCGEMM_ERR_CUDA;
}

int run_plain(lcgemm_ctx* h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
              int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep, cudaStream_t st) {
  int variant = plain_variant(h, M, N, K);
  // a fused epilogue lengthens the wide tiles' epilogue, which does not overlap the next
  // tile's main loop: 256 x 256 tiles then, unless the caller asked for the wide ones
  if (variant == 5 && ep.on && h->plain_kernel != 5) variant = 2;
  if (variant == 4) return run_gemv(M, N, K, A, lda, B, ldb, C, ldc, bf16, ep, h->pdl != 0, st);
  if (variant == 3) return run_skinny(h, M, N, K, A, lda, B, ldb, C, ldc, bf16, ep, st);
  PlainLaunch L{};
  L.bf16 = bf16;
  L.pdl = h->pdl != 0;
  const bool pair = variant == 2 || variant == 5;
  const int bm = pair ? 2 * kPlainBM : kPlainBM;
  L.bn = variant == 5 ? 512 : pair ? 256 : plain_single_bn(M, N, grid_cap(h));
  L.cluster_k = 1;
  if (!pair && M <= 32) {
    // A few rows and a K deep enough for the deep split-K (its chunks summed by a
    // separate kernel): when 128-column tiles in four K chunks about fill the SMs in
    // clusters of four, each cluster runs one tile's chunks and sums them in shared
    // memory instead (N = 4096: 32 tiles on 128 SMs).  With more rows every CTA's
    // copy of A grows to the size of its slice of B, and the deep split stays ahead
    // (128 x 4096 x 14336: 38.9 against 36.9 us).
    const int cap = grid_cap(h);
    const int64_t num_kb = (K + kPlainBK - 1) / kPlainBK, tiles_bn = (N + L.bn - 1) / L.bn;
    const int64_t t128 = (N + 127) / 128, cl = t128 * kPlainClusterK;
    const bool deep_split = tiles_bn < cap / 2 && num_kb >= kSplitKMinSlabs &&
                            std::min<int64_t>(cap / tiles_bn, num_kb / 16) >= kSeparateReduceSplits;
    if (deep_split && num_kb >= 16 * kPlainClusterK && cl <= cap && cl * 10 >= int64_t(7) * cap &&
        t128 <= plain_cluster_capacity()) {
      L.bn = 128;
      L.cluster_k = kPlainClusterK;
    }
  }
  // one tile row: the A box covers only the rows that exist (a multiple of 8)
  const int a_rows = (!pair && M < kPlainBM) ? static_cast<int>((M + 7) / 8 * 8) : kPlainBM;
  if (!encode_kmajor(&L.tmA, bf16, A, M, K, lda, a_rows)) return LCGEMM_ERR_CUDA;
  if (!encode_kmajor(&L.tmB, bf16, B, N, K, ldb, pair ? 128 : L.bn)) return LCGEMM_ERR_CUDA;
  PlainArgs& a = L.args;
  a.C = C;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + bm - 1) / bm);
  a.tiles_n = static_cast<int>((N + L.bn - 1) / L.bn);
  const int64_t tiles = int64_t(a.tiles_m) * a.tiles_n;
  if (tiles > kMaxDim) return LCGEMM_ERR_UNSUPPORTED;
  a.num_tiles = static_cast<int>(tiles);
  a.group_m = pair ? 8 : 16;
  a.err = h->err_dev;
  a.timeout_ns = h->timeout_ns;
  a.ep = ep;
  a.splits = 1;
  a.kb_per_split = static_cast<int>((K + kPlainBK - 1) / kPlainBK);
  // one tile row: each B tile is read by one CTA (per K chunk) and never again
  a.b_read_once = (!pair && a.tiles_m == 1) ? 1 : 0;
  a.a_rows = a_rows;
  if (!pair) {
    // Too few tiles to fill the machine (skinny M, small N) and a long enough K
    // (kSplitKMinSlabs): cut K into chunks of at least 16 slabs so that
    // tiles x chunks approaches the SM count.  Rounding the chunk length up
    // never raises the chunk count, so the last arriver sums two or three.
    const int num_kb = a.kb_per_split;
    const int cap = grid_cap(h);
    if (L.cluster_k > 1) {
      // each cluster: one tile's K chunks, summed in shared memory (no workspace)
      a.splits = L.cluster_k;
      a.kb_per_split = (num_kb + L.cluster_k - 1) / L.cluster_k;
    } else if (tiles < cap / 2 && num_kb >= kSplitKMinSlabs) {
      // chunks of at least 16 slabs: the fix-up's latency grows with the number of chunks
      int splits = std::min<int64_t>(cap / tiles, num_kb / 16);
      splits = std::max(1, std::min(splits, 64));
      if (splits > 1) {
        const int kps = (num_kb + splits - 1) / splits;
        splits = (num_kb + kps - 1) / kps;
        const size_t part_bytes = static_cast<size_t>(tiles) * splits * kPlainBM * L.bn * sizeof(float);
        const size_t ctr_bytes = static_cast<size_t>(tiles) * 4 * sizeof(int);
        const size_t off = (part_bytes + 255) / 256 * 256;
        int rc = ensure_workspace(h, off + ctr_bytes, st);
        if (rc) return rc;
        a.splits = splits;
        a.kb_per_split = kps;
        a.partial = static_cast<float*>(h->ws);
        a.counters = reinterpret_cast<int*>(static_cast<char*>(h->ws) + off);
        // with many chunks the last arriver's serial sum is latency-bound: a
        // separate, fully parallel reduction is faster, and needs no counters
        a.reduce_separately = splits >= kSeparateReduceSplits ? 1 : 0;
        if (!a.reduce_separately && cudaMemsetAsync(a.counters, 0, ctr_bytes, st) != cudaSuccess)
          return LCGEMM_ERR_CUDA;
      }
    }
  }
  if (pair) {
    // C for the tensor stores of whole tiles: 32 x 32 boxes (one epilogue warp's
    // chunk), 64-byte swizzle in shared memory
    // the map ends at the last whole 16-byte unit of a row (the kernel stores the
    // remaining < 8 columns from registers: a tensor store writes whole units)
    const uint64_t cdims[2] = {static_cast<uint64_t>(std::max<int64_t>(N & ~int64_t(7), 8)),
                               static_cast<uint64_t>(M)};
    const uint64_t cstrides[1] = {static_cast<uint64_t>(ldc) * 2};
    const uint32_t cbox[2] = {32u, 32u};
    if (!encode_map(&L.tmC, bf16, C, 2, cdims, cstrides, cbox, CU_TENSOR_MAP_SWIZZLE_64B)) return LCGEMM_ERR_CUDA;
    // many waves: claimed items; else the partial last wave runs as K halves when
    // its tiles fit twice over
    const int P = grid_cap(h) / 2;
    const bool claimed = a.num_tiles >= kPairClaimMinWaves * P;
    const int full = a.num_tiles / P, rem = a.num_tiles - full * P;
    const int num_kb = static_cast<int>((K + kPlainBK - 1) / kPlainBK);
    const bool split = !claimed && h->split && rem > 0 && 2 * rem <= P && num_kb >= kTailSplitMinSlabs;
    a.tail_first = split ? full * P : a.num_tiles;
    a.num_items = split ? full * P + 2 * rem : a.num_tiles;
    a.debug_drop = h->debug_drop;
    if (split) {
      const size_t part_bytes = static_cast<size_t>(rem) * 2 * 256 * (L.bn / 2) * sizeof(float);
      const size_t off = (part_bytes + 255) / 256 * 256;
      const size_t ctr_bytes = static_cast<size_t>(rem) * 2 * 2 * 4 * sizeof(int);
      int rc = ensure_workspace(h, off + ctr_bytes, st);
      if (rc) return rc;
      a.partial = static_cast<float*>(h->ws);
      a.counters = reinterpret_cast<int*>(static_cast<char*>(h->ws) + off);
      if (cudaMemsetAsync(a.counters, 0, ctr_bytes, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
    }
    L.grid = 2 * static_cast<int>(std::min<int64_t>(a.num_items, P));
    // claimed items: the counter starts at zero (a memset before each launch also
    // covers a launch that aborted, and graph replays)
    a.tile_ctr = nullptr;
    if (claimed) {
      if (cudaMemsetAsync(h->tile_ctr, 0, sizeof(int), st) != cudaSuccess) return LCGEMM_ERR_CUDA;
      a.tile_ctr = h->tile_ctr;
    }
    return launch_plain_pair(L, st) == cudaSuccess ? LCGEMM_OK : LCGEMM_ERR_CUDA;
  }
  L.grid = static_cast<int>(std::min<int64_t>(tiles * a.splits, grid_cap(h)));
  if (launch_plain(L, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
  if (a.reduce_separately && launch_splitk_reduce(L, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
  return LCGEMM_OK;
}

}  // namespace lcg

// ---------------------------------------------------------------- C ABI

extern "C" {

int lcgemm_create(lcgemm_t* out, int device) {
  if (!out) return LCGEMM_ERR_ARG;
  *out = nullptr;
  if (device == LCGEMM_PLANNING_DEVICE) {
    // cost-model queries only: no CUDA call, GB300 machine model
    auto* h = new (std::nothrow) lcgemm_ctx();
    if (!h) return LCGEMM_ERR_NOMEM;
    h->device = LCGEMM_PLANNING_DEVICE;
    h->num_sms = 152;
    *out = h;
    return LCGEMM_OK;
  }
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) return LCGEMM_ERR_ARG;
  DeviceGuard g(device);
  if (!g.ok) return LCGEMM_ERR_CUDA;
  auto* h = new (std::nothrow) lcgemm_ctx();
  if (!h) return LCGEMM_ERR_NOMEM;
  h->device = device;
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete h;
    return LCGEMM_ERR_CUDA;
  }
  if (cudaHostAlloc(reinterpret_cast<void**>(&h->err_host), 64, cudaHostAllocMapped) != cudaSuccess) {
    delete h;
    return LCGEMM_ERR_NOMEM;
  }
  *h->err_host = 0;
  if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->err_dev), h->err_host, 0) != cudaSuccess) {
    cudaFreeHost(h->err_host);
    delete h;
    return LCGEMM_ERR_CUDA;
  }
  if (cudaMalloc(&h->tile_ctr, 256) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(h->err_host);
    delete h;
    return LCGEMM_ERR_NOMEM;
  }
  if (const char* s = std::getenv("LCGEMM_PEAK_GFLOPS")) {
    const double v = std::atof(s);
    if (v > 0) h->peak_gflops = v;
  }
  if (const char* s = std::getenv("LCGEMM_HBM_GBPS")) {
    const double v = std::atof(s);
    if (v > 0) h->hbm_gbps = v;
  }
  *out = h;
  return LCGEMM_OK;
}

int lcgemm_destroy(lcgemm_t h) {
  if (!h) return LCGEMM_OK;
  if (h->device == LCGEMM_PLANNING_DEVICE) {
    delete h;
    return LCGEMM_OK;
  }
  DeviceGuard g(h->device);
  cudaDeviceSynchronize();
  if (h->ws) cudaFree(h->ws);
  if (h->stage) cudaFree(h->stage);
  if (h->skinny_ctr) cudaFree(h->skinny_ctr);
  if (h->pad) cudaFree(h->pad);
  if (h->tile_ctr) cudaFree(h->tile_ctr);
  for (cudaEvent_t e : h->ev) cudaEventDestroy(e);
  if (h->copy_in) cudaStreamDestroy(h->copy_in);
  if (h->copy_out) cudaStreamDestroy(h->copy_out);
  if (h->err_host) cudaFreeHost(h->err_host);
  delete h;
  return LCGEMM_OK;
}

int lcgemm_run(lcgemm_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
               void* C, int64_t ldc, int dtype, int algo, void* cuda_stream) {
  return lcgemm_run_epilogue(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, algo, nullptr, cuda_stream);
}

int lcgemm_run_epilogue(lcgemm_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                        int64_t ldb, void* C, int64_t ldc, int dtype, int algo, const lcgemm_epilogue* epilogue,
                        void* cuda_stream) {
  if (!h || h->device == LCGEMM_PLANNING_DEVICE) return LCGEMM_ERR_ARG;
  int rc = check_shape(M, N, K, dtype, algo);
  if (rc) return rc;
  if (M == 0 || N == 0) return LCGEMM_OK;
  rc = check_device_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (rc) return rc;
  lcg::Epilogue ep;
  rc = make_epilogue(epilogue, M, N, C, ldc, &ep);
  if (rc) return rc;
  rc = take_error(h);
  if (rc) return rc;
  DeviceGuard g(h->device);
  if (!g.ok) return LCGEMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const bool bf16 = dtype == LCGEMM_BF16;
  if (K == 0) {
    if (ep.on) {
      if (launch_epilogue_only(C, ldc, static_cast<int>(M), static_cast<int>(N), ep, bf16, h->num_sms, st) !=
          cudaSuccess)
        return LCGEMM_ERR_CUDA;
    } else if (cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 2, 0, static_cast<size_t>(N) * 2,
                                 static_cast<size_t>(M), st) != cudaSuccess) {
      return LCGEMM_ERR_CUDA;
    }
    h->last_algo = LCGEMM_PLAIN;
    return LCGEMM_OK;
  }
  int chosen = algo == LCGEMM_AUTO ? select_algo(h, M, N, K, dtype) : algo;
  rc = dispatch(h, chosen, M, N, K, A, lda, B, ldb, C, ldc, bf16, ep, st);
  if (rc == LCGEMM_OK) h->last_algo = chosen;
  return rc;
}

// Host buffers: plain GEMMs (explicit or chosen by the cost model) run as a grid
// of C blocks.  A row chunks and B column chunks go to the device alternately on
// a copy stream (A0, B0, A1, B1, ...); each block's GEMM runs on the caller's
// stream as soon as its two chunks have arrived, and each block of C goes back on
// a second copy stream -- host->device copies, tensor-core work and
// device->host copies overlap, and the first GEMM waits for two chunks instead
// of all of B.  A block may sum the K range in a different FP32 order than the
// whole GEMM would (split choices depend on the tile count), so results agree to
// FP32 rounding, not bit for bit.  Strassen runs unchunked.
int lcgemm_run_host(lcgemm_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, void* C, int64_t ldc, int dtype, int algo, void* cuda_stream) {
  if (!h || h->device == LCGEMM_PLANNING_DEVICE) return LCGEMM_ERR_ARG;
  int rc = check_shape(M, N, K, dtype, algo);
  if (rc) return rc;
  if (M == 0 || N == 0) return LCGEMM_OK;
  if (!C || ldc < N || (K > 0 && (!A || !B || lda < K || ldb < K))) return LCGEMM_ERR_ARG;
  DeviceGuard g(h->device);
  if (!g.ok) return LCGEMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (capturing(st)) return LCGEMM_ERR_CAPTURE;   // copy streams and host buffers: not capturable
  // device staging: pitches rounded up to 8 elements (16 bytes), 256-byte aligned sub-buffers
  const int64_t kp = std::max<int64_t>(8, (K + 7) / 8 * 8);
  const int64_t np = (N + 7) / 8 * 8;
  auto rup = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t a_bytes = rup(M * kp * 2), b_bytes = rup(N * kp * 2), c_bytes = rup(M * np * 2);
  const size_t need = static_cast<size_t>(a_bytes + b_bytes + c_bytes);
  if (need > h->stage_bytes) {
    if (h->stage) {
      cudaStreamSynchronize(st);
      if (h->copy_in) cudaStreamSynchronize(h->copy_in);
      if (h->copy_out) cudaStreamSynchronize(h->copy_out);
      cudaFree(h->stage);
      h->stage = nullptr;
      h->stage_bytes = 0;
    }
    if (cudaMalloc(&h->stage, need) != cudaSuccess) {
      h->stage = nullptr;
      return LCGEMM_ERR_NOMEM;
    }
    h->stage_bytes = need;
  }
  char* dA = static_cast<char*>(h->stage);
  char* dB = dA + a_bytes;
  char* dC = dB + b_bytes;
  if (K == 0) {
    rc = lcgemm_run(h, M, N, K, dA, kp, dB, kp, dC, np, dtype, algo, cuda_stream);
    if (rc) return rc;
    return cudaMemcpy2DAsync(C, ldc * 2, dC, np * 2, N * 2, M, cudaMemcpyDeviceToHost, st) == cudaSuccess
               ? LCGEMM_OK
               : LCGEMM_ERR_CUDA;
  }
  const int chosen = algo == LCGEMM_AUTO ? select_algo(h, M, N, K, dtype) : algo;
  // Plain GEMMs run as a grid of nr x nc blocks of C (2048-row/column chunks, at
  // most 8 x 8), so that the first block can start as soon as one chunk of A and
  // one of B have arrived, instead of after all of B.
  int nr = 1, nc = 1;
  if (chosen == LCGEMM_PLAIN) {
    nr = static_cast<int>(std::min<int64_t>(8, std::max<int64_t>(1, M / 2048)));
    nc = static_cast<int>(std::min<int64_t>(8, std::max<int64_t>(1, N / 2048)));
  }
  if (nr * nc == 1) {
    if (cudaMemcpy2DAsync(dA, kp * 2, A, lda * 2, K * 2, M, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpy2DAsync(dB, kp * 2, B, ldb * 2, K * 2, N, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return LCGEMM_ERR_CUDA;
    rc = lcgemm_run(h, M, N, K, dA, kp, dB, kp, dC, np, dtype, chosen, cuda_stream);
    if (rc) return rc;
    if (cudaMemcpy2DAsync(C, ldc * 2, dC, np * 2, N * 2, M, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return LCGEMM_ERR_CUDA;
    return LCGEMM_OK;
  }
  if (!h->copy_in) {
    if (cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking) != cudaSuccess)
      return LCGEMM_ERR_CUDA;
  }
  // events: [0] start, [1, 1 + nr) A chunk i in, [1 + nr, 1 + nr + nc) B chunk j in,
  // then one per C block done, and the last: every block copied out
  const size_t need_ev = 2 + static_cast<size_t>(nr + nc + nr * nc);
  while (h->ev.size() < need_ev) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return LCGEMM_ERR_CUDA;
    h->ev.push_back(e);
  }
  cudaEvent_t* ev = h->ev.data();
  cudaEvent_t* ev_a = ev + 1;
  cudaEvent_t* ev_b = ev + 1 + nr;
  cudaEvent_t* ev_c = ev + 1 + nr + nc;
  cudaEvent_t ev_out = ev[need_ev - 1];
  const int64_t rows = ((M + nr - 1) / nr + 255) / 256 * 256;   // chunk extents, multiples of 256
  const int64_t cols = ((N + nc - 1) / nc + 255) / 256 * 256;
  nr = static_cast<int>((M + rows - 1) / rows);
  nc = static_cast<int>((N + cols - 1) / cols);
  bool ok = cudaEventRecord(ev[0], st) == cudaSuccess && cudaStreamWaitEvent(h->copy_in, ev[0], 0) == cudaSuccess &&
            cudaStreamWaitEvent(h->copy_out, ev[0], 0) == cudaSuccess;
  const auto copy_a = [&](int i) {
    const int64_t r0 = i * rows, mr = std::min(rows, M - r0);
    return cudaMemcpy2DAsync(dA + r0 * kp * 2, kp * 2, static_cast<const char*>(A) + r0 * lda * 2, lda * 2, K * 2,
                             mr, cudaMemcpyHostToDevice, h->copy_in) == cudaSuccess &&
           cudaEventRecord(ev_a[i], h->copy_in) == cudaSuccess;
  };
  const auto copy_b = [&](int j) {
    const int64_t c0 = j * cols, nn = std::min(cols, N - c0);
    return cudaMemcpy2DAsync(dB + c0 * kp * 2, kp * 2, static_cast<const char*>(B) + c0 * ldb * 2, ldb * 2, K * 2,
                             nn, cudaMemcpyHostToDevice, h->copy_in) == cudaSuccess &&
           cudaEventRecord(ev_b[j], h->copy_in) == cudaSuccess;
  };
  const auto block = [&](int i, int j) -> int {
    const int64_t r0 = i * rows, mr = std::min(rows, M - r0), c0 = j * cols, nn = std::min(cols, N - c0);
    if (cudaStreamWaitEvent(st, ev_a[i], 0) != cudaSuccess || cudaStreamWaitEvent(st, ev_b[j], 0) != cudaSuccess)
      return LCGEMM_ERR_CUDA;
    const int r = lcgemm_run(h, mr, nn, K, dA + r0 * kp * 2, kp, dB + c0 * kp * 2, kp, dC + (r0 * np + c0) * 2, np,
                             dtype, LCGEMM_PLAIN, cuda_stream);
    if (r) return r;
    cudaEvent_t e = ev_c[i * nc + j];
    const bool out = cudaEventRecord(e, st) == cudaSuccess && cudaStreamWaitEvent(h->copy_out, e, 0) == cudaSuccess &&
                     cudaMemcpy2DAsync(static_cast<char*>(C) + (r0 * ldc + c0) * 2, ldc * 2,
                                       dC + (r0 * np + c0) * 2, np * 2, nn * 2, mr, cudaMemcpyDeviceToHost,
                                       h->copy_out) == cudaSuccess;
    return out ? LCGEMM_OK : LCGEMM_ERR_CUDA;
  };
  // growing square: A chunk k, then the blocks it completes with B chunks < k;
  // B chunk k, then the blocks it completes with A chunks <= k
  for (int k = 0; ok && k < std::max(nr, nc); ++k) {
    if (k < nr) {
      ok = copy_a(k);
      for (int j = 0; ok && j < std::min(k, nc); ++j) {
        rc = block(k, j);
        if (rc) return rc;
      }
    }
    if (ok && k < nc) {
      ok = copy_b(k);
      for (int i = 0; ok && i < std::min(k + 1, nr); ++i) {
        rc = block(i, k);
        if (rc) return rc;
      }
    }
  }
  ok = ok && cudaEventRecord(ev_out, h->copy_out) == cudaSuccess && cudaStreamWaitEvent(st, ev_out, 0) == cudaSuccess;
  if (!ok) return LCGEMM_ERR_CUDA;
  h->last_algo = LCGEMM_PLAIN;
  return LCGEMM_OK;
}

int lcgemm_last_algo(lcgemm_t h) { return h ? h->last_algo : LCGEMM_ERR_ARG; }

int lcgemm_select(lcgemm_t h, int64_t M, int64_t N, int64_t K, int dtype) {
  if (!h) return LCGEMM_ERR_ARG;
  const int rc = check_shape(M, N, K, dtype, LCGEMM_AUTO);
  if (rc) return rc;
  return select_algo(h, M, N, K, dtype);
}

int lcgemm_estimate(lcgemm_t h, int64_t M, int64_t N, int64_t K, int dtype, int algo, double* seconds) {
  if (!h || !seconds) return LCGEMM_ERR_ARG;
  int rc = check_shape(M, N, K, dtype, algo);
  if (rc) return rc;
  // mirror lcgemm_run's early exits: an empty C launches nothing, and with K = 0
  // C is only filled (or the epilogue applied), whatever algorithm was asked for
  if (M == 0 || N == 0) {
    *seconds = 0.0;
    return LCGEMM_OK;
  }
  if (K == 0) algo = LCGEMM_PLAIN;
  if (algo == LCGEMM_AUTO) algo = select_algo(h, M, N, K, dtype);
  if (!algo_supported(algo, M, N, K)) return LCGEMM_ERR_UNSUPPORTED;
  *seconds = estimate_seconds(h, algo, M, N, K);
  return LCGEMM_OK;
}

int lcgemm_sync_status(lcgemm_t h, void* cuda_stream) {
  if (!h || h->device == LCGEMM_PLANNING_DEVICE) return LCGEMM_ERR_ARG;
  DeviceGuard g(h->device);
  if (!g.ok) return LCGEMM_ERR_CUDA;
  const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  const int rc = take_error(h);
  if (rc) return rc;
  return e == cudaSuccess ? LCGEMM_OK : LCGEMM_ERR_CUDA;
}

int lcgemm_set_option(lcgemm_t h, int option, int64_t value) {
  if (!h) return LCGEMM_ERR_ARG;
  switch (option) {
    case LCGEMM_OPT_WAIT_TIMEOUT_US:
      if (value <= 0 || value > int64_t(60) * 1000000) return LCGEMM_ERR_ARG;
      h->timeout_ns = static_cast<uint64_t>(value) * 1000u;
      return LCGEMM_OK;
    case LCGEMM_OPT_GROUP_ORDER:
      if (value != 0 && value != 1) return LCGEMM_ERR_ARG;
      h->group_order = static_cast<int>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_SPLIT:
      if (value != 0 && value != 1) return LCGEMM_ERR_ARG;
      h->split = static_cast<int>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_MAX_CTAS:
      if (value < 0 || value > 65536) return LCGEMM_ERR_ARG;
      h->max_ctas = static_cast<int>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_PEAK_GFLOPS:
      if (value <= 0) return LCGEMM_ERR_ARG;
      h->peak_gflops = static_cast<double>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_HBM_GBPS:
      if (value <= 0) return LCGEMM_ERR_ARG;
      h->hbm_gbps = static_cast<double>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_DEBUG_DROP_SIGNAL:
      if (value != 0 && value != 1) return LCGEMM_ERR_ARG;
      h->debug_drop = static_cast<int>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_PLAIN_KERNEL:
      if (value < 0 || value > 5) return LCGEMM_ERR_ARG;
      h->plain_kernel = static_cast<int>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_PDL:
      if (value < 0 || value > 1) return LCGEMM_ERR_ARG;
      h->pdl = static_cast<int>(value);
      return LCGEMM_OK;
    case LCGEMM_OPT_LCMA_KERNEL:
      if (value < 0 || value > 2) return LCGEMM_ERR_ARG;
      h->lcma_kernel = static_cast<int>(value);
      return LCGEMM_OK;
    default:
      return LCGEMM_ERR_ARG;
  }
}

const char* lcgemm_strerror(int code) {
  switch (code) {
    case LCGEMM_OK: return "ok";
    case LCGEMM_ERR_ARG: return "invalid argument";
    case LCGEMM_ERR_ALIGN: return "pointer not 16-byte aligned or leading dimension not a multiple of 8";
    case LCGEMM_ERR_UNSUPPORTED: return "algorithm does not support these dimensions";
    case LCGEMM_ERR_ALIAS: return "C overlaps A, B or the bias, or partly overlaps the residual";
    case LCGEMM_ERR_CUDA: return "CUDA call or kernel launch failed";
    case LCGEMM_ERR_TIMEOUT: return "a bounded device-side wait gave up in an earlier launch";
    case LCGEMM_ERR_NOMEM: return "workspace allocation failed";
    case LCGEMM_ERR_TOO_LARGE: return "problem too large for the fixed scratch of lcgemm_strassen1_noalloc";
    case LCGEMM_ERR_CAPTURE: return "stream capture: the call would grow a handle buffer, or cannot be captured";
    default: return "unknown status code";
  }
}

}  // extern "C"
