// Host runtime shared by the C ABI, the dispatcher and the cost model.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>

struct lcgemm_ctx {
  int device = 0;
  int num_sms = 0;
  int* err_host = nullptr;   // mapped, page-locked error word (host view)
  int* err_dev = nullptr;    // the same word as the device sees it
  int* tile_ctr = nullptr;   // CTA-pair kernel's item counter (device)
  uint64_t timeout_ns = 2000000000ull;
  int group_order = 1;
  int split = 1;
  int max_ctas = 0;
  int debug_drop = 0;
  int plain_kernel = 0;         // 0: choose, 1: single-CTA 128 x 256 tiles, 2: CTA-pair 256 x 256 tiles,
                                // 3: skinny (M <= 256; larger M choose), 4: CUDA-core GEMV (M <= 4)
  int pdl = 1;                  // launch GEMM kernels as programmatic dependents of the kernel before them
  int lcma_kernel = 0;          // fused one-level: 0 choose, 1 single-CTA 128 x 128 Groups, 2 CTA-pair 256 x 128
  double peak_gflops = 2.25e6;  // dense FP16/BF16 tensor peak (GFLOP/s)
  double hbm_gbps = 8000.0;     // HBM bandwidth (GB/s)
  int last_algo = -1;
  void* ws = nullptr;           // Strassen workspace (summed operands, partials, flags)
  size_t ws_bytes = 0;
  unsigned long long* skinny_ctr = nullptr;   // skinny kernel's epoch-tagged arrival counters
  size_t skinny_ctr_n = 0;
  unsigned int epoch = 0;       // per skinny launch; counters of older epochs read as zero
  void* pad = nullptr;          // zero-padded operand copies for Strassen on non-divisible shapes
  size_t pad_bytes = 0;
  void* stage = nullptr;        // staging for lcgemm_run_host
  size_t stage_bytes = 0;
  // lcgemm_run_host pipeline: copy streams (host->device, device->host) and events
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  std::vector<cudaEvent_t> ev;
};

namespace lcg {

bool encode_map(CUtensorMap* m, bool bf16, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);
bool encode_kmajor(CUtensorMap* m, bool bf16, const void* base, int64_t rows, int64_t k, int64_t ld, int box_rows);
int grid_cap(const lcgemm_ctx* h);
int plain_single_bn(int64_t M, int64_t N, int sms);
// CTA-pair tiles of 256 x bn (bn = 256 or 512) on `pairs` pairs: the launch's time
// in units of one 256 x 256 tile's main loop (full waves, the partial last wave as
// K halves when the launcher splits it, each wave bn / 256 units long, plus the
// wide tiles' epilogues and the split tail's exchange).
double pair_waves(int64_t M, int64_t N, int64_t K, int bn, int pairs, bool split);
// The width the dispatcher takes for CTA-pair tiles (256 or 512).
int pair_tile_bn(int64_t M, int64_t N, int64_t K, int pairs, bool split);
int ensure_workspace(lcgemm_ctx* h, size_t bytes, cudaStream_t st);
// True while `st` is capturing a CUDA graph (no allocation or synchronisation allowed then).
bool capturing(cudaStream_t st);

struct Epilogue;

int run_plain(lcgemm_ctx* h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
              int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep, cudaStream_t st);

int run_strassen(lcgemm_ctx* h, int levels, bool fused, int64_t M, int64_t N, int64_t K, const void* A,
                 int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep,
                 cudaStream_t st);

// Dispatcher and cost model (runtime.cu).
bool algo_supported(int algo, int64_t M, int64_t N, int64_t K);
int select_algo(const lcgemm_ctx* h, int64_t M, int64_t N, int64_t K, int dtype);
double estimate_seconds(const lcgemm_ctx* h, int algo, int64_t M, int64_t N, int64_t K);
int dispatch(lcgemm_ctx* h, int algo, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
             int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep, cudaStream_t st);

}  // namespace lcg
