// Host-side declarations shared by the C-ABI layer and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lcg {

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
};

struct PlainLaunch {
  CUtensorMap tmA, tmB;
  PlainArgs args;
  int bn;               // 128 or 256
  bool bf16;
  int grid;
};

// Box sizes the plain kernel expects in its tensor maps.
constexpr int kPlainBM = 128;
constexpr int kPlainBK = 64;

cudaError_t launch_plain(const PlainLaunch& L, cudaStream_t stream);

}  // namespace lcg
