// GEMV-shaped products (M <= 4: single-token and few-token decode) on the CUDA
// cores: C = A . B with every element of B read from HBM once in fully
// coalesced 16-byte loads, FP32 accumulation, one rounding.
//
// A block of 256 threads owns kRows consecutive rows n of B (the K-major
// operand) and all M rows of A.  Its 8 warps split K into 256-element chunks
// (warp w takes chunks w, w + 8, ...); in a chunk, lane l reads 8 consecutive
// elements of each of the kRows B rows (one 512-byte contiguous run per row
// and warp) and of each A row (L1/L2 resident: A is small and shared by all
// blocks), and accumulates the kRows x M products in FP32.  For M = 1 a block
// owns 4 rows (twice the blocks: short B, e.g. N = 128, still reaches many
// SMs) and two chunks' loads per warp are in flight; M = 2 and 4 keep 8 rows
// and one chunk, which measured faster at their register counts.  The per-lane sums
// are reduced across the warp (shuffles), then across the 8 warps (shared
// memory, fixed order), and the epilogue is applied once per output.
#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace lcg {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 256;       // K elements per warp iteration (32 lanes x 8)

template <int MT>
struct GemvShape {
  static constexpr int kRows = MT == 1 ? 4 : 8;     // rows of B per block
  static constexpr int kUnroll = MT == 1 ? 2 : 1;   // K chunks in flight per warp
};

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  unpack2<BF16>(u.x, f[0], f[1]);
  unpack2<BF16>(u.y, f[2], f[3]);
  unpack2<BF16>(u.z, f[4], f[5]);
  unpack2<BF16>(u.w, f[6], f[7]);
}

// 8 elements of a K-contiguous row starting at k (zeros past K), as raw 16-bit pairs.
__device__ __forceinline__ uint4 load8(const uint16_t* row, int64_t k, int64_t K, bool stream) {
  if (k + 8 <= K) {
    const uint4* p = reinterpret_cast<const uint4*>(row + k);
    return stream ? __ldcs(p) : __ldg(p);
  }
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = k + 2 * i < K ? row[k + 2 * i] : 0u;
    const uint32_t hi = k + 2 * i + 1 < K ? row[k + 2 * i + 1] : 0u;
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int MT, bool BF16>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const GemvArgs a) {
  constexpr int kRows = GemvShape<MT>::kRows;
  constexpr int kUnroll = GemvShape<MT>::kUnroll;
  __shared__ float red[kWarps][kRows][MT];
  // Programmatic dependent launch: let the next kernel be scheduled, then wait
  // for the kernel before this one (A, B or C may be its output).
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kRows;
  const uint16_t* A = static_cast<const uint16_t*>(a.A);
  const uint16_t* B = static_cast<const uint16_t*>(a.B);

  float acc[kRows][MT];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

  // rows past N read row N - 1 (a valid address); their sums are never stored
  const uint16_t* brow[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) brow[r] = B + (n0 + r < a.N ? n0 + r : a.N - 1) * a.ldb;

#pragma unroll kUnroll
  for (int64_t k = (static_cast<int64_t>(warp) * kChunk) + lane * 8; k < a.K; k += kWarps * kChunk) {
    uint4 braw[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) braw[r] = load8(brow[r], k, a.K, true);
    float av[MT][8];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < a.M) {
        unpack8<BF16>(load8(A + m * a.lda, k, a.K, false), av[m]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) av[m][i] = 0.f;
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float bv[8];
      unpack8<BF16>(braw[r], bv);
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[r][m] = fmaf(bv[i], av[m][i], acc[r][m]);
    }
  }

  // warp reduction (butterfly: every lane ends with the total), then across warps in warp order
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = acc[r][m];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[r][m] = v;
    }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) red[warp][r][m] = acc[r][m];
  }
  __syncthreads();
  if (threadIdx.x < kRows * MT) {
    const int r = threadIdx.x / MT, m = threadIdx.x % MT;
    const int64_t n = n0 + r;
    if (m < a.M && n < a.N) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red[w][r][m];
      float v[1] = {s};
      uint16_t* C = static_cast<uint16_t*>(a.C);
      store_run<BF16, 1>(C + m * a.ldc + n, m, n, 1, v, a.ep);
    }
  }
}

template <int MT, bool BF16>
cudaError_t launch_impl(const GemvArgs& a, bool pdl, cudaStream_t st) {
  constexpr int kRows = GemvShape<MT>::kRows;
  const int64_t blocks = (a.N + kRows - 1) / kRows;
  return launch_maybe_pdl(gemv_kernel<MT, BF16>, static_cast<int>(blocks), kThreads, 0, st, pdl, a);
}

template <bool BF16>
cudaError_t launch_m(const GemvArgs& a, bool pdl, cudaStream_t st) {
  if (a.M <= 1) return launch_impl<1, BF16>(a, pdl, st);
  if (a.M <= 2) return launch_impl<2, BF16>(a, pdl, st);
  return launch_impl<4, BF16>(a, pdl, st);
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, bool bf16, bool pdl, cudaStream_t st) {
  if (a.M < 1 || a.M > kGemvMaxM) return cudaErrorInvalidValue;
  return bf16 ? launch_m<true>(a, pdl, st) : launch_m<false>(a, pdl, st);
}

}  // namespace lcg
