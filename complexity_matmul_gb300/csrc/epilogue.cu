// The epilogue alone, for an empty product (K = 0): C = act(bias) + residual.
//
// Grid-stride over runs of 8 columns of C; every run goes through the same
// store_run() that the GEMM kernels use, starting from a zero accumulator.
#include "epilogue.cuh"
#include "kernels.h"

namespace lcg {

namespace {

template <bool BF16>
__global__ void __launch_bounds__(256) epilogue_only_kernel(uint16_t* C, int64_t ldc, int M, int N,
                                                            const Epilogue ep) {
  const int64_t runs_per_row = (N + 7) / 8;
  const int64_t total = int64_t(M) * runs_per_row;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < total; v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = v / runs_per_row;
    const int64_t col = (v - row * runs_per_row) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int n = static_cast<int>(N - col < 8 ? N - col : 8);
    store_run<BF16, 8>(C + row * ldc + col, row, col, n, acc, ep);
  }
}

}  // namespace

cudaError_t launch_epilogue_only(void* C, int64_t ldc, int M, int N, const Epilogue& ep, bool bf16, int num_sms,
                                 cudaStream_t st) {
  const int64_t total = int64_t(M) * ((N + 7) / 8);
  int64_t blocks = (total + 255) / 256;
  blocks = blocks < int64_t(num_sms) * 8 ? blocks : int64_t(num_sms) * 8;
  if (blocks < 1) blocks = 1;
  uint16_t* Cp = static_cast<uint16_t*>(C);
  if (bf16)
    epilogue_only_kernel<true><<<static_cast<int>(blocks), 256, 0, st>>>(Cp, ldc, M, N, ep);
  else
    epilogue_only_kernel<false><<<static_cast<int>(blocks), 256, 0, st>>>(Cp, ldc, M, N, ep);
  return cudaGetLastError();
}

}  // namespace lcg
