// One-level Strassen without any allocation: lcgemm_strassen1_noalloc.
//
// The regular entry points keep their Strassen workspace (the summed operand
// blocks) in memory the handle allocates with cudaMalloc.  Some callers may
// not allocate device memory at all once they are running: a framework whose
// caching allocator already owns the device's memory (a cudaMalloc behind its
// back competes for the same pool and fails when the pool holds everything),
// or a service or safety-critical process that allows allocation only at
// start-up.  This entry point serves them: its scratch is one fixed array in
// this file, created when the library is loaded, and the call itself never
// calls cudaMalloc, cudaFree or any allocating library routine.
//
// Limits and sharing rules (also in include/lcgemm.h):
//   * the summed operands of A and B must fit in kNoallocScratchBytes
//     (2.5 * K * (M + N) bytes plus alignment), else LCGEMM_ERR_TOO_LARGE;
//   * every call on a device uses the same array, so calls that overlap on the
//     GPU (different streams, or other host threads) race; serialise them;
//   * the array keeps the previous call's contents; the only value that must
//     start at zero, the device error word, is zero when the library is
//     loaded and is cleared again only by lcgemm_noalloc_status, so an error
//     stays visible until the caller asks for it;
//   * the first call on each device looks up the array's device address with
//     cudaGetSymbolAddress (with that device current) and caches it.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "lcgemm.h"
#include "lcma_tables.h"
#include "ptx.cuh"
#include "runtime.h"

namespace {
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;   // 16 MiB for the summed operands
constexpr size_t kErrBytes = 256;                             // device error word, kept apart from them
}  // namespace

// The scratch array.  In host code this name is only a host-side stand-in:
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kErrBytes + kNoallocScratchBytes];

namespace lcg {

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Device address of the scratch array for `dev` (the current device).
int scratch_for_device(int dev, unsigned char** out, int* num_sms) {
  if (dev < 0 || dev >= kMaxDevices) return LCGEMM_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return LCGEMM_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return LCGEMM_ERR_CUDA;
    g_scratch_addr[dev] = p;
    g_num_sms[dev] = sms;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  *num_sms = g_num_sms[dev];
  return LCGEMM_OK;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

}  // namespace lcg

using namespace lcg;

extern "C" LCGEMM_API int lcgemm_strassen1_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                                   const void* B, int64_t ldb, void* C, int64_t ldc, int dtype,
                                                   void* cuda_stream) {
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return LCGEMM_ERR_ARG;
  if (dtype != LCGEMM_F16 && dtype != LCGEMM_BF16) return LCGEMM_ERR_ARG;
  if (M == 0 || N == 0) return LCGEMM_OK;
  // with K = 0 A and B are not read (and may be null), as for lcgemm_run
  if (!C || ldc < N || (K > 0 && (!A || !B || lda < K || ldb < K))) return LCGEMM_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(C) & 15u) || (ldc & 7)) return LCGEMM_ERR_ALIGN;
  if (K > 0 && (((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) || ((lda | ldb) & 7)))
    return LCGEMM_ERR_ALIGN;
  if (M % 2 || N % 2 || K % 16) return LCGEMM_ERR_UNSUPPORTED;
  if (K > 0) {
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(C), c1 = c0 + uintptr_t((M - 1) * ldc + N) * 2;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(A), a1 = a0 + uintptr_t((M - 1) * lda + K) * 2;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(B), b1 = b0 + uintptr_t((N - 1) * ldb + K) * 2;
    if ((c0 < a1 && a0 < c1) || (c0 < b1 && b0 < c1)) return LCGEMM_ERR_ALIAS;
  }

  if (K == 0) {
    // an empty product: C = 0, as lcgemm_run gives (a 2-D memset allocates nothing)
    return cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 2, 0, static_cast<size_t>(N) * 2, static_cast<size_t>(M),
                             static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
               ? LCGEMM_OK
               : LCGEMM_ERR_CUDA;
  }

  constexpr LcmaPlan<1> plan{};
  const int64_t mb = M / 2, nb = N / 2, kb = K / 2;
  const int na = plan.side[0].nslots, nbs = plan.side[1].nslots;
  const int64_t a_bytes = round_up(na * mb * kb * 2, 256);
  const int64_t b_bytes = round_up(nbs * nb * kb * 2, 256);
  if (static_cast<size_t>(a_bytes + b_bytes) > kNoallocScratchBytes) return LCGEMM_ERR_TOO_LARGE;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LCGEMM_ERR_CUDA;
  unsigned char* scratch = nullptr;
  int num_sms = 0;
  int rc = scratch_for_device(dev, &scratch, &num_sms);
  if (rc) return rc;
  int* err = reinterpret_cast<int*>(scratch);
  uint16_t* wsA = reinterpret_cast<uint16_t*>(scratch + kErrBytes);
  uint16_t* wsB = reinterpret_cast<uint16_t*>(scratch + kErrBytes + a_bytes);
  const bool bf16 = dtype == LCGEMM_BF16;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);

  CombineArgs ca{};
  ca.side[0] = CombineSide{static_cast<const uint16_t*>(A), lda, wsA, kb, mb * kb, mb, kb, mb * kb / 8};
  ca.side[1] = CombineSide{static_cast<const uint16_t*>(B), ldb, wsB, kb, nb * kb, nb, kb, nb * kb / 8};
  if (launch_combine_ab(ca, 1, bf16, num_sms, st) != cudaSuccess) return LCGEMM_ERR_CUDA;

  LcmaLaunch ll{};
  ll.levels = 1;
  ll.bf16 = bf16;
  const uint32_t box3[3] = {64u, 128u, 1u};
  const uint32_t box4[4] = {64u, 1u, 128u, 1u};
  const uint64_t dA[3] = {uint64_t(kb), uint64_t(mb), uint64_t(na)};
  const uint64_t sA[2] = {uint64_t(kb) * 2, uint64_t(mb * kb) * 2};
  const uint64_t dB[3] = {uint64_t(kb), uint64_t(nb), uint64_t(nbs)};
  const uint64_t sB[2] = {uint64_t(kb) * 2, uint64_t(nb * kb) * 2};
  const uint64_t rA[4] = {uint64_t(kb), 2u, uint64_t(mb), 2u};
  const uint64_t rsA[3] = {uint64_t(kb) * 2, uint64_t(lda) * 2, uint64_t(mb * lda) * 2};
  const uint64_t rB[4] = {uint64_t(kb), 2u, uint64_t(nb), 2u};
  const uint64_t rsB[3] = {uint64_t(kb) * 2, uint64_t(ldb) * 2, uint64_t(nb * ldb) * 2};
  if (!encode_map(&ll.tmA_sum, bf16, wsA, 3, dA, sA, box3) || !encode_map(&ll.tmB_sum, bf16, wsB, 3, dB, sB, box3) ||
      !encode_map(&ll.tmA_raw, bf16, A, 4, rA, rsA, box4) || !encode_map(&ll.tmB_raw, bf16, B, 4, rB, rsB, box4))
    return LCGEMM_ERR_CUDA;
  LcmaArgs& a = ll.args;
  a.C = C;
  a.ldc = ldc;
  a.mb = static_cast<int>(mb);
  a.nb = static_cast<int>(nb);
  a.kb = static_cast<int>(kb);
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.tiles_m = static_cast<int>((mb + 127) / 128);
  a.tiles_n = static_cast<int>((nb + 127) / 128);
  a.num_groups = a.tiles_m * a.tiles_n;
  a.group_m = 16;
  for (int p = 0; p < plan.R; ++p) {
    const auto& s0 = plan.side[0];
    const auto& s1 = plan.side[1];
    a.a_src[p] = s0.slot[p] >= 0 ? LcmaOperand{s0.slot[p], 0, 0} : LcmaOperand{-1, s0.alias_r[p], s0.alias_c[p]};
    a.b_src[p] = s1.slot[p] >= 0 ? LcmaOperand{s1.slot[p], 0, 0} : LcmaOperand{-1, s1.alias_c[p], s1.alias_r[p]};
  }
  a.prod = nullptr;
  a.ldp = 0;
  a.num_products = plan.R;
  a.err = err;
  a.timeout_ns = 2000000000ull;
  ll.grid = std::min(a.num_groups, num_sms);
  if (launch_lcma_fused(ll, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
  return LCGEMM_OK;
}

// The error word is the first int of the array; both calls work on the current
// device's copy with synchronous symbol copies into and out of a host integer.
extern "C" LCGEMM_API int lcgemm_noalloc_status(void* cuda_stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
    cudaGetLastError();
    return LCGEMM_ERR_CUDA;
  }
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_noalloc_scratch, sizeof(int), 0, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return LCGEMM_ERR_CUDA;
  }
  if (word == 0) return LCGEMM_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(int), 0, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return LCGEMM_ERR_CUDA;
  }
  return LCGEMM_ERR_TIMEOUT;
}

extern "C" LCGEMM_API int lcgemm_noalloc_debug_fail(void) {
  const int word = kErrWaitTimeout;
  if (cudaMemcpyToSymbol(g_noalloc_scratch, &word, sizeof(int), 0, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return LCGEMM_ERR_CUDA;
  }
  return LCGEMM_OK;
}
