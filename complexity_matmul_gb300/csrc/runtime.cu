// Algorithm dispatch and the roofline-style cost model behind LCGEMM_AUTO.
//
// Cost model (FalconGEMM write-up, section "从缓存重排到 Cost Model"): the
// aim is to pick the right algorithm, not to predict time exactly.  Each
// candidate is a short sequence of kernels; every kernel is charged
// max(flops / (eta * peak), bytes / (beta * bandwidth)) -- the roofline bound
// F <= min(F_max, I * B_max) of the kernel-performance notes
// (wineandchord.com kernels-performance, "Roofline") -- stretched by the wave
// quantisation of its tile grid over the SMs, plus a launch overhead.  The
// low-complexity algorithms trade 1/8 (one level) or 15/64 (two levels) of
// the multiplications for extra operand traffic, so they only win where the
// plain GEMM is compute-bound and large.
#include <algorithm>
#include <cmath>

#include "lcgemm.h"
#include "runtime.h"

namespace lcg {

// Strassen splits every dimension into 2 (4) equal blocks; the block width
// along K must keep 16-byte row starts for the tensor-memory-access engine.
bool algo_supported(int algo, int64_t M, int64_t N, int64_t K) {
  switch (algo) {
    case LCGEMM_PLAIN:
      return true;
    case LCGEMM_STRASSEN1:
    case LCGEMM_STRASSEN1_UNFUSED:
      return M >= 2 && N >= 2 && K >= 16 && M % 2 == 0 && N % 2 == 0 && K % 16 == 0;
    case LCGEMM_STRASSEN2:
      return M >= 4 && N >= 4 && K >= 32 && M % 4 == 0 && N % 4 == 0 && K % 32 == 0;
    default:
      return false;
  }
}

namespace {

// Fractions of the tensor peak and of the HBM bandwidth each kernel reaches
// when it is not limited by its tile grid (calibrated on GB300).
constexpr double kEtaPlain = 0.70;
constexpr double kBetaStream = 0.85;
constexpr double kLaunchSec = 4e-6;

double wave_efficiency(int64_t tiles, int sms) {
  if (tiles <= 0) return 1.0;
  const int64_t waves = (tiles + sms - 1) / sms;
  return static_cast<double>(tiles) / static_cast<double>(waves * sms);
}

}  // namespace

double estimate_seconds(const lcgemm_ctx* h, int algo, int64_t M, int64_t N, int64_t K) {
  const double P = h->peak_gflops * 1e9;
  const double BW = h->hbm_gbps * 1e9;
  const double m = static_cast<double>(M), n = static_cast<double>(N), k = static_cast<double>(K);
  const int sms = std::max(1, h->max_ctas > 0 ? std::min(h->max_ctas, h->num_sms) : h->num_sms);
  if (algo == LCGEMM_PLAIN) {
    const int bn = N <= 128 ? 128 : 256;
    const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
    const double flops = 2.0 * m * n * k;
    const double bytes = 2.0 * (m * k + k * n + m * n);
    const double t_mma = flops / (kEtaPlain * P * wave_efficiency(tiles, sms));
    return std::max(t_mma, bytes / (kBetaStream * BW)) + kLaunchSec;
  }
  return INFINITY;
}

int select_algo(const lcgemm_ctx* h, int64_t M, int64_t N, int64_t K, int dtype) {
  (void)dtype;
  int best = LCGEMM_PLAIN;
  double best_t = estimate_seconds(h, LCGEMM_PLAIN, M, N, K);
  for (int a : {LCGEMM_STRASSEN1, LCGEMM_STRASSEN2}) {
    if (!algo_supported(a, M, N, K)) continue;
    const double t = estimate_seconds(h, a, M, N, K);
    if (t < best_t) {
      best_t = t;
      best = a;
    }
  }
  return best;
}

int dispatch(lcgemm_ctx* h, int algo, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
             int64_t ldb, void* C, int64_t ldc, bool bf16, cudaStream_t st) {
  if (!algo_supported(algo, M, N, K)) return LCGEMM_ERR_UNSUPPORTED;
  switch (algo) {
    case LCGEMM_PLAIN:
      return run_plain(h, M, N, K, A, lda, B, ldb, C, ldc, bf16, st);
    case LCGEMM_STRASSEN1:
      return run_strassen(h, 1, true, M, N, K, A, lda, B, ldb, C, ldc, bf16, st);
    case LCGEMM_STRASSEN1_UNFUSED:
      return run_strassen(h, 1, false, M, N, K, A, lda, B, ldb, C, ldc, bf16, st);
    case LCGEMM_STRASSEN2:
      return run_strassen(h, 2, false, M, N, K, A, lda, B, ldb, C, ldc, bf16, st);
    default:
      return LCGEMM_ERR_UNSUPPORTED;
  }
}

}  // namespace lcg
