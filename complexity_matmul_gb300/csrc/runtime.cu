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

#include "kernels.h"
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
    case LCGEMM_STRASSEN2:
      // any shape: non-divisible dimensions run on zero-padded operand copies
      return M >= 1 && N >= 1 && K >= 1;
    default:
      return false;
  }
}

namespace {

// Calibration: the fraction of the dense tensor peak each product kernel
// sustains once its tile grid fills the machine, and the fraction of HBM
// bandwidth the streaming kernels reach.  Measured on GB300 (1 CTA per SM).
constexpr double kEtaPlainPair = 0.86;    // CTA-pair 256 x 256 tiles
constexpr double kEtaPlainSingle = 0.78;  // single-CTA 128 x 256 tiles
constexpr double kEtaLcmaSingle = 0.55;   // single-CTA 128 x 128 product tiles (shared-memory bound)
// Fused one-level Groups on CTA pairs (256 x 256, 7 products): each product
// streams the same operand bytes per flop as a plain CTA-pair tile, but every
// switch to the next product's operand panels costs about this many 64-deep K
// slabs of MMA time (pipeline refill from L2 misses), so the products run at
// kEtaPlainPair * (1 - kLcmaSwitchSlabs / slabs per product).  Measured on
// GB300 against the plain kernel in the same process: 0.76 of its rate at 32
// slabs per product, 0.87-0.89 at 64, 0.93 at 128.
constexpr double kLcmaSwitchSlabs = 8.0;
constexpr double kBetaStream = 0.80;      // combine pre-pass / recombination, fraction of HBM bandwidth
constexpr double kLaunchSec = 6e-6;       // launch + prologue + pipeline fill of one kernel

double wave_efficiency(int64_t tiles, int units) {
  if (tiles <= 0 || units <= 0) return 1.0;
  const int64_t waves = (tiles + units - 1) / units;
  return static_cast<double>(tiles) / static_cast<double>(waves * units);
}

// Same with the tail split: when the partial last wave fits twice over, its
// Groups run as halves (the longer half is 4 of 7 products).
double wave_efficiency_split(int64_t tiles, int units) {
  if (tiles <= 0 || units <= 0) return 1.0;
  const int64_t full = tiles / units, rem = tiles - full * units;
  const double waves = static_cast<double>(full) + (rem == 0 ? 0.0 : (2 * rem <= units ? 4.0 / 7.0 : 1.0));
  return static_cast<double>(tiles) / (waves * units);
}

// One kernel on the roofline: compute time at eta * peak stretched by wave
// quantisation, or streaming time, whichever is longer, plus launch overhead.
double kernel_time(double flops, double bytes, int64_t tiles, int units, double eta, double P, double BW) {
  const double t_c = flops > 0 ? flops / (eta * P * wave_efficiency(tiles, units)) : 0.0;
  const double t_m = bytes / (kBetaStream * BW);
  return std::max(t_c, t_m) + kLaunchSec;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

double estimate_divisible(const lcgemm_ctx* h, int algo, int64_t M, int64_t N, int64_t K, double P, double BW,
                          int sms);

double estimate_seconds(const lcgemm_ctx* h, int algo, int64_t M, int64_t N, int64_t K) {
  const double P = h->peak_gflops * 1e9;
  const double BW = h->hbm_gbps * 1e9;
  const double m = static_cast<double>(M), n = static_cast<double>(N), k = static_cast<double>(K);
  const int sms = std::max(1, h->max_ctas > 0 ? std::min(h->max_ctas, h->num_sms) : h->num_sms);
  const double mnk2 = 2.0 * m * n * k;
  if (algo == LCGEMM_PLAIN) {
    const double bytes = 2.0 * (m * k + k * n + m * n);
    const int64_t pair_tiles = cdiv(M, 256) * cdiv(N, 256);
    const bool pair = sms >= 2 && (h->plain_kernel == 2 || h->plain_kernel == 5 ||
                                   (h->plain_kernel == 0 && M > 128 && N > 128 && pair_tiles >= sms / 4));
    if (pair) {
      // waves of 256 x 256 or 256 x 512 tiles (the dispatcher's width), the partial
      // last wave as K halves when it is split; wide tiles do more per unit of time
      const int units = sms / 2;
      const int bn = h->plain_kernel == 2 ? 256 : h->plain_kernel == 5 ? 512
                                                 : pair_tile_bn(M, N, K, units, h->split != 0);
      const double eff = static_cast<double>(pair_tiles) / (units * pair_waves(M, N, K, bn, units, h->split != 0));
      const double eta = kEtaPlainPair * (bn == 512 ? kWideTileGain : 1.0);
      return std::max(mnk2 / (eta * P * eff), bytes / (kBetaStream * BW)) + kLaunchSec;
    }
    // single-CTA tiles with the launcher's split-K: tiles x chunks work items, FP32
    // partials written and read back, deep splits summed by a separate kernel
    const int64_t bn = plain_single_bn(M, N, sms);
    const int64_t tiles = cdiv(M, 128) * cdiv(N, bn), num_kb = cdiv(K, 64);
    int64_t splits = 1;
    if (tiles < sms / 2 && num_kb >= kSplitKMinSlabs) splits = std::max<int64_t>(1, std::min<int64_t>(sms / tiles, num_kb / 16));
    const double part_bytes = splits > 1 ? 2.0 * 4.0 * static_cast<double>(tiles * splits) * 128.0 * bn : 0.0;
    double t = kernel_time(mnk2, bytes + part_bytes, tiles * splits, sms, kEtaPlainSingle, P, BW);
    if (splits >= kSeparateReduceSplits) t += kernel_time(0, part_bytes / 2 + 2.0 * m * n, 0, 1, 1.0, P, BW);
    return t;
  }
  if (!algo_supported(algo, M, N, K)) return INFINITY;
  // non-divisible shapes run on zero-padded copies: the copy (read the operands,
  // write the padded ones) comes first, then the algorithm on the padded extents
  const int64_t G = algo == LCGEMM_STRASSEN2 ? 4 : 2;
  const int64_t Mp = cdiv(M, G) * G, Np = cdiv(N, 8 * G) * 8 * G, Kp = cdiv(K, 8 * G) * 8 * G;
  const bool pad_a = Mp != M || Kp != K, pad_b = Np != N || Kp != K;
  double t_pad = 0.0;
  if (pad_a || pad_b) {
    const double kp = static_cast<double>(Kp);
    const double bytes = (pad_a ? 2.0 * m * k + 2.0 * static_cast<double>(Mp) * kp : 0.0) +
                         (pad_b ? 2.0 * n * k + 2.0 * static_cast<double>(Np) * kp : 0.0);
    t_pad = kernel_time(0, bytes, 0, 1, 1.0, P, BW);
    M = Mp;
    N = Np;
    K = Kp;
  }
  return t_pad + estimate_divisible(h, algo, M, N, K, P, BW, sms);
}

// Strassen time on divisible extents.
double estimate_divisible(const lcgemm_ctx* h, int algo, int64_t M, int64_t N, int64_t K, double P, double BW,
                          int sms) {
  const double m = static_cast<double>(M), n = static_cast<double>(N), k = static_cast<double>(K);
  const double mnk2 = 2.0 * m * n * k;
  if (algo == LCGEMM_STRASSEN1 || algo == LCGEMM_STRASSEN1_UNFUSED) {
    const int64_t mb = M / 2, nb = N / 2;
    // pre-pass: read A and B once, write 5 summed blocks of each (2 of 7 products alias raw blocks)
    const double t_pre = kernel_time(0, 4.5 * (m * k + k * n), 0, 1, 1.0, P, BW);
    const double flops = 7.0 / 8.0 * mnk2;
    if (algo == LCGEMM_STRASSEN1) {
      const double bytes = 3.5 * (m * k + k * n) + 2.0 * m * n;
      const bool pair = sms >= 2 && (h->lcma_kernel == 2 || (h->lcma_kernel == 0 && mb > 128));
      if (pair) {
        const int64_t groups = cdiv(mb, 256) * cdiv(nb, 256);
        const double eff = h->split ? wave_efficiency_split(groups, sms / 2) : wave_efficiency(groups, sms / 2);
        const double slabs = static_cast<double>(cdiv(K / 2, 64));
        const double eta = kEtaPlainPair * std::max(0.1, 1.0 - kLcmaSwitchSlabs / slabs);
        const double t = std::max(flops / (eta * P * eff), bytes / (kBetaStream * BW)) + kLaunchSec;
        return t_pre + t;
      }
      return t_pre + kernel_time(flops, bytes, cdiv(mb, 128) * cdiv(nb, 128), sms, kEtaLcmaSingle, P, BW);
    }
    const double t_prod = kernel_time(flops, 3.5 * (m * k + k * n) + 7.0 * m * n, 7 * cdiv(mb, 128) * cdiv(nb, 128),
                                      sms, kEtaLcmaSingle, P, BW);
    const double t_h = kernel_time(0, 9.0 * m * n, 0, 1, 1.0, P, BW);
    return t_pre + t_prod + t_h;
  }
  if (algo == LCGEMM_STRASSEN2) {
    const int64_t mb = M / 4, nb = N / 4;
    const double t_pre = kernel_time(0, 7.625 * (m * k + k * n), 0, 1, 1.0, P, BW);
    const double flops = 49.0 / 64.0 * mnk2;
    const bool pair = sms >= 2 && (h->lcma_kernel == 2 || (h->lcma_kernel == 0 && mb > 128));
    if (pair) {
      // hierarchical: seven launches of the one-level CTA-pair kernel over the inner
      // (M/4 x N/4) grid; the outer level goes through three FP32 slots of M/2 x N/2
      // (eight slot writes and eight reads of MN bytes each, then C)
      const int64_t groups = cdiv(mb, 256) * cdiv(nb, 256);
      const double eff = h->split ? wave_efficiency_split(groups, sms / 2) : wave_efficiency(groups, sms / 2);
      const double slabs = static_cast<double>(cdiv(K / 4, 64));
      const double eta = kEtaPlainPair * std::max(0.1, 1.0 - kLcmaSwitchSlabs / slabs);
      const double bytes = (6.125 * (m * k + k * n) + 16.0 * m * n + 2.0 * m * n) / 7.0;   // per launch
      const double t = std::max(flops / 7.0 / (eta * P * eff), bytes / (kBetaStream * BW)) + kLaunchSec;
      return t_pre + 7.0 * t;
    }
    // unfused: 49 FP32 products of (M/4 x N/4) written and read back, then C
    const double t_prod = kernel_time(flops, 6.125 * (m * k + k * n) + 12.25 * m * n,
                                      49 * cdiv(mb, 128) * cdiv(nb, 128), sms, kEtaLcmaSingle, P, BW);
    const double t_h = kernel_time(0, 14.25 * m * n, 0, 1, 1.0, P, BW);
    return t_pre + t_prod + t_h;
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
             int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep, cudaStream_t st) {
  if (!algo_supported(algo, M, N, K)) return LCGEMM_ERR_UNSUPPORTED;
  switch (algo) {
    case LCGEMM_PLAIN:
      return run_plain(h, M, N, K, A, lda, B, ldb, C, ldc, bf16, ep, st);
    case LCGEMM_STRASSEN1:
      return run_strassen(h, 1, true, M, N, K, A, lda, B, ldb, C, ldc, bf16, ep, st);
    case LCGEMM_STRASSEN1_UNFUSED:
      return run_strassen(h, 1, false, M, N, K, A, lda, B, ldb, C, ldc, bf16, ep, st);
    case LCGEMM_STRASSEN2:
      return run_strassen(h, 2, true, M, N, K, A, lda, B, ldb, C, ldc, bf16, ep, st);
    default:
      return LCGEMM_ERR_UNSUPPORTED;
  }
}

}  // namespace lcg
