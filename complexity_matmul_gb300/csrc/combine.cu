// Combine-A/B pre-pass and Combine-H recombination for the LCMA path.
//
// FalconGEMM write-up (hyper.ai news 54396, section "从 LCMA 到 FalconGEMM"):
// the basic GPU Strassen pipeline first combines sub-blocks of A and of B into
// the operands of the 7 products; the input-side combination is kept as a
// separate pass because one summed block is read by many SMs (fusing it into
// the GEMM would repeat the loads and the sums).  This kernel reads every
// element of A and B once and writes each summed operand block once.  Sums are
// formed in FP32 in ascending block order and rounded once (round to nearest
// even) to the input type.  Products whose operand is a single raw block with
// coefficient +1 read that block in place and get no workspace slot.
//
// The recombination kernel (C_q = sum_p W[q,p] M_p from FP32 products in
// HBM) is the last step of the basic, unfused pipeline; the fused path folds
// it into the product kernel's epilogue instead.
#include <utility>

#include "epilogue.cuh"
#include "kernels.h"
#include "lcma_tables.h"
#include "ptx.cuh"

namespace lcg {

namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8], bool bf16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0xffffu, hi = w[i] >> 16;
    if (bf16) {
      f[2 * i] = __uint_as_float(lo << 16);
      f[2 * i + 1] = __uint_as_float(hi << 16);
    } else {
      f[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(lo)));
      f[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(hi)));
    }
  }
}

// One summed operand (product P, side SIDE), all indices compile-time constants.
template <int L, int SIDE, int P, bool BF16, int G>
__device__ __forceinline__ void combine_product(const uint4 (&x)[G][G], const CombineSide& s, int64_t i, int64_t k) {
  constexpr LcmaPlan<L> plan{};
  constexpr int slot = plan.side[SIDE].slot[P];
  if constexpr (slot >= 0) {
    constexpr int nt = plan.side[SIDE].nterm[P];
    float acc[8];
#pragma unroll
    for (int t = 0; t < nt; ++t) {
      // math block (R, C); A is stored by (R, C), B (K x N stored N x K) by (C, R)
      const int r = plan.side[SIDE].term_r[P][t], c = plan.side[SIDE].term_c[P][t];
      const int srb = SIDE == 0 ? r : c, scb = SIDE == 0 ? c : r;
      float f[8];
      unpack8(x[srb][scb], f, BF16);
      const float sg = static_cast<float>(plan.side[SIDE].term_s[P][t]);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = (t == 0) ? sg * f[e] : acc[e] + sg * f[e];
    }
    uint4 o;
    o.x = pack2(acc[0], acc[1], BF16);
    o.y = pack2(acc[2], acc[3], BF16);
    o.z = pack2(acc[4], acc[5], BF16);
    o.w = pack2(acc[6], acc[7], BF16);
    *reinterpret_cast<uint4*>(s.dst + slot * s.slot_stride + i * s.dst_ld + k) = o;
  }
}

template <int L, int SIDE, bool BF16, int G, int... Ps>
__device__ __forceinline__ void combine_all(const uint4 (&x)[G][G], const CombineSide& s, int64_t i, int64_t k,
                                            std::integer_sequence<int, Ps...>) {
  (combine_product<L, SIDE, Ps, BF16, G>(x, s, i, k), ...);
}

template <int L, int SIDE, bool BF16>
__device__ __forceinline__ void combine_vec(const CombineSide& s, int64_t v) {
  constexpr int G = 1 << L;
  const int64_t kvecs = s.kb / 8;
  const int64_t i = v / kvecs;
  const int64_t k = (v - i * kvecs) * 8;
  // x[srb][scb]: storage row block srb, storage column block scb (storage = rows x K)
  uint4 x[G][G];
#pragma unroll
  for (int rb = 0; rb < G; ++rb)
#pragma unroll
    for (int cb = 0; cb < G; ++cb)
      x[rb][cb] = __ldg(reinterpret_cast<const uint4*>(s.src + (rb * s.rows_b + i) * s.ld + cb * s.kb + k));
  combine_all<L, SIDE, BF16, G>(x, s, i, k, std::make_integer_sequence<int, ipow(7, L)>{});
}

template <int L, bool BF16>
__global__ void __launch_bounds__(256) combine_ab_kernel(const __grid_constant__ CombineArgs args) {
  griddep_launch_dependents();   // the product kernel may be scheduled now; it waits for this grid's writes
  const int64_t na = args.side[0].vecs;
  const int64_t total = na + args.side[1].vecs;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < total; v += int64_t(gridDim.x) * blockDim.x) {
    if (v < na)
      combine_vec<L, 0, BF16>(args.side[0], v);
    else
      combine_vec<L, 1, BF16>(args.side[1], v - na);
  }
}

// C block (R, C) = sum_p W[(R,C), p] * P_p, FP32 products [R][Mb][ldp] -> C (dtype).
template <int L, bool BF16>
__global__ void __launch_bounds__(256) combine_h_kernel(const __grid_constant__ CombineHArgs a) {
  griddep_wait();   // the products come from the kernel before this one
  constexpr int G = 1 << L;
  constexpr int R = ipow(7, L);
  constexpr WTable<L> wt{};
  const int64_t nvec = (a.nb + 3) / 4;
  const int64_t total = int64_t(a.mb) * nvec;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < total; v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t i = v / nvec;
    const int64_t j = (v - i * nvec) * 4;
#pragma unroll
    for (int br = 0; br < G; ++br)
#pragma unroll
      for (int bc = 0; bc < G; ++bc) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < R; ++p) {
          const int w = wt.w[br][bc][p];
          if (w == 0) continue;
          const float4 m = *reinterpret_cast<const float4*>(a.prod + (p * int64_t(a.mb) + i) * a.ldp + j);
          acc[0] += w * m.x;
          acc[1] += w * m.y;
          acc[2] += w * m.z;
          acc[3] += w * m.w;
        }
        const int64_t row = br * int64_t(a.mb) + i;
        const int64_t gcol = bc * int64_t(a.nb) + j;
        if (row >= a.M || gcol >= a.N) continue;
        uint16_t* crow = a.C + row * a.ldc + bc * int64_t(a.nb);
        int n = static_cast<int>(a.nb - j < 4 ? a.nb - j : 4);
        if (a.N - gcol < n) n = static_cast<int>(a.N - gcol);
        store_run<BF16, 4>(crow + j, row, gcol, n, acc, a.ep);
      }
  }
}

// Zero-padded copy of both operands: dst row r = src row r (K values) then
// zeros up to kp; rows >= rows_src are all zeros.  One thread per 8 elements of
// the destination; 16-byte loads where a run of 8 lies inside the source row.
__global__ void __launch_bounds__(256) pad_copy_kernel(const __grid_constant__ PadArgs a) {
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < a.vecs[0] + a.vecs[1];
       v += int64_t(gridDim.x) * blockDim.x) {
    const int s = v < a.vecs[0] ? 0 : 1;
    const PadSide& p = a.side[s];
    const int64_t w = s == 0 ? v : v - a.vecs[0];
    const int64_t per_row = p.kp / 8;
    const int64_t r = w / per_row;
    const int64_t k = (w - r * per_row) * 8;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (r < p.rows) {
      const uint16_t* src = p.src + r * p.ld + k;
      if (k + 8 <= p.k) {
        out = *reinterpret_cast<const uint4*>(src);
      } else if (k < p.k) {
        uint16_t e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e[i] = k + i < p.k ? src[i] : uint16_t(0);
        out = make_uint4(e[0] | (uint32_t(e[1]) << 16), e[2] | (uint32_t(e[3]) << 16), e[4] | (uint32_t(e[5]) << 16),
                         e[6] | (uint32_t(e[7]) << 16));
      }
    }
    *reinterpret_cast<uint4*>(p.dst + r * p.kp + k) = out;
  }
}

template <typename K, typename Args>
cudaError_t launch_grid_stride(K kern, const Args& a, int64_t total, int num_sms, cudaStream_t st) {
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  blocks = blocks < int64_t(num_sms) * 8 ? blocks : int64_t(num_sms) * 8;
  if (blocks < 1) blocks = 1;
  kern<<<static_cast<int>(blocks), threads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine_ab(const CombineArgs& a, int levels, bool bf16, int num_sms, cudaStream_t st) {
  const int64_t total = a.side[0].vecs + a.side[1].vecs;
  if (total == 0) return cudaSuccess;
  if (levels == 1)
    return bf16 ? launch_grid_stride(combine_ab_kernel<1, true>, a, total, num_sms, st)
                : launch_grid_stride(combine_ab_kernel<1, false>, a, total, num_sms, st);
  if (levels == 2)
    return bf16 ? launch_grid_stride(combine_ab_kernel<2, true>, a, total, num_sms, st)
                : launch_grid_stride(combine_ab_kernel<2, false>, a, total, num_sms, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_pad_copy(const PadArgs& a, int num_sms, cudaStream_t st) {
  const int64_t total = a.vecs[0] + a.vecs[1];
  if (total == 0) return cudaSuccess;
  return launch_grid_stride(pad_copy_kernel, a, total, num_sms, st);
}

cudaError_t launch_combine_h(const CombineHArgs& a, int levels, bool bf16, int num_sms, cudaStream_t st, bool pdl) {
  const int64_t total = int64_t(a.mb) * ((a.nb + 3) / 4);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  blocks = blocks < int64_t(num_sms) * 8 ? blocks : int64_t(num_sms) * 8;
  const int g = static_cast<int>(blocks < 1 ? 1 : blocks);
  if (levels == 1)
    return bf16 ? launch_maybe_pdl(combine_h_kernel<1, true>, g, 256, 0, st, pdl, a)
                : launch_maybe_pdl(combine_h_kernel<1, false>, g, 256, 0, st, pdl, a);
  if (levels == 2)
    return bf16 ? launch_maybe_pdl(combine_h_kernel<2, true>, g, 256, 0, st, pdl, a)
                : launch_maybe_pdl(combine_h_kernel<2, false>, g, 256, 0, st, pdl, a);
  return cudaErrorInvalidValue;
}

}  // namespace lcg
