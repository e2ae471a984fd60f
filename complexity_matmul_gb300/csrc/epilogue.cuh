// The fused element-wise epilogue and the one rounding of C.
//
// Every kernel that finishes an output element hands a run of W consecutive
// FP32 values of one C row to store_run(): it applies
//
//     D = act(acc + bias[col]) + residual[row, col]
//
// in FP32 while the values are still in registers, rounds D once to the
// output type (round to nearest even) and stores it.  This is the fusion the
// DeepGEMM tuning blog describes in section 3.3 (bias broadcast onto the
// finished tile, a tanh-approximated GeLU, then the store) and the "bias +
// activation" / "residual" fusions of the "Fusion" section of "Kernel 与性能"
// (wineandchord.com kernels-performance): the epilogue costs no extra pass
// over C.
//
// GELU_TANH evaluates tanh with the hardware approximation (tanh.approx.f32),
// the fast tanh the DeepGEMM blog uses; GELU uses a published erfc
// approximation (gelu_erf below).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lcg {

__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x Phi(x) with Phi(x) = erfc(-x / sqrt 2) / 2.  erfc(z) for z >= 0 is the
// rational-times-Gaussian approximation of Abramowitz and Stegun, Handbook of
// Mathematical Functions, formula 7.1.26 (absolute error at most 1.5e-7):
//   erfc(z) ~ t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),  t = 1 / (1 + p z),
// and erfc(-z) = 2 - erfc(z).  The GELU's absolute error is then below
// 1e-7 |x| (as for the usual FP32 evaluation through erf), at two special-function
// unit operations per element instead of a full erfc.
__device__ __forceinline__ float gelu_erf(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.f, fmaf(0.3275911f, z, 1.f));
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  const float e = poly * t * __expf(-z * z);   // erfc(|x| / sqrt 2)
  return x * (x >= 0.f ? fmaf(-0.5f, e, 1.f) : 0.5f * e);
}

__device__ __forceinline__ float activate(float x, int act) {
  if (act == kActRelu) return x > 0.f ? x : 0.f;
  if (act == kActGelu) return gelu_erf(x);
  if (act == kActGeluTanh) {
    // sqrt(2/pi) * (x + 0.044715 x^3)
    const float u = 0.79788456080286536f * fmaf(0.044715f * x, x * x, x);
    return 0.5f * x * (1.f + tanh_hw(u));
  }
  return x;
}

// Two 16-bit values (low half first) of the output type to FP32.
template <bool BF16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if (BF16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  }
}

template <bool BF16>
__device__ __forceinline__ float unpack1(uint16_t b) {
  return BF16 ? __uint_as_float(static_cast<uint32_t>(b) << 16) : __half2float(__ushort_as_half(b));
}

// Adds W values of a 16-bit vector starting at p (16-byte aligned when vec) to v.
// RO: read through the read-only path (the bias, which no thread writes);
// otherwise a streaming load (the residual, read once, and possibly C itself).
template <bool BF16, int W, bool RO>
__device__ __forceinline__ void add_run(float (&v)[W], const uint16_t* p, int n, bool vec) {
  if (W % 8 == 0 && vec) {
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
      const uint4* src = reinterpret_cast<const uint4*>(p) + q;
      const uint4 u = RO ? __ldg(src) : __ldcs(src);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float lo, hi;
        unpack2<BF16>(w[t], lo, hi);
        v[8 * q + 2 * t] += lo;
        v[8 * q + 2 * t + 1] += hi;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < W; ++j)
      if (j < n) v[j] += unpack1<BF16>(p[j]);
  }
}

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// The bias and residual words of one run, loaded ahead of the run's epilogue
// so that their latency overlaps other work (the previous run's epilogue, the
// tensor-memory load, the partial sums of a split).  Only whole, 16-byte
// aligned runs are preloaded; store_run() loads anything else itself.
template <int W>
struct EpiLoads {
  static constexpr int kVec = W >= 8 ? W / 8 : 1;
  uint4 b[kVec];
  uint4 r[kVec];
  bool vb, vr;
};

template <int W>
__device__ __forceinline__ void epilogue_load(const Epilogue& e, int64_t row, int64_t col, int n, EpiLoads<W>& L) {
  L.vb = L.vr = false;
  if (!e.on || n != W) return;
  if (e.bias && aligned16(e.bias + col)) {
    L.vb = true;
#pragma unroll
    for (int q = 0; q < W / 8; ++q) L.b[q] = __ldg(reinterpret_cast<const uint4*>(e.bias + col) + q);
  }
  const uint16_t* rp = e.residual ? e.residual + row * e.ldr + col : nullptr;
  if (rp && aligned16(rp)) {
    L.vr = true;
#pragma unroll
    for (int q = 0; q < W / 8; ++q) L.r[q] = __ldcs(reinterpret_cast<const uint4*>(rp) + q);
  }
}

template <bool BF16, int W>
__device__ __forceinline__ void add_loaded(float (&v)[W], const uint4 (&u)[EpiLoads<W>::kVec]) {
#pragma unroll
  for (int q = 0; q < W / 8; ++q) {
    const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float lo, hi;
      unpack2<BF16>(w[t], lo, hi);
      v[8 * q + 2 * t] += lo;
      v[8 * q + 2 * t + 1] += hi;
    }
  }
}

// One rounding of v[0 .. n) to the output type and its store at dst (n <= W):
// 16-byte stores for a whole, aligned run, 2-byte stores otherwise.
template <bool BF16, int W>
__device__ __forceinline__ void cast_store(uint16_t* dst, int n, const float (&v)[W]) {
  if (W % 8 == 0 && n == W && aligned16(dst)) {
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
      uint4 o;
      o.x = pack2(v[8 * q + 0], v[8 * q + 1], BF16);
      o.y = pack2(v[8 * q + 2], v[8 * q + 3], BF16);
      o.z = pack2(v[8 * q + 4], v[8 * q + 5], BF16);
      o.w = pack2(v[8 * q + 6], v[8 * q + 7], BF16);
      reinterpret_cast<uint4*>(dst)[q] = o;
    }
  } else {
#pragma unroll
    for (int j = 0; j < W; j += 2) {
      const uint32_t p = pack2(v[j], j + 1 < W ? v[j + 1] : 0.f, BF16);
      if (j < n) dst[j] = static_cast<uint16_t>(p & 0xffffu);
      if (j + 1 < n) dst[j + 1] = static_cast<uint16_t>(p >> 16);
    }
  }
}

// The epilogue act(v + bias) + residual, in place, of v[0 .. n) = C[row, col ..
// col + n) (n <= W; the values past n are left as they are).  `pre`: this run's
// bias / residual words if epilogue_load() fetched them, else null.
template <bool BF16, int W>
__device__ __forceinline__ void apply_epilogue(int64_t row, int64_t col, int n, float (&v)[W], const Epilogue& e,
                                               const EpiLoads<W>* pre = nullptr) {
  const bool full = n == W;
  if (e.on) {
    if (e.bias) {
      if (pre && pre->vb) {
        add_loaded<BF16, W>(v, pre->b);
      } else {
        const uint16_t* bp = e.bias + col;
        add_run<BF16, W, true>(v, bp, n, full && aligned16(bp));
      }
    }
    // one branch per run, then a straight loop per activation
    if (e.act == kActRelu) {
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] = activate(v[j], kActRelu);
    } else if (e.act == kActGelu) {
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] = activate(v[j], kActGelu);
    } else if (e.act == kActGeluTanh) {
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] = activate(v[j], kActGeluTanh);
    }
    if (e.residual) {
      if (pre && pre->vr) {
        add_loaded<BF16, W>(v, pre->r);
      } else {
        const uint16_t* rp = e.residual + row * e.ldr + col;
        add_run<BF16, W, false>(v, rp, n, full && aligned16(rp));
      }
    }
  }
}

// Epilogue + cast + store of v[0 .. n) = C[row, col .. col + n); dst points at C[row, col].
template <bool BF16, int W>
__device__ __forceinline__ void store_run(uint16_t* dst, int64_t row, int64_t col, int n, float (&v)[W],
                                          const Epilogue& e, const EpiLoads<W>* pre = nullptr) {
  apply_epilogue<BF16, W>(row, col, n, v, e, pre);
  cast_store<BF16, W>(dst, n, v);
}

// A tensor store writes whole 16-byte units of a row: a unit that reaches past
// C's last column is written entire.  The maps of C therefore end at the last
// whole unit inside C (columns below N rounded down to a multiple of 8), and
// the rest of a row, fewer than 8 elements, is stored from registers here:
// v[j0 .. j1) of this lane's run, cast once; dst points at the run's first column.
template <bool BF16>
__device__ __forceinline__ void store_cols(uint16_t* dst, const float (&v)[32], int j0, int j1) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j >= j0 && j < j1) dst[j] = static_cast<uint16_t>(pack2(v[j], 0.f, BF16) & 0xffffu);
}

// Cast of one 32 x 32 chunk of C (lane = row, v = its 32 columns) into a
// shared-memory box of 32 rows x 64 bytes for a tensor store, laid out in the
// tensor map's 64-byte swizzle: 16-byte unit j of row r at r * 64 +
// (j ^ ((r >> 1) & 3)) * 16, so that the warp's stores of one unit hit every
// bank once per quarter warp.  The caller fences the async proxy before the
// store reads the box.
template <bool BF16>
__device__ __forceinline__ void stage_chunk(uint32_t box, int lane, const float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t addr = box + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pack2(v[8 * j], v[8 * j + 1], BF16)),
                 "r"(pack2(v[8 * j + 2], v[8 * j + 3], BF16)), "r"(pack2(v[8 * j + 4], v[8 * j + 5], BF16)),
                 "r"(pack2(v[8 * j + 6], v[8 * j + 7], BF16))
                 : "memory");
  }
}

}  // namespace lcg
