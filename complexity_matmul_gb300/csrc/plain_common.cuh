// Device helpers shared by the plain GEMM kernels (gemm_plain.cu, gemm_pair.cu).
#pragma once

#include <cstdint>

#include "epilogue.cuh"
#include "kernels.h"

namespace lcg {

// Grouped raster: tiles are numbered down bands of `group_m` tile rows, one
// tile column after another, so that a wave of consecutive tiles shares a few
// A panels and B panels in L2.
__device__ __forceinline__ void tile_coords(int tile, const PlainArgs& a, int& mb, int& nb) {
  const int group_tiles = a.group_m * a.tiles_n;
  const int g = tile / group_tiles;
  const int first_m = g * a.group_m;
  const int rows = min(a.tiles_m - first_m, a.group_m);
  const int local = tile - g * group_tiles;
  mb = first_m + local % rows;
  nb = local / rows;
}

// Epilogue (EPI), cast and store of 32 FP32 values of one C row (columns col .. col+31,
// clipped to C).
template <bool BF16, bool EPI>
__device__ __forceinline__ void store_chunk(uint16_t* crow, int row, int col, const uint32_t (&r)[32],
                                            const PlainArgs& args, const EpiLoads<32>* pre = nullptr) {
  if (row >= args.M || col >= args.N) return;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  if constexpr (EPI) store_run<BF16, 32>(crow + col, row, col, min(32, args.N - col), v, args.ep, pre);
  else cast_store<BF16, 32>(crow + col, min(32, args.N - col), v);
}

// Issues the bias / residual loads of the 32-column chunk at (row, col), if it lies in C.
__device__ __forceinline__ void load_chunk(int row, int col, const PlainArgs& args, EpiLoads<32>& pre) {
  if (row < args.M && col < args.N)
    epilogue_load<32>(args.ep, row, col, min(32, args.N - col), pre);
  else
    pre.vb = pre.vr = false;
}

// Split-K partial sums.  A slot holds one K chunk's FP32 partial of one tile
// column-major: element (row r, column j) at j * ld + r.  The 32 lanes of an
// epilogue warp hold 32 consecutive rows (the tcgen05.ld 32x32b layout: lane =
// row, register = column), so every warp-wide access below covers 128
// contiguous bytes, one cache line, instead of 32 lines.
// p points at (this lane's row, the first of the 32 columns) of the slot.
__device__ __forceinline__ void publish_partial(float* p, int ld, const uint32_t (&r)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) __stcg(p + j * ld, __uint_as_float(r[j]));
}

// Sum of the S chunks' partials of 32 columns of one row, in chunk order
// (slots slot_stride floats apart); all 32 x S loads are issued before the sums.
template <int S>
__device__ __forceinline__ void sum_partials(const float* p, int ld, int64_t slot_stride, uint32_t (&r)[32]) {
  float x[S][32];
#pragma unroll
  for (int s = 0; s < S; ++s)
#pragma unroll
    for (int j = 0; j < 32; ++j) x[s][j] = __ldcg(p + s * slot_stride + j * ld);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float a = 0.f;
#pragma unroll
    for (int s = 0; s < S; ++s) a += x[s][j];
    r[j] = __float_as_uint(a);
  }
}

__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

}  // namespace lcg
