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

__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

}  // namespace lcg
