// Host side of the LCMA path: workspace, the Combine-A/B pre-pass and the
// product kernels for one- and two-level Strassen.
#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "lcgemm.h"
#include "lcma_tables.h"
#include "runtime.h"

namespace lcg {

namespace {

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus s = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &s) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return s != cudaStreamCaptureStatusNone;
}

// Grow the handle's workspace to at least `bytes` (stream-ordered with `st`).
int ensure_workspace(lcgemm_ctx* h, size_t bytes, cudaStream_t st) {
  if (bytes <= h->ws_bytes) return LCGEMM_OK;
  if (capturing(st)) return LCGEMM_ERR_CAPTURE;
  if (h->ws) {
    cudaStreamSynchronize(st);
    cudaFree(h->ws);
    h->ws = nullptr;
    h->ws_bytes = 0;
  }
  if (cudaMalloc(&h->ws, bytes) != cudaSuccess) {
    h->ws = nullptr;
    cudaGetLastError();
    return LCGEMM_ERR_NOMEM;
  }
  h->ws_bytes = bytes;
  return LCGEMM_OK;
}

namespace {

// Outer level of hierarchical two-level Strassen: the order of the 7 outer
// products (one launch each) and where each launch's product P goes, over
// three FP32 outer slots of M/2 x N/2.  The order M5 M3 M7 M1 M4 M2 M6 keeps
// at most three outer quadrants live (C12 retires after M3, C11 after M4,
// C21 after M2, C22 after M6).
struct OuterStep {
  int product;
  LcmaOuterTarget t[2];
};
constexpr OuterStep kOuterProgram[7] = {
    {4, {{kOuterInit, 0, -1, 0}, {kOuterInit, 1, 1, 1}}},    // M5: s0 = -P (C11), s1 = P (C12)
    {2, {{kOuterFinal, 1, 1, 1}, {kOuterInit, 1, 1, 3}}},   // M3: C12 = s1 + P; s1 = P (C22)
    {6, {{kOuterAcc, 0, 1, 0}, {kOuterNone, 0, 0, 0}}},     // M7: s0 += P
    {0, {{kOuterAcc, 0, 1, 0}, {kOuterAcc, 1, 1, 3}}},      // M1: s0 += P, s1 += P
    {3, {{kOuterFinal, 0, 1, 0}, {kOuterInit, 2, 1, 2}}},   // M4: C11 = s0 + P; s2 = P (C21)
    {1, {{kOuterFinal, 2, 1, 2}, {kOuterAcc, 1, -1, 3}}},   // M2: C21 = s2 + P; s1 -= P
    {5, {{kOuterFinal, 1, 1, 3}, {kOuterNone, 0, 0, 0}}},   // M6: C22 = s1 + P
};

// Symbolic run: every outer quadrant is stored once and equals sum_p W[q,p] P_p;
// within a step, a target that reads a slot comes before one that rewrites it.
constexpr bool outer_program_ok() {
  int slot[3][7] = {};
  bool written[3] = {};
  bool done[4] = {};
  for (const OuterStep& st : kOuterProgram) {
    for (int i = 0; i < 2; ++i) {
      const LcmaOuterTarget t = st.t[i];
      if (t.kind == kOuterNone) continue;
      if (t.kind != kOuterInit && !written[t.slot]) return false;
      if (t.kind == kOuterInit) {
        for (int j = 0; j < 7; ++j) slot[t.slot][j] = 0;
        slot[t.slot][st.product] = t.sign;
        written[t.slot] = true;
      } else if (t.kind == kOuterAcc) {
        slot[t.slot][st.product] += t.sign;
      } else {
        if (done[t.quad]) return false;
        done[t.quad] = true;
        for (int j = 0; j < 7; ++j)
          if (slot[t.slot][j] + (j == st.product ? t.sign : 0) != kW1[t.quad][j]) return false;
      }
    }
    if (st.t[0].kind == kOuterInit && st.t[1].kind >= kOuterAcc && st.t[0].slot == st.t[1].slot) return false;
  }
  return done[0] && done[1] && done[2] && done[3];
}
static_assert(outer_program_ok(), "the outer program must compute C_q = sum_p W[q,p] P_p");

// M, N, K: the (divisible) operand extents; Mc x Nc: C's extents (smaller when the
// operands are zero-padded copies).
template <int L>
int run_levels(lcgemm_ctx* h, bool fused, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
               const void* B, int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep, cudaStream_t st,
               int64_t Mc, int64_t Nc) {
  constexpr LcmaPlan<L> plan{};
  constexpr int G = plan.G;
  const int64_t mb = M / G, nb = N / G, kb = K / G;
  const int na = plan.side[0].nslots, nbs = plan.side[1].nslots;
  const int64_t a_bytes = round_up(na * mb * kb * 2, 256);
  const int64_t b_bytes = round_up(nbs * nb * kb * 2, 256);
  // fused Groups run on CTA pairs (256 x 256 tiles) unless the block is small; one level
  // also has the single-CTA fused kernel, two levels otherwise run unfused
  const bool pair = fused && grid_cap(h) >= 2 && (h->lcma_kernel == 2 || (h->lcma_kernel == 0 && mb > 128));
  if (L == 2 && !pair) fused = false;
  const bool hier = L == 2 && pair;           // seven launches, one per outer product
  const int64_t mbp = round_up(mb, 256), nbp = round_up(nb, 256);
  const int64_t ldp = round_up(nb, 4);
  const int64_t p_bytes = fused ? 0 : round_up(int64_t(plan.R) * mb * ldp * 4, 256);
  const int64_t s_bytes = fused ? round_up(static_cast<int64_t>(lcma_pair_scratch_bytes(grid_cap(h))), 256) : 0;
  const int launches = hier ? 7 : 1;
  const int64_t f_bytes = fused ? round_up(int64_t(sizeof(int)) * grid_cap(h) * launches, 256) : 0;   // split flags
  const int64_t o_bytes = hier ? 3 * (2 * mbp) * (2 * nbp) * 4 : 0;                                // outer slots
  int rc = ensure_workspace(h, static_cast<size_t>(a_bytes + b_bytes + p_bytes + s_bytes + f_bytes + o_bytes), st);
  if (rc) return rc;
  uint16_t* wsA = static_cast<uint16_t*>(h->ws);
  uint16_t* wsB = reinterpret_cast<uint16_t*>(static_cast<char*>(h->ws) + a_bytes);
  float* prod = reinterpret_cast<float*>(static_cast<char*>(h->ws) + a_bytes + b_bytes);
  float* scratch = reinterpret_cast<float*>(static_cast<char*>(h->ws) + a_bytes + b_bytes + p_bytes);
  float* oslot =
      reinterpret_cast<float*>(static_cast<char*>(h->ws) + a_bytes + b_bytes + p_bytes + s_bytes + f_bytes);

  // ---- Combine-A/B pre-pass
  CombineArgs ca{};
  ca.side[0] = CombineSide{static_cast<const uint16_t*>(A), lda, wsA, kb, mb * kb, mb, kb, mb * kb / 8};
  ca.side[1] = CombineSide{static_cast<const uint16_t*>(B), ldb, wsB, kb, nb * kb, nb, kb, nb * kb / 8};
  // the split-Group flags are cleared before the pre-pass, so that the product kernel
  // directly follows the pre-pass and can be launched as its programmatic dependent
  int* flags = fused ? reinterpret_cast<int*>(static_cast<char*>(h->ws) + a_bytes + b_bytes + p_bytes + s_bytes)
                     : nullptr;
  if (fused && cudaMemsetAsync(flags, 0, static_cast<size_t>(f_bytes), st) != cudaSuccess) return LCGEMM_ERR_CUDA;
  if (launch_combine_ab(ca, L, bf16, h->num_sms, st) != cudaSuccess) return LCGEMM_ERR_CUDA;

  // ---- products
  const int b_box = 128;
  LcmaLaunch ll{};
  ll.levels = L;
  ll.bf16 = bf16;
  ll.pdl = h->pdl != 0;
  // CTA-pair kernel: summed operands as one 2-D (slots * rows) x kb map; raw
  // blocks as a 2-D map of the whole operand when kb is a multiple of 64.
  const bool raw2d = pair && kb % 64 == 0;
  {
    const uint64_t dA[3] = {uint64_t(kb), uint64_t(mb), uint64_t(na)};
    const uint64_t sA[2] = {uint64_t(kb) * 2, uint64_t(mb * kb) * 2};
    const uint32_t boxA3[3] = {64u, 128u, 1u};
    const uint32_t boxB3[3] = {64u, uint32_t(b_box), 1u};
    const uint64_t dB[3] = {uint64_t(kb), uint64_t(nb), uint64_t(nbs)};
    const uint64_t sB[2] = {uint64_t(kb) * 2, uint64_t(nb * kb) * 2};
    if (pair) {
      if (!encode_kmajor(&ll.tmA_sum, bf16, wsA, int64_t(na) * mb, kb, kb, 128)) return LCGEMM_ERR_CUDA;
      if (!encode_kmajor(&ll.tmB_sum, bf16, wsB, int64_t(nbs) * nb, kb, kb, b_box)) return LCGEMM_ERR_CUDA;
    } else {
      if (!encode_map(&ll.tmA_sum, bf16, wsA, 3, dA, sA, boxA3)) return LCGEMM_ERR_CUDA;
      if (!encode_map(&ll.tmB_sum, bf16, wsB, 3, dB, sB, boxB3)) return LCGEMM_ERR_CUDA;
    }
    const uint32_t boxA4[4] = {64u, 1u, 128u, 1u};
    const uint32_t boxB4[4] = {64u, 1u, uint32_t(b_box), 1u};
    const uint64_t rA[4] = {uint64_t(kb), uint64_t(G), uint64_t(mb), uint64_t(G)};
    const uint64_t rsA[3] = {uint64_t(kb) * 2, uint64_t(lda) * 2, uint64_t(mb * lda) * 2};
    const uint64_t rB[4] = {uint64_t(kb), uint64_t(G), uint64_t(nb), uint64_t(G)};
    const uint64_t rsB[3] = {uint64_t(kb) * 2, uint64_t(ldb) * 2, uint64_t(nb * ldb) * 2};
    if (raw2d) {
      if (!encode_kmajor(&ll.tmA_raw, bf16, A, M, K, lda, 128)) return LCGEMM_ERR_CUDA;
      if (!encode_kmajor(&ll.tmB_raw, bf16, B, N, K, ldb, b_box)) return LCGEMM_ERR_CUDA;
    } else {
      if (!encode_map(&ll.tmA_raw, bf16, A, 4, rA, rsA, boxA4)) return LCGEMM_ERR_CUDA;
      if (!encode_map(&ll.tmB_raw, bf16, B, 4, rB, rsB, boxB4)) return LCGEMM_ERR_CUDA;
    }
  }
  LcmaArgs& a = ll.args;
  a.C = C;
  a.ldc = ldc;
  a.mb = static_cast<int>(mb);
  a.nb = static_cast<int>(nb);
  a.kb = static_cast<int>(kb);
  a.tiles_m = static_cast<int>(pair ? (mb + 255) / 256 : (mb + 127) / 128);
  a.tiles_n = static_cast<int>(pair ? (nb + 255) / 256 : (nb + 127) / 128);
  a.num_groups = a.tiles_m * a.tiles_n;
  a.group_m = pair ? 8 : 12;   // ~square wave footprint: sqrt(#pairs) resp. sqrt(#CTAs) tile rows
  for (int p = 0; p < plan.R; ++p) {
    // A is stored by (block row, block column); B (K x N stored N x K) by (N block, K block)
    const auto& sa = plan.side[0];
    const auto& sb = plan.side[1];
    a.a_src[p] = sa.slot[p] >= 0 ? LcmaOperand{sa.slot[p], 0, 0} : LcmaOperand{-1, sa.alias_r[p], sa.alias_c[p]};
    a.b_src[p] = sb.slot[p] >= 0 ? LcmaOperand{sb.slot[p], 0, 0} : LcmaOperand{-1, sb.alias_c[p], sb.alias_r[p]};
  }
  a.prod = prod;
  a.scratch = scratch;
  a.ldp = ldp;
  a.num_products = plan.R;
  a.err = h->err_dev;
  a.timeout_ns = h->timeout_ns;
  a.ep = ep;
  a.M = static_cast<int>(Mc);
  a.N = static_cast<int>(Nc);
  if (pair) {
    // Stream-K style split of the tail: when the last, partial wave of Groups
    // fits twice over, its Groups run as two halves on two pairs each.
    const int P = grid_cap(h) / 2;
    const int full_waves = a.num_groups / P, rem = a.num_groups - full_waves * P;
    const bool split = h->split && rem > 0 && 2 * rem <= P;
    a.split_first = split ? full_waves * P : a.num_groups;
    a.num_items = split ? full_waves * P + 2 * rem : a.num_groups;
    a.flags = split ? flags : nullptr;
    a.debug_drop = h->debug_drop;
    a.raw2d = raw2d ? 1 : 0;
    a.group_order = h->group_order;
    ll.grid = 2 * std::min(a.num_items, P);
    if (!hier) {
      // quadrant q of C: rows [qr * mb, qr * mb + mb) and columns [qc * nb, qc * nb + nb),
      // clipped to C; a map's base must sit on a 16-byte boundary and its row pitch be a
      // multiple of 16 bytes, else the kernel stores from registers
      const bool tma_ok = reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 8 == 0 && nb % 8 == 0;
      a.c_tma = 0;
      if (tma_ok) {
        a.c_tma = 1;
        for (int q = 0; q < 4; ++q) {
          const int64_t qr = q >> 1, qc = q & 1;
          const int64_t rows = std::min<int64_t>(mb, Mc - qr * mb), cols = std::min<int64_t>(nb, Nc - qc * nb);
          // whole 16-byte units only: the kernel stores a row's last < 8 columns itself
          const uint64_t cdims[2] = {static_cast<uint64_t>(std::max<int64_t>(cols & ~int64_t(7), 8)),
                                     static_cast<uint64_t>(std::max<int64_t>(rows, 1))};
          const uint64_t cstrides[1] = {static_cast<uint64_t>(ldc) * 2};
          const uint32_t cbox[2] = {32u, 32u};
          const void* base = static_cast<const uint16_t*>(C) + qr * mb * ldc + qc * nb;
          if (!encode_map(&ll.tmC.q[q], bf16, base, 2, cdims, cstrides, cbox, CU_TENSOR_MAP_SWIZZLE_64B))
            return LCGEMM_ERR_CUDA;
        }
      }
      if (launch_lcma_pair(ll, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
      return LCGEMM_OK;
    }
    if constexpr (L == 2) {
      // two levels: outer product po runs the one-level kernel on the inner products
      // p = 7 * po + pi of the two-level tables; its four inner quadrants go to the
      // outer targets (stream order, and each launch's wait for the one before it,
      // keep the outer slots consistent)
      LcmaOperand as[49], bs[49];
      for (int p = 0; p < plan.R; ++p) {
        as[p] = a.a_src[p];
        bs[p] = a.b_src[p];
      }
      a.outer = 1;
      a.oslot = oslot;
      a.mbp = static_cast<int>(mbp);
      a.nbp = static_cast<int>(nbp);
      for (int step = 0; step < 7; ++step) {
        const OuterStep& os = kOuterProgram[step];
        for (int pi = 0; pi < 7; ++pi) {
          a.a_src[pi] = as[7 * os.product + pi];
          a.b_src[pi] = bs[7 * os.product + pi];
        }
        a.otgt[0] = os.t[0];
        a.otgt[1] = os.t[1];
        a.flags = split ? flags + step * grid_cap(h) : nullptr;
        if (launch_lcma_pair(ll, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
      }
      return LCGEMM_OK;
    }
    return LCGEMM_OK;   // (one level: hier is false and the run ended above)
  }
  if (fused) {
    ll.grid = std::min(a.num_groups, grid_cap(h));
    if (launch_lcma_fused(ll, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
    return LCGEMM_OK;
  }
  ll.grid = std::min(a.num_groups * plan.R, grid_cap(h));
  if (launch_lcma_products(ll, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
  CombineHArgs ch{prod, ldp, static_cast<uint16_t*>(C), ldc, static_cast<int>(mb), static_cast<int>(nb), ep,
                  static_cast<int>(Mc), static_cast<int>(Nc)};
  // (no programmatic dependency here: measured slower for two levels, whose recombination
  // blocks would wait on SMs the products still use)
  if (launch_combine_h(ch, L, bf16, h->num_sms, st, false) != cudaSuccess) return LCGEMM_ERR_CUDA;
  return LCGEMM_OK;
}

}  // namespace

// Strassen on any shape: dimensions that the block split cannot divide (M by
// 2^levels, K by 8 * 2^levels) -- and N unless its blocks start on 16-byte
// boundaries (N by 8 * 2^levels), which keeps C's quadrant stores vectorised --
// run on zero-padded copies of the operand(s) concerned.  The products of the
// padding are zero and the kernels store only C's M x N elements, so C is exact
// up to the same rounding as on a divisible shape.
int run_strassen(lcgemm_ctx* h, int levels, bool fused, int64_t M, int64_t N, int64_t K, const void* A,
                 int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, bool bf16, const Epilogue& ep,
                 cudaStream_t st) {
  if (levels != 1 && levels != 2) return LCGEMM_ERR_UNSUPPORTED;
  const int64_t G = int64_t(1) << levels;
  const int64_t Mp = round_up(M, G), Np = round_up(N, 8 * G), Kp = round_up(K, 8 * G);
  const bool pad_a = Mp != M || Kp != K, pad_b = Np != N || Kp != K;
  const void* Ap = A;
  const void* Bp = B;
  int64_t ldap = lda, ldbp = ldb;
  if (pad_a || pad_b) {
    const int64_t a_bytes = pad_a ? round_up(Mp * Kp * 2, 256) : 0, b_bytes = pad_b ? round_up(Np * Kp * 2, 256) : 0;
    const size_t need = static_cast<size_t>(a_bytes + b_bytes);
    if (need > h->pad_bytes) {
      if (capturing(st)) return LCGEMM_ERR_CAPTURE;
      if (h->pad) {
        cudaStreamSynchronize(st);
        cudaFree(h->pad);
        h->pad = nullptr;
        h->pad_bytes = 0;
      }
      if (cudaMalloc(&h->pad, need) != cudaSuccess) {
        h->pad = nullptr;
        cudaGetLastError();
        return LCGEMM_ERR_NOMEM;
      }
      h->pad_bytes = need;
    }
    char* pa = static_cast<char*>(h->pad);
    char* pb = pa + a_bytes;
    PadArgs pad{};
    if (pad_a) {
      pad.side[0] = PadSide{static_cast<const uint16_t*>(A), lda, M, K, reinterpret_cast<uint16_t*>(pa), Mp, Kp};
      pad.vecs[0] = Mp * Kp / 8;
      Ap = pa;
      ldap = Kp;
    }
    if (pad_b) {
      pad.side[1] = PadSide{static_cast<const uint16_t*>(B), ldb, N, K, reinterpret_cast<uint16_t*>(pb), Np, Kp};
      pad.vecs[1] = Np * Kp / 8;
      Bp = pb;
      ldbp = Kp;
    }
    if (launch_pad_copy(pad, h->num_sms, st) != cudaSuccess) return LCGEMM_ERR_CUDA;
  }
  if (levels == 1) return run_levels<1>(h, fused, Mp, Np, Kp, Ap, ldap, Bp, ldbp, C, ldc, bf16, ep, st, M, N);
  return run_levels<2>(h, fused, Mp, Np, Kp, Ap, ldap, Bp, ldbp, C, ldc, bf16, ep, st, M, N);
}

}  // namespace lcg
