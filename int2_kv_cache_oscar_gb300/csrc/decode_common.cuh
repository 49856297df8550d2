// Work decomposition shared by the split-K decode kernels and the combine
// kernel (split-K flash decoding, the structure of the pages' BF16
// FlashDecoding-v2 comparator, ai-papers.net summary section "実験結果").
//
// The units of all (sequence, KV head) rows are laid end to end, T in total.
// Persistent CTA i of N takes units [floor(i T / N), floor((i+1) T / N)): every
// CTA gets the same amount of work whatever the length mix.  The part of a
// row inside one CTA is a "segment"; each segment yields one partial softmax
// state (m, l, o) per query head.  With rho = the rank of a non-empty row,
// CTA i writes the partial of row rho to slot i + rho: slots are distinct, and
// the partials of one row are contiguous, [first_cta(row) + rho,
// last_cta(row) + rho].
#pragma once

#include "common.cuh"
#include "launch.h"

namespace oscar {

__device__ __forceinline__ int64_t cta_first_unit(int64_t i, int64_t T, int64_t N) { return (i * T) / N; }

// Largest CTA index whose range contains unit u.
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t T, int64_t N) {
  return ((u + 1) * N - 1) / T;
}

__device__ __forceinline__ int units_of_len(int len, int bf16_mode) {
  return bf16_mode ? (len + 63) / 64 : len / kGroup;
}

// Locate unit u: sequence b (the largest with ubase <= u; it is never empty),
// KV head j and unit index g within the row.
template <int MAXS>
__device__ __forceinline__ void locate_unit(const DecodeParams<MAXS>& p, int64_t u, int& b, int& j, int& g,
                                            int& ng) {
  int lo = 0, hi = p.h.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seq[mid].ubase <= u) lo = mid; else hi = mid - 1;
  }
  b = lo;
  ng = units_of_len(p.seq[b].len, p.h.bf16_mode);
  const int64_t off = u - p.seq[b].ubase;
  j = (int)(off / ng);
  g = (int)(off - (int64_t)j * ng);
}

// ------------------------------------------------ decode device helpers

// Floats per probability row: 128 tokens plus 16 of padding (see pb_col).
constexpr int kPbStride = kGroup + 16;

// Column of token (or channel) t in probability row `row` (a query head):
// rows 2 and 3 swap 8-column blocks.  With the 144-float row stride, the
// score stores (lane (g, tig): row tig, column 16 mt + g) and the P.V
// factor loads (float2; lane (g, tig): row g / 2, column 16 k + 2 tig +
// 8 (g & 1)) are both free of bank conflicts.
__device__ __forceinline__ int pb_col(int row, int t) { return t ^ (8 * ((row >> 1) & 1)); }

__device__ __forceinline__ float pow2f(int e) {
  e = max(-126, min(127, e));
  return __uint_as_float((uint32_t)(127 + e) << 23);
}

// 2^F with max|x| * 2^F <= 2^15 for |x| <= bound (F = 0 when bound == 0).
__device__ __forceinline__ int range_exponent(float bound) {
  if (!(bound > 0.0f)) return 0;
  int e;
  frexpf(bound, &e);  // bound <= 2^e
  return 15 - e;
}

// A fragment of k-step kk (= ks & 3) from the words of rows g and g+8.
template <int KK>
__device__ __forceinline__ void frag_a(uint32_t w0, uint32_t w1, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                       uint32_t& a3) {
  a0 = frag_extract<2 * KK>(w0);
  a1 = frag_extract<2 * KK>(w1);
  a2 = frag_extract<2 * KK + 1>(w0);
  a3 = frag_extract<2 * KK + 1>(w1);
}

__device__ __forceinline__ void frag_a_dyn(int kk, uint32_t w0, uint32_t w1, uint32_t& a0, uint32_t& a1,
                                           uint32_t& a2, uint32_t& a3) {
  switch (kk) {
    case 0: frag_a<0>(w0, w1, a0, a1, a2, a3); break;
    case 1: frag_a<1>(w0, w1, a0, a1, a2, a3); break;
    case 2: frag_a<2>(w0, w1, a0, a1, a2, a3); break;
    default: frag_a<3>(w0, w1, a0, a1, a2, a3); break;
  }
}

// Partner-lane split of a B-fragment column pair.  Lanes g = 2h (hi column of
// head h) and g = 2h + 1 (lo column) need the same fp32 values x for k-rows
// {2 tig, 2 tig + 1} (register b0) and {2 tig + 8, 2 tig + 9} (register b1).
// The hi lane computes the b0 pair, the lo lane the b1 pair; each splits its
// pair into hi + lo fp16 and they swap the half the other one needs.
__device__ __forceinline__ void split_exchange(float x0, float x1, bool lo_lane, uint32_t& b0, uint32_t& b1) {
  const uint32_t hi = pack_half2(x0, x1);
  const float2 r = __fadd2_rn(make_float2(x0, x1), make_float2(-half_lo_to_float(hi), -half_hi_to_float(hi)));
  const uint32_t lo = pack_half2(r.x, r.y);
  const uint32_t send = lo_lane ? hi : lo;
  const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 4);
  b0 = lo_lane ? recv : hi;
  b1 = lo_lane ? lo : recv;
}

// 2^x for softmax weights (x <= 0 or small): the hardware approximation,
// relative error ~2^-22, flushes results below 2^-126 to zero.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace oscar
