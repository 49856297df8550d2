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

}  // namespace oscar
