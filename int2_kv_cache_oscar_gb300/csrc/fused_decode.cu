// Fused INT2 decode attention over the packed OScaR cache (sm_103a): one
// launch per decode pass, split-K inside the grid, the log-sum-exp merge of a
// row done by the CTA that completes it.
//
// Score of a quantised token t for query q (OScaR abstract; ai-papers.net
// summary, section "OScaRの提案手法": keys are stored rotated by H_d and
// divided by their norm):
//   s_t = n_t * sum_c (H_d q)_c (code_tc s_c + z_c) * scale
//       = n_t * (sum_c code_tc (q_rot_c s_c) + sum_c q_rot_c z_c) * scale;
// of a window token (bf16 residual): s_t = q . k_t * scale.
// Output: o = sum_t p_t v_t / sum_t p_t, v_t = code^V_tc s^V_t,gr(c) + z^V_t,gr(c)
// for quantised tokens and the bf16 row for window tokens.
//
// Work.  A (sequence, KV head) row is a list of units: its 128-token groups,
// then its bf16 window in pieces of 16 tokens.  The units of all rows lie end
// to end; persistent CTA i of N (one per SM) takes units [i T / N, (i+1) T / N).
//
// CTA: 7 score warps, 7 value warps, 1 producer warp (each SM sub-partition
// runs one role).  Unit k of the CTA goes to pair k mod 7.
//   producer (one lane): copies each unit's key part (group: codes, scales,
//     zeros, norms; window piece: bf16 key rows) into a key ring and its value
//     part into a value ring with 1-D bulk copies, keys up to 7 units ahead.
//   score warp: the unit's scores for up to 4 query heads, on the tensor
//     cores for a group (mma.sync m16n8k16: 2-bit codes as fp16 subnormal A
//     operands, q_rot * s split into fp16 hi + lo B columns) and on the CUDA
//     cores for a window piece; the unit's maximum m_u and its probabilities
//     p = 2^(s - m_u) go to the pair's double-buffered hand-off.
//   value warp: keeps the running softmax state (m, l, o) of its units of the
//     row; P.V on the tensor cores for a group (codes^V as A, p * s^V hi + lo
//     as B), CUDA cores for a window piece.
// Row end in a CTA: the value warps merge their states into one partial
// record (o, m, l per query head).  The CTA whose record completes the row (a
// ticket per (slot, KV head) in the arena, zero between calls) merges the
// row's records, writes the output and zeroes the ticket.
#include <cstddef>

#include "decode_common.cuh"

namespace oscar {
namespace {

constexpr int kPairs = 7;            // 15 warps: at most 4 per SM sub-partition, 128 registers each
// Warp w runs on SM sub-partition w mod 4.  Score warps take sub-partitions
// 0 and 1 (warps 0, 1, 4, 5, 8, 9, 12), value warps 2 and 3 (2, 3, 6, 7, 10,
// 11, 14), the producer warp 13: each sub-partition's instruction cache then
// holds one role's code (with the roles mixed, instruction fetch misses were
// the largest stall).  Pair index of a score or value warp: 2 (w / 4) + w % 2.
constexpr int kProducerWarp = 13;
__device__ __forceinline__ bool is_score_warp(int w) { return (w & 2) == 0 && w != kProducerWarp; }
__device__ __forceinline__ int pair_of_warp(int w) { return 2 * (w >> 2) + (w & 1); }
constexpr int kFThreads = (2 * kPairs + 1) * 32;
constexpr int kValueThreads = kPairs * 32;
constexpr int kWinPiece = 16;          // window tokens per window unit
constexpr int kBarValue = 1;           // named barrier of the value warps
constexpr int kMaxCtas = 160;          // persistent CTAs at most (records per row in the merge)

// Ring geometry by metadata width.  The key part of a block is its first
// KB bytes (K codes, scale, zero, norm), the value part the rest.
template <bool M16>
struct FRing {
  static constexpr int kKBytes = Blk<M16>::kVCodes;
  static constexpr int kVBytes = Blk<M16>::kBytes - Blk<M16>::kVCodes;
  static constexpr int kKSlots = M16 ? 16 : 14;
  static constexpr int kVSlots = M16 ? 14 : 11;
  // value-part offsets of the value scales and zeros
  static constexpr int kVScale = Blk<M16>::kVScale - Blk<M16>::kVCodes;
  static constexpr int kVZero = Blk<M16>::kVZero - Blk<M16>::kVCodes;
};
static_assert(FRing<false>::kKBytes >= kWinPiece * kHeadDim * 2 && FRing<true>::kKBytes >= kWinPiece * kHeadDim * 2,
              "a window piece's key rows must fit a key slot");
static_assert(FRing<false>::kVBytes >= kWinPiece * kHeadDim * 2 && FRing<true>::kVBytes >= kWinPiece * kHeadDim * 2,
              "a window piece's value rows must fit a value slot");

template <bool M16>
struct FSmem {
  static constexpr int KS = FRing<M16>::kKSlots;
  static constexpr int VS = FRing<M16>::kVSlots;
  alignas(128) uint8_t kslot[KS][FRing<M16>::kKBytes];
  alignas(128) uint8_t vslot[VS][FRing<M16>::kVBytes];
  // hand-off per pair and buffer: probabilities [head][pb_col(head, token)];
  // at a row end the value warp's output rows; at a row start the score
  // warp's rotated queries [head][channel]
  alignas(16) float hp[kPairs][2][kMaxGqa][kPbStride];
  float hm[kPairs][2][kMaxGqa];       // unit maximum (log2 units)
  float hl[kPairs][2][kMaxGqa];       // sum of the unit's p
  // value warp running outputs (head tig, channels 16 mt + g and + 8, times
  // 2^(Fv - 24)), [warp][mt][lane]: updated once per unit, so they hold no
  // registers during the tensor-core loop
  alignas(16) float2 oacc[kPairs][8][32];
  float rw[kMaxGqa][kMaxCtas];        // row merge: each record's m, then its weight
  float rl[kMaxGqa][kMaxCtas];        //            each record's l
  float rsum[kMaxGqa];                //            sum of weight * l
  float mm[kPairs][kMaxGqa];          // row end: value warp state m
  float ml[kPairs][kMaxGqa];          //          and l
  alignas(8) uint64_t kfull[KS];
  uint64_t kempty[KS];
  uint64_t vfull[VS];
  uint64_t vempty[VS];
  uint64_t hfull[kPairs][2];
  uint64_t hempty[kPairs][2];
  uint64_t qready;
  uint32_t kissued[KS];
  uint32_t vissued[VS];
  int vlast[kPairs];                  // row end: the hand-off buffer holding a value warp's rows, -1: none
  int abort_flag;
  int last_flag;
};
static_assert(sizeof(FSmem<false>) + 1024 <= 232448 && sizeof(FSmem<true>) + 1024 <= 232448,
              "one CTA per SM");
static_assert(offsetof(FSmem<false>, hp) % 16 == 0 && offsetof(FSmem<true>, hp) % 16 == 0, "alignment");
static_assert(offsetof(FSmem<false>, kfull) % 8 == 0 && offsetof(FSmem<true>, kfull) % 8 == 0, "alignment");
static_assert(FRing<false>::kKBytes % 128 == 0 && FRing<false>::kVBytes % 128 == 0 &&
                  FRing<true>::kKBytes % 128 == 0 && FRing<true>::kVBytes % 128 == 0,
              "slots stay 128-byte aligned");

}  // namespace

int fused_units_of_len(int len) {
  const int wlen = len % kGroup;
  return len / kGroup + (wlen + kWinPiece - 1) / kWinPiece;
}

namespace {

__device__ __forceinline__ int funits(int len) { return len / kGroup + (len % kGroup + kWinPiece - 1) / kWinPiece; }

// Locate unit u: sequence b, KV head j, unit index g within the row, the
// row's group count ng and unit count nu (>= 1: every sequence is non-empty).
template <int MAXS>
__device__ __forceinline__ void locate_funit(const DecodeParams<MAXS>& p, int64_t u, int& b, int& j, int& g,
                                             int& ng, int& nu) {
  int lo = 0, hi = p.h.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seq[mid].ubase <= u) lo = mid; else hi = mid - 1;
  }
  b = lo;
  const int len = p.seq[b].len;
  ng = len / kGroup;
  nu = funits(len);
  const int64_t off = u - p.seq[b].ubase;
  j = (int)(off / nu);
  g = (int)(off - (int64_t)j * nu);
}

// Bytes of 16-byte-aligned bf16 row data: window rows [r0, r1) of one part
// (key rows at +0, value rows at +32768 of a window), the newest row taken
// from `newest` (fused append) when it is not NULL.
__device__ __forceinline__ uint32_t issue_window_rows(uint8_t* dst, const uint8_t* win_part, int r0, int r1,
                                                      const uint16_t* newest, uint64_t* bar) {
  const int rows = r1 - r0;
  const uint32_t bytes = (uint32_t)rows * kHeadDim * 2;
  mbar_arrive_expect_tx(bar, bytes);
  const int from_arena = newest ? rows - 1 : rows;
  if (from_arena > 0) bulk_g2s(dst, win_part + (int64_t)r0 * kHeadDim * 2, (uint32_t)from_arena * kHeadDim * 2, bar);
  if (newest) bulk_g2s(dst + (int64_t)(rows - 1) * kHeadDim * 2, newest, kHeadDim * 2, bar);
  return bytes;
}

template <int MAXS, bool M16>
__global__ void __launch_bounds__(kFThreads, 1)
    fused_decode_kernel(const __grid_constant__ DecodeParams<MAXS> p, uint8_t* __restrict__ arena) {
  using R = FRing<M16>;
  using MR = Meta<M16>;
  using SM = FSmem<M16>;
  constexpr int KS = SM::KS;
  constexpr int VS = SM::VS;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SM& S = *reinterpret_cast<SM*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t T = p.h.n_units;
  const int64_t N = p.h.n_ctas;
  const int64_t cta = blockIdx.x;
  const int64_t u0 = cta_first_unit(cta, T, N);
  const int64_t u1 = cta_first_unit(cta + 1, T, N);
  const int hkv = p.h.hkv;
  const int gqa = p.h.gqa;
  const uint8_t* blocks = arena + p.h.blocks_off;
  uint32_t* const err = p.h.err_word;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(&S.kfull[s], 1);
      mbar_init(&S.kempty[s], 1);
      S.kissued[s] = 0;
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&S.vfull[s], 1);
      mbar_init(&S.vempty[s], 1);
      S.vissued[s] = 0;
    }
    for (int i = 0; i < kPairs; ++i)
      for (int b = 0; b < 2; ++b) {
        mbar_init(&S.hfull[i][b], 1);
        mbar_init(&S.hempty[i][b], 1);
      }
    mbar_init(&S.qready, 2 * kPairs);
    S.abort_flag = 0;
    S.last_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Lane i issues the copy of unit k + i when its ring slot is free: each
    // pass tests the slots of the next units without blocking, and the lanes
    // of the leading run of free slots issue their copies together.  Keys run
    // at most kPairs units ahead of values.
    const int U = (int)(u1 - u0);
    int kK = 0, kV = 0;            // units whose key / value part is issued
    uint32_t idle = 0;
    {
      bool q_ok = true;
      if (lane == 0) q_ok = mbar_wait_bounded(&S.qready, 0, &S.abort_flag, err);
      if (!__shfl_sync(0xffffffffu, q_ok, 0)) goto drain;
    }
    while (kK < U || kV < U) {
      if (S.abort_flag) goto drain;
      // ---- key parts
      const int limK = min(min(U - kK, kV + kPairs - kK), 32);
      int k = kK + lane;
      bool ready = false;
      if (lane < limK) {
        const uint32_t use = (uint32_t)(k / KS);
        ready = use == 0 || mbar_test_wait(&S.kempty[k % KS], (use - 1) & 1);
      }
      uint32_t bal = __ballot_sync(0xffffffffu, ready);
      const int nK = bal == 0xffffffffu ? 32 : __ffs(~bal) - 1;
      if (lane < nK) {
        const int s = k % KS;
        int b, j, g, ng, nu;
        locate_funit(p, u0 + k, b, j, g, ng, nu);
        const int64_t sh = (int64_t)p.seq[b].slot * hkv + j;
        if (g < ng) {
          mbar_arrive_expect_tx(&S.kfull[s], R::kKBytes);
          bulk_g2s(S.kslot[s], blocks + (sh * p.h.max_groups + g) * (int64_t)Blk<M16>::kBytes, R::kKBytes,
                   &S.kfull[s]);
        } else {
          const int wlen = p.seq[b].len % kGroup;
          const int r0 = (g - ng) * kWinPiece, r1 = min(r0 + kWinPiece, wlen);
          const uint16_t* nw = (p.h.k_new && r1 == wlen) ? p.h.k_new + ((int64_t)b * hkv + j) * kHeadDim : nullptr;
          issue_window_rows(S.kslot[s], arena + p.h.windows_off + sh * kWindowBytes, r0, r1, nw, &S.kfull[s]);
        }
        reinterpret_cast<volatile uint32_t*>(S.kissued)[s] = (uint32_t)(k / KS) + 1;
      }
      kK += nK;
      // ---- value parts
      const int limV = min(U - kV, 32);
      k = kV + lane;
      ready = false;
      if (lane < limV) {
        const uint32_t use = (uint32_t)(k / VS);
        ready = use == 0 || mbar_test_wait(&S.vempty[k % VS], (use - 1) & 1);
      }
      bal = __ballot_sync(0xffffffffu, ready);
      const int nV = bal == 0xffffffffu ? 32 : __ffs(~bal) - 1;
      if (lane < nV) {
        const int s = k % VS;
        int b, j, g, ng, nu;
        locate_funit(p, u0 + k, b, j, g, ng, nu);
        const int64_t sh = (int64_t)p.seq[b].slot * hkv + j;
        if (g < ng) {
          mbar_arrive_expect_tx(&S.vfull[s], R::kVBytes);
          bulk_g2s(S.vslot[s], blocks + (sh * p.h.max_groups + g) * (int64_t)Blk<M16>::kBytes + R::kKBytes,
                   R::kVBytes, &S.vfull[s]);
        } else {
          const int wlen = p.seq[b].len % kGroup;
          const int r0 = (g - ng) * kWinPiece, r1 = min(r0 + kWinPiece, wlen);
          const uint16_t* nw = (p.h.v_new && r1 == wlen) ? p.h.v_new + ((int64_t)b * hkv + j) * kHeadDim : nullptr;
          issue_window_rows(S.vslot[s], arena + p.h.windows_off + sh * kWindowBytes + kGroup * kHeadDim * 2, r0,
                            r1, nw, &S.vfull[s]);
        }
        reinterpret_cast<volatile uint32_t*>(S.vissued)[s] = (uint32_t)(k / VS) + 1;
      }
      kV += nV;
      if (nK + nV == 0) {
        // nothing to issue: sleep a little (bounded), the consumers are behind
        if (++idle > kWaitTries * 8u) {
          if (lane == 0) {
            S.abort_flag = 1;
            if (err) atomicOr(err, kErrTimeout);
          }
          goto drain;
        }
        __nanosleep(128);
      } else {
        idle = 0;
      }
    }
  drain:
    if (lane == 0 && S.abort_flag) {
      // wait (bounded, once more) for the copies that may still be in flight
      for (int kk = kK > KS ? kK - KS : 0; kk < kK; ++kk) {
        const int s = kk % KS;
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(&S.kfull[s], (uint32_t)((kk / KS) & 1))) break;
      }
      for (int kk = kV > VS ? kV - VS : 0; kk < kV; ++kk) {
        const int s = kk % VS;
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(&S.vfull[s], (uint32_t)((kk / VS) & 1))) break;
      }
    }
    return;
  }

  const int g = lane >> 2;     // row group of the mma fragments
  const int tig = lane & 3;    // thread in group
  const int hb = g >> 1;       // head of this lane's B column
  const int half = g & 1;      // 0: hi column lane, 1: lo column lane
  const bool lo_lane = half != 0;
  const float scale_log2 = p.h.scale_log2;
  // lane-constant parts of the swizzled shared-memory columns (token bit 3 is
  // fixed for every access): probability rows (pb_col) and the float32 value
  // scale / zero rows (vmeta_row), each relative to its 16-token block
  const int pbs0 = g ^ (8 * ((tig >> 1) & 1));                      // row tig, token g
  const int pbs1 = (g + 8) ^ (8 * ((tig >> 1) & 1));                // row tig, token g + 8

  if (is_score_warp(warp)) {
    // ---------------------------------------------------------- score warps
    const int pi = pair_of_warp(warp);
    // the first row's query rows are requested before the producer's first
    // bulk copy (it waits on qready): requested after it they would queue
    // behind every CTA's ring fill
    uint2 qpre[kMaxGqa];
    {
      int b, j, gg, ng, nu;
      locate_funit(p, u0 < u1 ? u0 : 0, b, j, gg, ng, nu);
#pragma unroll
      for (int h = 0; h < kMaxGqa; ++h)
        qpre[h] = (u0 < u1 && h < gqa)
                      ? *reinterpret_cast<const uint2*>(
                            p.h.q + ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + h) * kHeadDim + 4 * lane)
                      : make_uint2(0u, 0u);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.qready);

    // per-row constants
    float2 q2[8];              // this lane's B-column query values x 2^(F - p), per k-step
    float kqs = 0.0f, inv2Fk_b = 1.0f;
    float zwk[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) zwk[kk] = pow2f(half ? frag_p(2 * kk + 1) : frag_p(2 * kk));
#pragma unroll
    for (int i = 0; i < 8; ++i) q2[i] = make_float2(0.0f, 0.0f);

    uint32_t n = 0;            // units of this pair so far
    int64_t seg_u = u0;
    bool first_seg = true;
    while (seg_u < u1) {
      int b, j, g0, ng, nu;
      locate_funit(p, seg_u, b, j, g0, ng, nu);
      const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * nu;
      const int64_t seg_end = row_end < u1 ? row_end : u1;
      const int64_t kfirst = seg_u - u0;
      bool setup = false;
      for (int64_t k = kfirst + ((pi - kfirst) % kPairs + kPairs) % kPairs; k < seg_end - u0; k += kPairs, ++n) {
        const int gi = g0 + (int)(k - kfirst);   // unit index within the row
        const int buf = n & 1;
        if (n >= 2 && !mbar_wait_bounded(&S.hempty[pi][buf], ((n >> 1) - 1) & 1, &S.abort_flag, err)) continue;
        float* ph = &S.hp[pi][buf][0][0];
        if (!setup && ng > 0) {
          // ---- row setup: rotate the queries (each head in full, channels
          // 4 lane .. 4 lane + 3 per lane), stage them in this hand-off
          // buffer, gather this lane's B-column values
          setup = true;
          float qmax[kMaxGqa];
#pragma unroll 1
          for (int h = 0; h < kMaxGqa; ++h) {
            const uint2 raw = first_seg ? qpre[h]
                              : (h < gqa ? *reinterpret_cast<const uint2*>(
                                              p.h.q + ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + h) *
                                                          kHeadDim + 4 * lane)
                                         : make_uint2(0u, 0u));
            float qv[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
            // channel c = 4 * lane + i: bits 0, 1 in registers, bits 2..6 across lanes
            const float a = qv[0] + qv[1], bq = qv[0] - qv[1], c = qv[2] + qv[3], d = qv[2] - qv[3];
            qv[0] = a + c;
            qv[2] = a - c;
            qv[1] = bq + d;
            qv[3] = bq - d;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const bool upper = (lane & o) != 0;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float other = __shfl_xor_sync(0xffffffffu, qv[i], o);
                qv[i] = upper ? other - qv[i] : qv[i] + other;
              }
            }
            const float inv_sqrt_d = 0.088388347648318440550f;   // 1/sqrt(128)
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[i] *= inv_sqrt_d;
            float mx = fmaxf(fmaxf(fabsf(qv[0]), fabsf(qv[1])), fmaxf(fabsf(qv[2]), fabsf(qv[3])));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            qmax[h] = mx;
            *reinterpret_cast<float4*>(ph + h * kPbStride + 4 * lane) = make_float4(qv[0], qv[1], qv[2], qv[3]);
          }
          __syncwarp();
          const float qm_b = hb == 0 ? qmax[0] : hb == 1 ? qmax[1] : hb == 2 ? qmax[2] : qmax[3];
          const float qm_s = tig == 0 ? qmax[0] : tig == 1 ? qmax[1] : tig == 2 ? qmax[2] : qmax[3];
          const int Fk_b = range_exponent(qm_b * (2.0f / 3.0f));     // B-column head hb
          const int Fk_s = range_exponent(qm_s * (2.0f / 3.0f));     // score head tig
          kqs = pow2f(24 - Fk_s) * scale_log2;
          inv2Fk_b = pow2f(-Fk_b);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int c = 16 * ks + 2 * tig + 8 * half;
            const int pp = half ? frag_p(2 * (ks & 3) + 1) : frag_p(2 * (ks & 3));
            const float f = pow2f(Fk_b - pp);
            const float2 v = *reinterpret_cast<const float2*>(ph + hb * kPbStride + c);
            q2[ks] = make_float2(v.x * f, v.y * f);
          }
          __syncwarp();
        }
        // ---- wait for the unit's key part
        const int s = (int)k % KS;
        const uint32_t use = (uint32_t)((int)k / KS);
        if (!wait_issued(&S.kissued[s], use, &S.abort_flag, err)) continue;
        if (!mbar_wait_bounded(&S.kfull[s], use & 1, &S.abort_flag, err)) continue;
        const uint8_t* blk = S.kslot[s];
        if (gi < ng) {
          // ---------------- group unit: B fragments and q_rot . z
          const uint8_t* ksc = blk + Blk<M16>::kKScale;
          const uint8_t* kze = blk + Blk<M16>::kKZero;
          const uint8_t* knm = blk + Blk<M16>::kKNorm;
          uint32_t bk[8][2];
          float2 qzc[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) qzc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int c = 16 * ks + 2 * tig + 8 * half;
            const float2 s2 = MR::two(ksc, c);
            const float2 z2 = MR::two(kze, c);
            const float2 x = __fmul2_rn(q2[ks], s2);
            split_exchange(x.x, x.y, lo_lane, bk[ks][0], bk[ks][1]);
            qzc[ks & 3] = __ffma2_rn(q2[ks], z2, qzc[ks & 3]);
          }
          float qz = 0.0f;
#pragma unroll
          for (int i = 0; i < 4; ++i) qz = fmaf(qzc[i].x + qzc[i].y, zwk[i], qz);
          qz += __shfl_xor_sync(0xffffffffu, qz, 1);
          qz += __shfl_xor_sync(0xffffffffu, qz, 2);
          qz += __shfl_xor_sync(0xffffffffu, qz, 4);
          qz *= inv2Fk_b;                                                          // q_rot[hb] . z
          const float qzs = __shfl_sync(0xffffffffu, qz, 8 * tig) * scale_log2;   // head tig, log2 units

          // ---- scores: S^T[token][head x {hi, lo}] = codes x B, 4 independent chains
          float2 sc[8];   // tokens 16 mt + g (.x) and + 8 (.y), head tig
          {
            const uint4* kc = reinterpret_cast<const uint4*>(blk + kOffKCodes);
            const float2 kq2 = make_float2(kqs, kqs), qz2 = make_float2(qzs, qzs);
#pragma unroll 1
            for (int mh = 0; mh < 2; ++mh) {
              uint4 w[4];
              float acc[4][4];
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                w[m] = kc[(4 * mh + m) * 32 + lane];
                acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.0f;
              }
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                  const uint32_t w0 = (ks < 4) ? w[m].x : w[m].z;
                  const uint32_t w1 = (ks < 4) ? w[m].y : w[m].w;
                  uint32_t a0, a1, a2, a3;
                  frag_a_dyn(ks & 3, w0, w1, a0, a1, a2, a3);
                  mma_f16_16816(acc[m], a0, a1, a2, a3, bk[ks][0], bk[ks][1]);
                }
              }
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const int mt = 4 * mh + m;
                const int t0 = 16 * mt + g;
                const float2 a = make_float2(acc[m][0] + acc[m][1], acc[m][2] + acc[m][3]);
                sc[mt] = __fmul2_rn(__ffma2_rn(a, kq2, qz2), make_float2(MR::one(knm, t0), MR::one(knm, t0 + 8)));
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.kempty[s]);     // the key part is no longer read

          // ---- the unit's maximum and probabilities (head tig)
          float gm = fmaxf(sc[0].x, sc[0].y);
#pragma unroll
          for (int i = 1; i < 8; ++i) gm = fmaxf(gm, fmaxf(sc[i].x, sc[i].y));
          gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
          gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
          gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
          const float2 neg_m = make_float2(-gm, -gm);
          float2 psum = make_float2(0.0f, 0.0f);
          float* pt = ph + tig * kPbStride;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const float2 d = __fadd2_rn(sc[mt], neg_m);
            const float2 e = make_float2(fast_exp2(d.x), fast_exp2(d.y));
            psum = __fadd2_rn(psum, e);
            pt[16 * mt + pbs0] = e.x;
            pt[16 * mt + pbs1] = e.y;
          }
          float l = psum.x + psum.y;
          l += __shfl_xor_sync(0xffffffffu, l, 4);
          l += __shfl_xor_sync(0xffffffffu, l, 8);
          l += __shfl_xor_sync(0xffffffffu, l, 16);
          if (g == 0) {
            S.hm[pi][buf][tig] = gm;
            S.hl[pi][buf][tig] = l;
          }
        } else {
          // ---------------- window piece: rows r0 .. r1 - 1 of the window, on the CUDA cores
          const int wlen = p.seq[b].len % kGroup;
          const int r0 = (gi - ng) * kWinPiece;
          const int rows = min(kWinPiece, wlen - r0);
          float qf[kMaxGqa][4];
#pragma unroll
          for (int h = 0; h < kMaxGqa; ++h) {
            const uint2 raw = h < gqa ? *reinterpret_cast<const uint2*>(
                                            p.h.q + ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + h) *
                                                        kHeadDim + 4 * lane)
                                      : make_uint2(0u, 0u);
            qf[h][0] = bf16_lo(raw.x);
            qf[h][1] = bf16_hi(raw.x);
            qf[h][2] = bf16_lo(raw.y);
            qf[h][3] = bf16_hi(raw.y);
          }
          // scores of tokens 4 qr + (lane >> 3) & 3, head (lane >> 1) & 3, for qr = 0..3
          float sq[4];
#pragma unroll 1
          for (int qr = 0; qr < 4; ++qr) {
            // partial dots of tokens 4 qr .. 4 qr + 3 x 4 heads over this lane's 4 channels
            float a[16];
#pragma unroll
            for (int tl = 0; tl < 4; ++tl) {
              const uint2 kr = *reinterpret_cast<const uint2*>(blk + (4 * qr + tl) * kHeadDim * 2 + 8 * lane);
              const float k0 = bf16_lo(kr.x), k1 = bf16_hi(kr.x), k2 = bf16_lo(kr.y), k3 = bf16_hi(kr.y);
#pragma unroll
              for (int h = 0; h < kMaxGqa; ++h)
                a[4 * tl + h] = fmaf(qf[h][0], k0, fmaf(qf[h][1], k1, fmaf(qf[h][2], k2, qf[h][3] * k3)));
            }
            // reduce-scatter over lane bits 4..1: lanes L and L ^ 1 end with entry (L >> 1) & 15
#pragma unroll
            for (int m = 16, cnt = 8; m >= 2; m >>= 1, cnt >>= 1) {
              const bool upper = (lane & m) != 0;
#pragma unroll
              for (int i = 0; i < cnt; ++i) {
                const float keep = upper ? a[i + cnt] : a[i];
                const float send = upper ? a[i] : a[i + cnt];
                a[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
              }
            }
            a[0] += __shfl_xor_sync(0xffffffffu, a[0], 1);
            const int t = 4 * qr + ((lane >> 3) & 3);
            sq[qr] = t < rows ? a[0] * scale_log2 : -INFINITY;
          }
          // rows were read: release the key slot (the fused step first stores the newest key row)
          if (p.h.k_new && r0 + rows == wlen && lane < 16) {
            const int64_t sh = (int64_t)p.seq[b].slot * hkv + j;
            uint8_t* dst = arena + p.h.windows_off + sh * kWindowBytes + (int64_t)(wlen - 1) * kHeadDim * 2;
            *reinterpret_cast<uint4*>(dst + 16 * lane) =
                *reinterpret_cast<const uint4*>(blk + (rows - 1) * kHeadDim * 2 + 16 * lane);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.kempty[s]);
          const int h = (lane >> 1) & 3;
          float gm = fmaxf(fmaxf(sq[0], sq[1]), fmaxf(sq[2], sq[3]));
          gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
          gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
          float e[4];
#pragma unroll
          for (int qr = 0; qr < 4; ++qr) e[qr] = fast_exp2(sq[qr] - gm);
          float l = (e[0] + e[1]) + (e[2] + e[3]);
          l += __shfl_xor_sync(0xffffffffu, l, 8);
          l += __shfl_xor_sync(0xffffffffu, l, 16);
          if ((lane & 1) == 0) {
            float* prow = ph + h * kPbStride;
#pragma unroll
            for (int qr = 0; qr < 4; ++qr) prow[pb_col(h, 4 * qr + ((lane >> 3) & 3))] = e[qr];
          }
          if (lane < 8 && (lane & 1) == 0) {
            S.hm[pi][buf][h] = gm;
            S.hl[pi][buf][h] = l;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.hfull[pi][buf]);
      }
      first_seg = false;
      seg_u = seg_end;
    }
    return;
  }

  // -------------------------------------------------------------- value warps
  const int pi = pair_of_warp(warp);
  const int tv = pi * 32 + lane;                 // 0 .. 223 over the value warps
  uint32_t vpre = 0u;
  if (u0 < u1) {
    int b, j, gg, ng, nu;
    locate_funit(p, u0, b, j, gg, ng, nu);
    vpre = reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[(int64_t)p.seq[b].slot * hkv + j];
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&S.qready);

  const int pbl = (2 * tig + 8 * half) ^ (8 * ((hb >> 1) & 1));     // row hb, tokens 2 tig + 8 half, + 1
  const int vsl0 = 16 * (2 * tig + 8 * half + half);                // bytes: token 2 tig + 8 half
  const int vsl1 = 16 * (2 * tig + 8 * half + 1 - half);            //        token 2 tig + 8 half + 1
  const int vzl0 = 16 * g, vzl1 = 16 * ((g + 8) ^ 1);               //        tokens g, g + 8

  uint32_t n = 0;
  int64_t seg_u = u0;
  bool first_seg = true;
  while (seg_u < u1) {
    int b, j, g0, ng, nu;
    locate_funit(p, seg_u, b, j, g0, ng, nu);
    const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * nu;
    const int64_t seg_end = row_end < u1 ? row_end : u1;
    const int64_t kfirst = seg_u - u0;
    const int64_t sh = (int64_t)p.seq[b].slot * hkv + j;

    // per-row constants: value factors carry 2^(Fv - p) so that the fp16
    // operands stay below 2^15; o_acc holds o * 2^(Fv - 24)
    const float vmax = __uint_as_float(first_seg ? vpre : reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[sh]);
    const int Fv = range_exponent(vmax);
    const float kv = pow2f(24 - Fv);
    const float inv_kv = pow2f(Fv - 24);
    float fsc[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) fsc[kk] = pow2f(Fv) * pow2f(-(half ? frag_p(2 * kk + 1) : frag_p(2 * kk)));

    float m_t = -INFINITY;     // running max of head tig (log2 units)
    float m_b = -INFINITY;     // of head hb (the B column's head)
    float l_t = 0.0f;          // running sum of p, head tig
    float2* oacc = &S.oacc[pi][0][lane];   // [mt * 32]: head tig, channels 16 mt + g (.x), + 8 (.y)
    float zacc[kVGroups];      // sum_t p_t z^V_t,gr over this lane's tokens
#pragma unroll
    for (int i = 0; i < 8; ++i) oacc[32 * i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < kVGroups; ++i) zacc[i] = 0.0f;
    int last_buf = -1;

    for (int64_t k = kfirst + ((pi - kfirst) % kPairs + kPairs) % kPairs; k < seg_end - u0; k += kPairs, ++n) {
      const int gi = g0 + (int)(k - kfirst);
      const int buf = n & 1;
      const bool my_last = k + kPairs >= seg_end - u0;
      if (!mbar_wait_bounded(&S.hfull[pi][buf], (n >> 1) & 1, &S.abort_flag, err)) continue;
      const int s = (int)k % VS;
      const uint32_t use = (uint32_t)((int)k / VS);
      if (!wait_issued(&S.vissued[s], use, &S.abort_flag, err)) continue;
      if (!mbar_wait_bounded(&S.vfull[s], use & 1, &S.abort_flag, err)) continue;
      const uint8_t* blk = S.vslot[s];
      const float* ph = &S.hp[pi][buf][0][0];
      const float mg_t = S.hm[pi][buf][tig], mg_b = S.hm[pi][buf][hb], lg_t = S.hl[pi][buf][tig];
      const float mn_t = fmaxf(m_t, mg_t);
      const float alpha = fast_exp2(m_t - mn_t);
      const float beta_t = fast_exp2(mg_t - mn_t);
      m_t = mn_t;
      const float mn_b = fmaxf(m_b, mg_b);
      const float beta_b = fast_exp2(mg_b - mn_b);
      m_b = mn_b;
      l_t = fmaf(l_t, alpha, beta_t * lg_t);
      const float2 al2 = make_float2(alpha, alpha);
      if (gi < ng) {
        // ---------------- group unit
        const uint8_t* vsc = blk + R::kVScale;
        const uint8_t* vze = blk + R::kVZero;
        const float* pt = ph + tig * kPbStride;
        {
          float zl[kVGroups] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int t0 = 16 * mt + g;
            const float p0 = pt[16 * mt + pbs0], p1 = pt[16 * mt + pbs1];
            float4 z0, z1;
            if constexpr (M16) {
              z0 = MR::v4(vze, t0);
              z1 = MR::v4(vze, t0 + 8);
            } else {
              z0 = *reinterpret_cast<const float4*>(vze + 256 * mt + vzl0);
              z1 = *reinterpret_cast<const float4*>(vze + 256 * mt + vzl1);
            }
            zl[0] = fmaf(p0, z0.x, fmaf(p1, z1.x, zl[0]));
            zl[1] = fmaf(p0, z0.y, fmaf(p1, z1.y, zl[1]));
            zl[2] = fmaf(p0, z0.z, fmaf(p1, z1.z, zl[2]));
            zl[3] = fmaf(p0, z0.w, fmaf(p1, z1.w, zl[3]));
          }
#pragma unroll
          for (int gr = 0; gr < kVGroups; ++gr) zacc[gr] = fmaf(zacc[gr], alpha, beta_t * zl[gr]);
        }
        // ---- P.V: O^T[channel][head x {hi, lo}] = codes^V^T x (p * s^V); each
        // k-step's factors are built once and feed all 8 channel m-tiles
        const float* pbh = ph + hb * kPbStride;
        float fb[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) fb[kk] = fsc[kk] * beta_b;
        float pacc[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) pacc[mt][0] = pacc[mt][1] = pacc[mt][2] = pacc[mt][3] = 0.0f;
#pragma unroll 1
        for (int jh = 0; jh < 2; ++jh) {
          uint2 vw[8];
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) vw[mt] = *reinterpret_cast<const uint2*>(blk + vword_off(mt, jh, lane));
#pragma unroll
          for (int kk2 = 0; kk2 < 4; ++kk2) {
            const int t = 16 * (4 * jh + kk2) + 2 * tig + 8 * half;   // this lane's two tokens
            const float2 pr = __fmul2_rn(*reinterpret_cast<const float2*>(pbh + 16 * (4 * jh + kk2) + pbl),
                                         make_float2(fb[kk2], fb[kk2]));
            float4 s0, s1;
            if constexpr (M16) {
              MR::v4x2(vsc, t, s0, s1);
            } else {
              s0 = *reinterpret_cast<const float4*>(vsc + 256 * (4 * jh + kk2) + vsl0);
              s1 = *reinterpret_cast<const float4*>(vsc + 256 * (4 * jh + kk2) + vsl1);
            }
#pragma unroll
            for (int gr = 0; gr < kVGroups; ++gr) {
              const float sa = gr == 0 ? s0.x : gr == 1 ? s0.y : gr == 2 ? s0.z : s0.w;
              const float sb = gr == 0 ? s1.x : gr == 1 ? s1.y : gr == 2 ? s1.z : s1.w;
              uint32_t b0, b1;
              split_exchange(pr.x * sa, pr.y * sb, lo_lane, b0, b1);
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const int mt = 2 * gr + h2;
                uint32_t a0, a1, a2, a3;
                frag_a_dyn(kk2, vw[mt].x, vw[mt].y, a0, a1, a2, a3);
                mma_f16_16816(pacc[mt], a0, a1, a2, a3, b0, b1);
              }
            }
          }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          oacc[32 * mt] = __ffma2_rn(oacc[32 * mt], al2, make_float2(pacc[mt][0] + pacc[mt][1], pacc[mt][2] + pacc[mt][3]));
      } else {
        // ---------------- window piece: o += p v on the CUDA cores (head tig)
        const int wlen = p.seq[b].len % kGroup;
        const int r0 = (gi - ng) * kWinPiece;
        const int rows = min(kWinPiece, wlen - r0);
        const float* pt = ph + tig * kPbStride;
        const float f = beta_t * inv_kv;
        float2 o_acc[8];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) o_acc[mt] = __fmul2_rn(oacc[32 * mt], al2);
        for (int t = 0; t < rows; ++t) {
          const float pv = pt[pb_col(tig, t)] * f;
          const uint16_t* vrow = reinterpret_cast<const uint16_t*>(blk + t * kHeadDim * 2);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const float v0 = __uint_as_float((uint32_t)vrow[16 * mt + g] << 16);
            const float v1 = __uint_as_float((uint32_t)vrow[16 * mt + g + 8] << 16);
            o_acc[mt].x = fmaf(pv, v0, o_acc[mt].x);
            o_acc[mt].y = fmaf(pv, v1, o_acc[mt].y);
          }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) oacc[32 * mt] = o_acc[mt];
#pragma unroll
        for (int gr = 0; gr < kVGroups; ++gr) zacc[gr] *= alpha;
        if (p.h.v_new && r0 + rows == wlen && lane < 16) {
          uint8_t* dst = arena + p.h.windows_off + sh * kWindowBytes + kGroup * kHeadDim * 2 +
                         (int64_t)(wlen - 1) * kHeadDim * 2;
          *reinterpret_cast<uint4*>(dst + 16 * lane) =
              *reinterpret_cast<const uint4*>(blk + (rows - 1) * kHeadDim * 2 + 16 * lane);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.vempty[s]);
        if (!my_last) mbar_arrive(&S.hempty[pi][buf]);   // the row's last buffer is released after the merge
      }
      if (my_last) last_buf = buf;
    }

    // ---- row end in this CTA: value-warp states -> one partial record
    {
      float zs[kVGroups];
#pragma unroll
      for (int gr = 0; gr < kVGroups; ++gr) {
        float z = zacc[gr];
        z += __shfl_xor_sync(0xffffffffu, z, 4);
        z += __shfl_xor_sync(0xffffffffu, z, 8);
        z += __shfl_xor_sync(0xffffffffu, z, 16);
        zs[gr] = z;
      }
      if (g == 0) {
        S.mm[pi][tig] = last_buf >= 0 ? m_t : -INFINITY;
        S.ml[pi][tig] = last_buf >= 0 ? l_t : 0.0f;
      }
      if (lane == 0) S.vlast[pi] = last_buf;
      if (last_buf >= 0) {
        float* orow = &S.hp[pi][last_buf][tig][0];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const float zg = zs[mt >> 1];
          const float2 o = oacc[32 * mt];
          orow[16 * mt + pbs0] = fmaf(o.x, kv, zg);
          orow[16 * mt + pbs1] = fmaf(o.y, kv, zg);
        }
      }
    }
    named_bar_sync(kBarValue, kValueThreads);
    const int64_t rho = (int64_t)hkv * p.seq[b].rank + j;
    const bool ok = !S.abort_flag;
    if (ok) {
      float* part = p.h.partials + (cta + rho) * (int64_t)gqa * kPartialFloats;
      for (int idx = tv; idx < gqa * kHeadDim; idx += kValueThreads) {
        const int h = idx >> 7;
        const int c = idx & (kHeadDim - 1);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kPairs; ++w) M = fmaxf(M, S.mm[w][h]);
        float o = 0.0f, l = 0.0f;
#pragma unroll
        for (int w = 0; w < kPairs; ++w) {
          const int lb = S.vlast[w];
          if (lb >= 0) {
            const float f = exp2f(S.mm[w][h] - M);
            o = fmaf(f, S.hp[w][lb][h][pb_col(h, c)], o);
            l = fmaf(f, S.ml[w][h], l);
          }
        }
        part[h * kPartialFloats + c] = o;
        if (c == 0) {
          part[h * kPartialFloats + 128] = M;
          part[h * kPartialFloats + 129] = l;
        }
      }
      __threadfence();
    }
    named_bar_sync(kBarValue, kValueThreads);
    if (lane == 0 && last_buf >= 0) mbar_arrive(&S.hempty[pi][last_buf]);
    // ---- ticket: the CTA completing the row's records merges them
    const int64_t U_first = p.seq[b].ubase + (int64_t)j * nu;
    const int64_t first = cta_of_unit(U_first, T, N);
    const int64_t count = cta_of_unit(U_first + nu - 1, T, N) - first + 1;
    if (tv == 0) {
      int last = 0;
      if (ok) {
        const uint32_t prev = atomicAdd(p.h.tickets + sh, 1u);
        last = prev == (uint32_t)(count - 1);
        if (last) {
          __threadfence();
          p.h.tickets[sh] = 0u;        // every record of this launch has arrived
        }
      }
      S.last_flag = last;
    }
    named_bar_sync(kBarValue, kValueThreads);
    if (S.last_flag) {
      // merge the row's records (contiguous slots first + rho ..): gather
      // every record's m and l, one warp per head forms the weights
      // 2^(m_i - M), then each thread sums 4 channels over the records with
      // 8 independent loads in flight
      const float* rec = p.h.partials + (first + rho) * (int64_t)gqa * kPartialFloats;
      const int nrec = (int)count;
      for (int idx = tv; idx < nrec * gqa; idx += kValueThreads) {
        const int i = idx / gqa, h = idx - i * gqa;
        const float* r = rec + ((int64_t)i * gqa + h) * kPartialFloats;
        S.rw[h][i] = __ldcg(r + 128);
        S.rl[h][i] = __ldcg(r + 129);
      }
      named_bar_sync(kBarValue, kValueThreads);
      if (pi < gqa) {
        const int h = pi;
        float M = -INFINITY;
        for (int i = lane; i < nrec; i += 32) M = fmaxf(M, S.rw[h][i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.0f;
        for (int i = lane; i < nrec; i += 32) {
          const float mi = S.rw[h][i];
          const float f = (mi == -INFINITY) ? 0.0f : exp2f(mi - M);
          S.rw[h][i] = f;
          L = fmaf(f, S.rl[h][i], L);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) S.rsum[h] = L;
      }
      named_bar_sync(kBarValue, kValueThreads);
      for (int qd = tv; qd < gqa * (kHeadDim / 4); qd += kValueThreads) {
        const int h = qd >> 5, c4 = (qd & 31) * 4;
        const float* r = rec + h * kPartialFloats + c4;
        const int64_t stride = (int64_t)gqa * kPartialFloats;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 8
        for (int i = 0; i < nrec; ++i) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(r + i * stride));
          const float f = S.rw[h][i];
          acc.x = fmaf(f, v.x, acc.x);
          acc.y = fmaf(f, v.y, acc.y);
          acc.z = fmaf(f, v.z, acc.z);
          acc.w = fmaf(f, v.w, acc.w);
        }
        const float inv = 1.0f / S.rsum[h];
        const int64_t oi = ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + h) * kHeadDim + c4;
        if (p.h.out_f32) {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.h.out) + oi) =
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
          const uint32_t lo = f32_to_bf16_bits(acc.x * inv) | (f32_to_bf16_bits(acc.y * inv) << 16);
          const uint32_t hi = f32_to_bf16_bits(acc.z * inv) | (f32_to_bf16_bits(acc.w * inv) << 16);
          *reinterpret_cast<uint2*>(p.h.out + oi) = make_uint2(lo, hi);
        }
      }
    }
    named_bar_sync(kBarValue, kValueThreads);
    first_seg = false;
    seg_u = seg_end;
  }
}

}  // namespace

template <int MAXS>
cudaError_t launch_fused_decode(const DecodeParams<MAXS>& p, uint8_t* arena, bool meta16, cudaStream_t stream,
                                cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (p.h.n_units <= 0) return cudaSuccess;
  static bool attr_done[2][64] = {};
  cudaError_t e;
  if (ev_start) cudaEventRecord(ev_start, stream);
  if (meta16) {
    const int smem = (int)sizeof(FSmem<true>);
    e = ensure_smem_attr(fused_decode_kernel<MAXS, true>, smem, attr_done[1]);
    if (e != cudaSuccess) return e;
    fused_decode_kernel<MAXS, true><<<p.h.n_ctas, kFThreads, smem, stream>>>(p, arena);
  } else {
    const int smem = (int)sizeof(FSmem<false>);
    e = ensure_smem_attr(fused_decode_kernel<MAXS, false>, smem, attr_done[0]);
    if (e != cudaSuccess) return e;
    fused_decode_kernel<MAXS, false><<<p.h.n_ctas, kFThreads, smem, stream>>>(p, arena);
  }
  e = cudaGetLastError();
  if (ev_stop) cudaEventRecord(ev_stop, stream);
  return e;
}

template cudaError_t launch_fused_decode<kDecodeSeqsSmall>(const DecodeParams<kDecodeSeqsSmall>&, uint8_t*, bool,
                                                           cudaStream_t, cudaEvent_t, cudaEvent_t);
template cudaError_t launch_fused_decode<kDecodeSeqsLarge>(const DecodeParams<kDecodeSeqsLarge>&, uint8_t*, bool,
                                                           cudaStream_t, cudaEvent_t, cudaEvent_t);

}  // namespace oscar
