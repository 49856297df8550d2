// Chunked-prefill attention over the packed OScaR cache (sm_103a): the
// queries of a new chunk attend to every token already in the cache (its
// quantised groups and its bf16 window; no mask, the cache precedes the
// chunk).  Each output row also gets its log-sum-exp, so that the chunk's own
// causal attention can be merged in.  Scores and outputs follow the decode
// path (OScaR abstract; ai-papers.net "OScaRの提案手法"): s_t = n_t (H_d q) .
// (code_t s + z) * scale for quantised tokens, q . k_t * scale for window
// tokens, o = softmax(s) . v_hat.
//
// With many queries the contraction is a matrix product, so the rows go on
// the mma M dimension (FlashAttention-2 style; the decode kernel instead puts
// the 4 heads of one query on N):
//   * a CTA takes 128 (query, head) rows of one KV head (8 warps x 16 rows,
//     two per SM sub-partition) and streams every group block of that head
//     through a shared-memory ring of 1-D bulk copies; every warp reads every
//     stage, and the last warp to release a stage issues its refill (no
//     producer warp: 8 warps keep 255 registers each);
//   * a group is taken in two 64-token halves, one online-softmax step each
//     (32 score registers per lane);
//   * scores, m16n8k16 f16: A = the rows' rotated queries times the group's
//     key scales, fp16 hi + lo (~22 bits), pre-scaled by 2^(F_row - p); B =
//     the packed key codes: a fragment-order word of token row t is exactly
//     the B fragment of the 8-token tile holding t (one AND per register,
//     the code a subnormal fp16 code * 2^(p - 24));
//   * P.V: the score accumulators are the A operand (the C layout of one
//     16-token pair of tiles is the A layout of one k-step), times the value
//     scales of each 32-channel group, fp16 hi + lo; B = the packed value
//     codes, whose words are the B fragments of 8-channel tiles;
//   * online softmax in the log2 domain per row; value zeros and the key
//     zero term on the CUDA cores;
//   * the window last, on bf16 mma (q and k are exact bf16; P as bf16 hi + lo);
//   * with a workspace, grid.z splits the history's groups into parts (the
//     last part also takes the window) so that the CTAs fill whole waves of
//     SMs; each part writes per-row records (o unnormalised, m, l) that
//     prefill_merge_kernel combines.
#include <cstddef>

#include "common.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int kPfConsumers = 8;
constexpr int kPfThreads = kPfConsumers * 32;     // no producer warp: the last reader refills a stage
constexpr int kPfRows = 16 * kPfConsumers;   // (query, head) rows per CTA
constexpr int kPfStages = 6;
constexpr int kQrStride = 136;               // floats per staged rotated query row (16-byte rows, spread banks)
constexpr int kQbStride = 68;                // bf16 pairs per staged raw query row

struct PfSmem {
  alignas(128) uint8_t stage[kPfStages][kBlockBytes];   // group blocks; the window rows at the end
  alignas(16) float qr[kPfRows][kQrStride];              // rotated query rows times 2^(F_row - p(c))
  alignas(16) uint32_t qb[kPfRows][kQbStride];           // raw query rows, bf16 pairs
  float fexp[kPfRows];                                   // 2^(24 - F_row)
  alignas(8) uint64_t full[kPfStages];
  uint64_t wbar;
  uint32_t released[kPfStages];   // warps done with a stage, summed over its uses
  uint32_t nissued[kPfStages];    // copies issued into a stage
  int abort_flag;
};
static_assert(offsetof(PfSmem, qr) % 16 == 0 && offsetof(PfSmem, qb) % 16 == 0, "alignment");
static_assert(offsetof(PfSmem, full) % 8 == 0, "mbarriers must be 8-byte aligned");
static_assert(kPfStages * kBlockBytes >= 2 * kGroup * kHeadDim * 2, "the window fits in the ring");

__device__ __forceinline__ float pf_pow2(int e) {
  e = max(-126, min(127, e));
  return __uint_as_float((uint32_t)(127 + e) << 23);
}

// 2^F with max|x| * 2^F <= 2^15 for |x| <= bound (F = 0 when bound == 0).
__device__ __forceinline__ int pf_range_exponent(float bound) {
  if (!(bound > 0.0f)) return 0;
  int e;
  frexpf(bound, &e);
  return 15 - e;
}

__device__ __forceinline__ float pf_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp16 hi + lo of a pair (x0 in the low half).
__device__ __forceinline__ void split_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_half2(x0, x1);
  lo = pack_half2(x0 - half_lo_to_float(hi), x1 - half_hi_to_float(hi));
}

// bf16 hi + lo of a pair (round to nearest even; the remainder is exact).
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const uint32_t h0 = f32_to_bf16_bits(x0), h1 = f32_to_bf16_bits(x1);
  hi = h0 | (h1 << 16);
  const uint32_t l0 = f32_to_bf16_bits(x0 - __uint_as_float(h0 << 16));
  const uint32_t l1 = f32_to_bf16_bits(x1 - __uint_as_float(h1 << 16));
  lo = l0 | (l1 << 16);
}

template <int KK>
__device__ __forceinline__ void pf_b(uint32_t w, uint32_t& b0, uint32_t& b1) {
  b0 = frag_extract<2 * KK>(w);
  b1 = frag_extract<2 * KK + 1>(w);
}

__device__ __forceinline__ void pf_b_dyn(int kk, uint32_t w, uint32_t& b0, uint32_t& b1) {
  switch (kk) {
    case 0: pf_b<0>(w, b0, b1); break;
    case 1: pf_b<1>(w, b0, b1); break;
    case 2: pf_b<2>(w, b0, b1); break;
    default: pf_b<3>(w, b0, b1); break;
  }
}

// Online-softmax step of the lane's two rows over new log2-domain scores
// sc[nt][0..1] (row g) and sc[nt][2..3] (row g + 8) of nt_used tiles: the
// scores become probabilities, the running maxima and sums are updated, and
// the factor that rescales the state accumulated so far is returned per row.
template <int NT>
__device__ __forceinline__ void pf_softmax(float (&sc)[NT][4], int nt_used, float (&m_run)[2], float (&l_run)[2],
                                           float (&alpha)[2]) {
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (nt < nt_used) {
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
  // rows whose every score so far is -inf keep a zero state (alpha 0, p 0)
  const float base0 = mn0 == -INFINITY ? 0.0f : mn0, base1 = mn1 == -INFINITY ? 0.0f : mn1;
  alpha[0] = pf_exp2(m_run[0] - base0);
  alpha[1] = pf_exp2(m_run[1] - base1);
  m_run[0] = mn0;
  m_run[1] = mn1;
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (nt < nt_used) {
      sc[nt][0] = pf_exp2(sc[nt][0] - base0);
      sc[nt][1] = pf_exp2(sc[nt][1] - base0);
      sc[nt][2] = pf_exp2(sc[nt][2] - base1);
      sc[nt][3] = pf_exp2(sc[nt][3] - base1);
      s0 += sc[nt][0] + sc[nt][1];
      s1 += sc[nt][2] + sc[nt][3];
    } else {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
    }
  }
  l_run[0] = fmaf(l_run[0], alpha[0], s0);
  l_run[1] = fmaf(l_run[1], alpha[1], s1);
}

template <bool M16>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_int2_kernel(const __grid_constant__ PrefillParams p, const uint8_t* __restrict__ arena) {
  using B = Blk<M16>;           // ring stages keep 13,824-byte slots; a block copy is B::kBytes
  using MR = Meta<M16>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PfSmem& S = *reinterpret_cast<PfSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.y;                 // KV head
  // this CTA's part of the history: groups [g_begin, g_end); the last part
  // also takes the window
  const int part = blockIdx.z;
  const int g_begin = (int)(((int64_t)part * p.ng) / p.n_parts);
  const int g_end = (int)(((int64_t)(part + 1) * p.ng) / p.n_parts);
  const int ng = g_end - g_begin;
  const uint8_t* blocks = arena + p.blocks_off +
                          (((int64_t)p.slot * p.hkv + j) * p.max_groups + g_begin) * (int64_t)B::kBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&S.full[s], 1);
      S.released[s] = 0;
      S.nissued[s] = 0;
    }
    mbar_init(&S.wbar, 1);
    S.abort_flag = 0;
    fence_mbar_init();
    for (int k = 0; k < ng && k < kPfStages; ++k) {
      mbar_arrive_expect_tx(&S.full[k], B::kBytes);
      bulk_g2s(S.stage[k], blocks + (int64_t)k * B::kBytes, B::kBytes, &S.full[k]);
      S.nissued[k] = 1;
    }
  }
  __syncthreads();

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, tig = lane & 3;
  const int row0 = blockIdx.x * kPfRows + 16 * warp;     // this warp's first global row
  const int gqa = p.gqa;

  // ---- stage this warp's 16 rows: raw bf16 pairs, and rotated rows
  // (q_rot = H_d q) times 2^(F_row - p(c)), F_row from the row's range
  for (int r = 0; r < 16; ++r) {
    const int row = row0 + r;
    const int lr = 16 * warp + r;
    uint2 raw = make_uint2(0u, 0u);
    if (row < p.rows) {
      const int qi = row / gqa, h = j * gqa + row % gqa;
      raw = *reinterpret_cast<const uint2*>(p.q + ((int64_t)qi * p.hq + h) * kHeadDim + 4 * lane);
    }
    S.qb[lr][2 * lane] = raw.x;
    S.qb[lr][2 * lane + 1] = raw.y;
    float qv[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    {
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
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[i] *= 0.088388347648318440550f;  // 1/sqrt(128)
    }
    float mx = fmaxf(fmaxf(fabsf(qv[0]), fabsf(qv[1])), fmaxf(fabsf(qv[2]), fabsf(qv[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int F = pf_range_exponent(mx * (2.0f / 3.0f));   // |q_rot * s| <= 2/3 max|q_rot|
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = 4 * lane + i;
      const int pp = frag_p(2 * ((c >> 4) & 3) + ((c >> 3) & 1));
      S.qr[lr][c] = qv[i] * pf_pow2(F - pp);
    }
    if (lane == 0) S.fexp[lr] = pf_pow2(24 - F);
  }
  __syncwarp();

  const int lr0 = 16 * warp + g, lr1 = lr0 + 8;          // this lane's rows (local)
  const float fe0 = S.fexp[lr0], fe1 = S.fexp[lr1];
  const float vmax = __uint_as_float(
      reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[(int64_t)p.slot * p.hkv + j]);
  const int Fv = pf_range_exponent(vmax);
  const float kv = pf_pow2(24 - Fv);
  float fsc[4][2];   // 2^(Fv - p) of the k-rows (tokens) 2 tig (+1) and 8 + 2 tig (+1) of k-step class kk
  float zw[4][2];    // 2^p of the key columns c0 / c1 of k-step class kk
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    fsc[kk][0] = pf_pow2(Fv - frag_p(2 * kk));
    fsc[kk][1] = pf_pow2(Fv - frag_p(2 * kk + 1));
    zw[kk][0] = pf_pow2(frag_p(2 * kk));
    zw[kk][1] = pf_pow2(frag_p(2 * kk + 1));
  }

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.0f, 0.0f};
  float oacc[16][4];      // rows g (0, 1) and g + 8 (2, 3), channels 8 nt + 2 tig + {0, 1}; x 2^(Fv - 24)
  float zacc[2][kVGroups];
#pragma unroll
  for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.0f;
#pragma unroll
  for (int i = 0; i < kVGroups; ++i) zacc[0][i] = zacc[1][i] = 0.0f;
  const float* q0row = S.qr[lr0];
  const float* q1row = S.qr[lr1];

  for (int k = 0; k < ng; ++k) {
    const int s = k % kPfStages;
    const uint32_t use = (uint32_t)(k / kPfStages);
    // every warp reads every use of a stage, and a refill waits for all of
    // them, so no warp can be two uses ahead: the parity test cannot alias
    if (!mbar_wait_bounded(&S.full[s], use & 1, &S.abort_flag, p.err_word)) break;
    const uint8_t* blk = S.stage[s];
    const uint8_t* ksc = blk + B::kKScale;
    const uint8_t* kze = blk + B::kKZero;
    const uint8_t* knm = blk + B::kKNorm;
    const uint8_t* vsc = blk + B::kVScale;
    const uint8_t* vze = blk + B::kVZero;
    const uint4* kc = reinterpret_cast<const uint4*>(blk + kOffKCodes);

    float qz0 = 0.0f, qz1 = 0.0f;   // q_rot . z of the lane's rows (times 2^F), from the first half
    float qzt0 = 0.0f, qzt1 = 0.0f;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // ---- scores of tokens 64 hh .. 64 hh + 63: sc[ntl] = tokens 64 hh + 8 ntl + 2 tig + {0, 1}
      float sc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.0f;
#pragma unroll
      for (int jh = 0; jh < 2; ++jh) {
        uint32_t kw[8];   // word (j = jh, r) of token m-tile 4 hh + mtl: tile ntl = 2 mtl + r
#pragma unroll
        for (int mtl = 0; mtl < 4; ++mtl) {
          const uint4 w4 = kc[(4 * hh + mtl) * 32 + lane];
          kw[2 * mtl] = jh ? w4.z : w4.x;
          kw[2 * mtl + 1] = jh ? w4.w : w4.y;
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ks = 4 * jh + kk;
          const int c0 = 16 * ks + 2 * tig, c1 = c0 + 8;
          const float2 x00 = *reinterpret_cast<const float2*>(q0row + c0);
          const float2 x01 = *reinterpret_cast<const float2*>(q0row + c1);
          const float2 x10 = *reinterpret_cast<const float2*>(q1row + c0);
          const float2 x11 = *reinterpret_cast<const float2*>(q1row + c1);
          const float2 s0 = MR::two(ksc, c0);
          const float2 s1 = MR::two(ksc, c1);
          if (hh == 0) {
            const float2 z0 = MR::two(kze, c0);
            const float2 z1 = MR::two(kze, c1);
            qz0 = fmaf(fmaf(x00.x, z0.x, x00.y * z0.y), zw[kk][0], qz0);
            qz0 = fmaf(fmaf(x01.x, z1.x, x01.y * z1.y), zw[kk][1], qz0);
            qz1 = fmaf(fmaf(x10.x, z0.x, x10.y * z0.y), zw[kk][0], qz1);
            qz1 = fmaf(fmaf(x11.x, z1.x, x11.y * z1.y), zw[kk][1], qz1);
          }
          uint32_t ah[4], al[4];
          split_f16(x00.x * s0.x, x00.y * s0.y, ah[0], al[0]);
          split_f16(x10.x * s0.x, x10.y * s0.y, ah[1], al[1]);
          split_f16(x01.x * s1.x, x01.y * s1.y, ah[2], al[2]);
          split_f16(x11.x * s1.x, x11.y * s1.y, ah[3], al[3]);
#pragma unroll
          for (int ntl = 0; ntl < 8; ++ntl) {
            uint32_t b0, b1;
            pf_b_dyn(kk, kw[ntl], b0, b1);
            mma_f16_16816(sc[ntl], ah[0], ah[1], ah[2], ah[3], b0, b1);
            mma_f16_16816(sc[ntl], al[0], al[1], al[2], al[3], b0, b1);
          }
        }
      }
      if (hh == 0) {
        qz0 += __shfl_xor_sync(0xffffffffu, qz0, 1);
        qz0 += __shfl_xor_sync(0xffffffffu, qz0, 2);
        qz1 += __shfl_xor_sync(0xffffffffu, qz1, 1);
        qz1 += __shfl_xor_sync(0xffffffffu, qz1, 2);
        // qr = q_rot 2^(F - p) and zw = 2^p: qz * 2^-F = q_rot . z; fexp = 2^(24 - F)
        qzt0 = qz0 * fe0 * (1.0f / 16777216.0f);
        qzt1 = qz1 * fe1 * (1.0f / 16777216.0f);
      }
#pragma unroll
      for (int ntl = 0; ntl < 8; ++ntl) {
        const float2 n2 = MR::two(knm, 64 * hh + 8 * ntl + 2 * tig);
        sc[ntl][0] = fmaf(sc[ntl][0], fe0, qzt0) * n2.x * p.scale_log2;
        sc[ntl][1] = fmaf(sc[ntl][1], fe0, qzt0) * n2.y * p.scale_log2;
        sc[ntl][2] = fmaf(sc[ntl][2], fe1, qzt1) * n2.x * p.scale_log2;
        sc[ntl][3] = fmaf(sc[ntl][3], fe1, qzt1) * n2.y * p.scale_log2;
      }

      // ---- online softmax, rescale the state
      float alpha[2];
      pf_softmax<8>(sc, 8, m_run, l_run, alpha);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        oacc[nt][0] *= alpha[0];
        oacc[nt][1] *= alpha[0];
        oacc[nt][2] *= alpha[1];
        oacc[nt][3] *= alpha[1];
      }
#pragma unroll
      for (int gv = 0; gv < kVGroups; ++gv) {
        zacc[0][gv] *= alpha[0];
        zacc[1][gv] *= alpha[1];
      }
      // value zeros: sum_t p_t z^V_t,gv over the lane's 16 tokens of this half
#pragma unroll
      for (int ntl = 0; ntl < 8; ++ntl) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 64 * hh + 8 * ntl + 2 * tig + e;
          // float32 zeros: token t is in row t ^ 1 when bit 3 (ntl & 1) is set
          const float4 z4 = M16 ? MR::v4(vze, t)
                                : *reinterpret_cast<const float4*>(vze + 16 * (64 * hh + 8 * ntl + 2 * tig +
                                                                              (e ^ (ntl & 1))));
          zacc[0][0] = fmaf(sc[ntl][e], z4.x, zacc[0][0]);
          zacc[0][1] = fmaf(sc[ntl][e], z4.y, zacc[0][1]);
          zacc[0][2] = fmaf(sc[ntl][e], z4.z, zacc[0][2]);
          zacc[0][3] = fmaf(sc[ntl][e], z4.w, zacc[0][3]);
          zacc[1][0] = fmaf(sc[ntl][2 + e], z4.x, zacc[1][0]);
          zacc[1][1] = fmaf(sc[ntl][2 + e], z4.y, zacc[1][1]);
          zacc[1][2] = fmaf(sc[ntl][2 + e], z4.z, zacc[1][2]);
          zacc[1][3] = fmaf(sc[ntl][2 + e], z4.w, zacc[1][3]);
        }
      }

      // ---- P.V over this half: k-steps ks = 4 hh + kk (score tiles 2 kk, 2 kk + 1)
      uint32_t vw[16];   // word (j = hh, r) of channel m-tile mt: channel tile nt = 2 mt + r
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint2 w2 = *reinterpret_cast<const uint2*>(blk + B::kVCodes + vword_off(mt, hh, lane));
        vw[2 * mt] = w2.x;
        vw[2 * mt + 1] = w2.y;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int t0 = 64 * hh + 16 * kk + 2 * tig, t1 = t0 + 8;
        float4 sa, sb, sc4, sd;
        if constexpr (M16) {
          MR::v4x2(vsc, t0, sa, sb);
          MR::v4x2(vsc, t1, sc4, sd);
        } else {   // float32 rows: t0, t0 + 1 in place (bit 3 clear); t1, t1 + 1 swapped (bit 3 set)
          sa = *reinterpret_cast<const float4*>(vsc + 16 * t0);
          sb = *reinterpret_cast<const float4*>(vsc + 16 * t0 + 16);
          sc4 = *reinterpret_cast<const float4*>(vsc + 16 * t1 + 16);
          sd = *reinterpret_cast<const float4*>(vsc + 16 * t1);
        }
        const float* p00 = sc[2 * kk];       // tokens t0, t0+1: rows g (0, 1), g + 8 (2, 3)
        const float* p01 = sc[2 * kk + 1];   // tokens t1, t1+1
        const float f0 = fsc[kk][0], f1 = fsc[kk][1];
#pragma unroll
        for (int gv = 0; gv < kVGroups; ++gv) {
          const float va = gv == 0 ? sa.x : gv == 1 ? sa.y : gv == 2 ? sa.z : sa.w;
          const float vb = gv == 0 ? sb.x : gv == 1 ? sb.y : gv == 2 ? sb.z : sb.w;
          const float vcc = gv == 0 ? sc4.x : gv == 1 ? sc4.y : gv == 2 ? sc4.z : sc4.w;
          const float vd = gv == 0 ? sd.x : gv == 1 ? sd.y : gv == 2 ? sd.z : sd.w;
          uint32_t ah[4], al[4];
          split_f16(p00[0] * va * f0, p00[1] * vb * f0, ah[0], al[0]);   // row g, tokens t0, t0+1
          split_f16(p00[2] * va * f0, p00[3] * vb * f0, ah[1], al[1]);   // row g + 8
          split_f16(p01[0] * vcc * f1, p01[1] * vd * f1, ah[2], al[2]);  // row g, tokens t1, t1+1
          split_f16(p01[2] * vcc * f1, p01[3] * vd * f1, ah[3], al[3]);  // row g + 8
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int nt = 4 * gv + q4;      // channels 8 nt .. 8 nt + 7
            uint32_t b0, b1;
            pf_b_dyn(kk, vw[nt], b0, b1);
            mma_f16_16816(oacc[nt], ah[0], ah[1], ah[2], ah[3], b0, b1);
            mma_f16_16816(oacc[nt], al[0], al[1], al[2], al[3], b0, b1);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();                                   // this warp's reads of the stage are done
      const uint32_t before = atomicAdd(&S.released[s], 1u);
      if (before == (use + 1) * kPfConsumers - 1 && k + kPfStages < ng) {
        __threadfence_block();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic reads before the async write
        mbar_arrive_expect_tx(&S.full[s], B::kBytes);
        bulk_g2s(S.stage[s], blocks + (int64_t)(k + kPfStages) * B::kBytes, B::kBytes, &S.full[s]);
        S.nissued[s] = use + 2;
      }
    }
  }
  // every warp leaves the group loop here, so all see the same abort state
  named_bar_sync(1, kPfConsumers * 32);
  if (S.abort_flag) {
    // a wait gave up: before the CTA exits, wait (bounded) for copies still in flight
    if (threadIdx.x == 0) {
      for (int s = 0; s < kPfStages; ++s) {
        const uint32_t n = *reinterpret_cast<volatile uint32_t*>(&S.nissued[s]);
        if (n == 0) continue;
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(&S.full[s], (n - 1) & 1)) break;
      }
    }
    return;
  }

  // ---- the window (bf16 rows after the last group), on bf16 tensor cores
  const int wlen = part == p.n_parts - 1 ? p.wlen : 0;
  if (wlen > 0) {   // every warp is done with the ring (barrier above)
    uint16_t* wk = reinterpret_cast<uint16_t*>(S.stage[0]);
    uint16_t* wv = wk + kGroup * kHeadDim;
    if (threadIdx.x == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint8_t* wsrc = arena + p.windows_off + ((int64_t)p.slot * p.hkv + j) * kWindowBytes;
      const uint32_t wbytes = (uint32_t)wlen * kHeadDim * 2;
      mbar_arrive_expect_tx(&S.wbar, 2 * wbytes);
      bulk_g2s(wk, wsrc, wbytes, &S.wbar);
      bulk_g2s(wv, wsrc + kGroup * kHeadDim * 2, wbytes, &S.wbar);
    }
    const int tpad = (wlen + 15) & ~15;   // rows up to the next 16 are zeroed (the k-step tail)
    for (int i = threadIdx.x; i < (tpad - wlen) * kHeadDim / 2; i += kPfConsumers * 32) {
      const int r = wlen + i / (kHeadDim / 2), c2 = i % (kHeadDim / 2);
      reinterpret_cast<uint32_t*>(wk + r * kHeadDim)[c2] = 0u;
      reinterpret_cast<uint32_t*>(wv + r * kHeadDim)[c2] = 0u;
    }
    const bool wok = mbar_wait_bounded(&S.wbar, 0, &S.abort_flag, p.err_word);
    named_bar_sync(1, kPfConsumers * 32);     // the zeroed tail rows are visible (every warp arrives)
    if (wok) {
      const int nt_used = (wlen + 7) >> 3;
      float sc[16][4];
#pragma unroll
      for (int i = 0; i < 16; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.0f;
      const uint32_t* qb0 = S.qb[lr0];
      const uint32_t* qb1 = S.qb[lr1];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t a0 = qb0[8 * ks + tig], a1 = qb1[8 * ks + tig];
        const uint32_t a2 = qb0[8 * ks + 4 + tig], a3 = qb1[8 * ks + 4 + tig];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          if (nt < nt_used) {
            const uint32_t* kr = reinterpret_cast<const uint32_t*>(wk + (8 * nt + g) * kHeadDim);
            mma_bf16_16816(sc[nt], a0, a1, a2, a3, kr[8 * ks + tig], kr[8 * ks + 4 + tig]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool in = 8 * nt + 2 * tig + e < wlen;
          sc[nt][e] = in ? sc[nt][e] * p.scale_log2 : -INFINITY;
          sc[nt][2 + e] = in ? sc[nt][2 + e] * p.scale_log2 : -INFINITY;
        }
      }
      float alpha[2];
      pf_softmax<16>(sc, nt_used, m_run, l_run, alpha);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        oacc[nt][0] *= alpha[0];
        oacc[nt][1] *= alpha[0];
        oacc[nt][2] *= alpha[1];
        oacc[nt][3] *= alpha[1];
      }
#pragma unroll
      for (int gv = 0; gv < kVGroups; ++gv) {
        zacc[0][gv] *= alpha[0];
        zacc[1][gv] *= alpha[1];
      }
      // P.V in the accumulators' units: P * 2^(Fv - 24) as bf16 hi + lo
      const float wsc = pf_pow2(Fv - 24);
      const int ks_used = (wlen + 15) >> 4;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (ks < ks_used) {
          const float* p00 = sc[2 * ks];
          const float* p01 = sc[2 * ks + 1];
          uint32_t ah[4], al[4];
          split_bf16(p00[0] * wsc, p00[1] * wsc, ah[0], al[0]);
          split_bf16(p00[2] * wsc, p00[3] * wsc, ah[1], al[1]);
          split_bf16(p01[0] * wsc, p01[1] * wsc, ah[2], al[2]);
          split_bf16(p01[2] * wsc, p01[3] * wsc, ah[3], al[3]);
          const int t0 = 16 * ks + 2 * tig, t1 = t0 + 8;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) {
            const int c = 8 * nt + g;
            const uint32_t b0 = (uint32_t)wv[t0 * kHeadDim + c] | ((uint32_t)wv[(t0 + 1) * kHeadDim + c] << 16);
            const uint32_t b1 = (uint32_t)wv[t1 * kHeadDim + c] | ((uint32_t)wv[(t1 + 1) * kHeadDim + c] << 16);
            mma_bf16_16816(oacc[nt], ah[0], ah[1], ah[2], ah[3], b0, b1);
            mma_bf16_16816(oacc[nt], al[0], al[1], al[2], al[3], b0, b1);
          }
        }
      }
    }
  }

  // ---- rows out: o = (kv * oacc + z) / l, lse = (m + log2 l) ln 2
  float l0 = l_run[0], l1 = l_run[1];
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  float zs[2][kVGroups];
#pragma unroll
  for (int gv = 0; gv < kVGroups; ++gv) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float z = zacc[rr][gv];
      z += __shfl_xor_sync(0xffffffffu, z, 1);
      z += __shfl_xor_sync(0xffffffffu, z, 2);
      zs[rr][gv] = z;
    }
  }
  if (p.n_parts > 1) {
    // partial record of each of the lane's rows: o unnormalised, m, l
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = row0 + g + 8 * rr;
      if (row >= p.rows) continue;
      float* rec = p.parts + (((int64_t)part * p.hkv + j) * p.rows + row) * kPrefillRecFloats;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const float z = zs[rr][nt >> 2];
        *reinterpret_cast<float2*>(rec + 8 * nt + 2 * tig) =
            make_float2(fmaf(oacc[nt][2 * rr], kv, z), fmaf(oacc[nt][2 * rr + 1], kv, z));
      }
      if (tig == 0) *reinterpret_cast<float2*>(rec + kHeadDim) = make_float2(m_run[rr], rr ? l1 : l0);
    }
    return;
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = row0 + g + 8 * rr;
    if (row >= p.rows) continue;
    const int qi = row / gqa, h = j * gqa + row % gqa;
    const float l = rr ? l1 : l0;
    const float inv = 1.0f / l;
    uint32_t* orow = reinterpret_cast<uint32_t*>(p.out + ((int64_t)qi * p.hq + h) * kHeadDim);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const float z = zs[rr][nt >> 2];
      const float o0 = fmaf(oacc[nt][2 * rr], kv, z) * inv;
      const float o1 = fmaf(oacc[nt][2 * rr + 1], kv, z) * inv;
      orow[4 * nt + tig] = f32_to_bf16_bits(o0) | (f32_to_bf16_bits(o1) << 16);
    }
    if (tig == 0 && p.lse != nullptr) p.lse[(int64_t)qi * p.hq + h] = (m_run[rr] + log2f(l)) * 0.69314718055994530942f;
  }
}

// Merge of the history parts: one warp per (KV head, row), 4 channels per
// lane.  m* = max m_i, l = sum 2^(m_i - m*) l_i, o = sum 2^(m_i - m*) o_i / l,
// lse = (m* + log2 l) ln 2.
constexpr int kPfMergeWarps = 8;

__global__ void __launch_bounds__(kPfMergeWarps * 32)
    prefill_merge_kernel(const __grid_constant__ PrefillParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * kPfMergeWarps + (threadIdx.x >> 5);   // KV head * rows + row
  if (gw >= (int64_t)p.hkv * p.rows) return;
  const int j = (int)(gw / p.rows), row = (int)(gw % p.rows);
  const int64_t stride = (int64_t)p.hkv * p.rows * kPrefillRecFloats;   // between parts
  const float* rec = p.parts + gw * kPrefillRecFloats;
  float M = -INFINITY;
  for (int i = 0; i < p.n_parts; ++i) M = fmaxf(M, rec[i * stride + kHeadDim]);
  float l = 0.0f;
  float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int i = 0; i < p.n_parts; ++i) {
    const float* r = rec + i * stride;
    const float mi = r[kHeadDim];
    const float w = mi == -INFINITY ? 0.0f : exp2f(mi - M);
    l = fmaf(w, r[kHeadDim + 1], l);
    const float4 v = *reinterpret_cast<const float4*>(r + 4 * lane);
    o.x = fmaf(w, v.x, o.x);
    o.y = fmaf(w, v.y, o.y);
    o.z = fmaf(w, v.z, o.z);
    o.w = fmaf(w, v.w, o.w);
  }
  const float inv = 1.0f / l;
  const int qi = row / p.gqa, h = j * p.gqa + row % p.gqa;
  uint2 packed;
  packed.x = f32_to_bf16_bits(o.x * inv) | (f32_to_bf16_bits(o.y * inv) << 16);
  packed.y = f32_to_bf16_bits(o.z * inv) | (f32_to_bf16_bits(o.w * inv) << 16);
  *reinterpret_cast<uint2*>(p.out + ((int64_t)qi * p.hq + h) * kHeadDim + 4 * lane) = packed;
  if (lane == 0 && p.lse != nullptr) p.lse[(int64_t)qi * p.hq + h] = (M + log2f(l)) * 0.69314718055994530942f;
}

}  // namespace

namespace {
template <bool M16>
cudaError_t launch_prefill_t(const PrefillParams& p, const uint8_t* arena, cudaStream_t stream) {
  static bool attr_done[64] = {};
  const int smem = (int)sizeof(PfSmem);
  cudaError_t e = ensure_smem_attr(prefill_int2_kernel<M16>, smem, attr_done);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.rows + kPfRows - 1) / kPfRows, p.hkv, p.n_parts);
  prefill_int2_kernel<M16><<<grid, kPfThreads, smem, stream>>>(p, arena);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.n_parts <= 1) return e;
  const int64_t warps = (int64_t)p.hkv * p.rows;
  prefill_merge_kernel<<<(unsigned)((warps + kPfMergeWarps - 1) / kPfMergeWarps), kPfMergeWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const uint8_t* arena, bool meta16, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  return meta16 ? launch_prefill_t<true>(p, arena, stream) : launch_prefill_t<false>(p, arena, stream);
}

}  // namespace oscar
