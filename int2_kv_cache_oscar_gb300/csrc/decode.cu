// INT2 split-K decode attention over the packed OScaR cache (sm_103a), and
// the log-sum-exp combine kernel that also attends to the bf16 window.
//
// Score of a quantised token t for query q (OScaR abstract and ai-papers.net
// "OScaRの提案手法": keys are stored rotated by H_d and divided by their norm):
//   s_t = n_t * sum_c (H_d q)_c (code_tc s_c + z_c) * scale
//       = n_t * (sum_c code_tc (q_rot_c s_c) + sum_c q_rot_c z_c) * scale.
// Output: o = sum_t p_t (code^V_tc s^V_t,gr(c) + z^V_t,gr(c)) / sum_t p_t.
//
// Kernel structure (persistent, one CTA per SM slot, 4 consumer warps + 1
// producer warp):
//   * the producer streams whole 13,824-byte group blocks (codes, scales,
//     zeros, norms of K and V) into a 6-stage shared-memory ring with 1-D
//     bulk copies (cp.async.bulk + mbarrier transaction counts);
//   * each consumer warp takes every 4th group and runs both contractions on
//     the tensor cores with mma.sync m16n8k16: the 2-bit codes are the A
//     operand, taken straight from the packed words with one AND each (an
//     fp16 subnormal code * 2^(p - 24)); the fp32 factors (q_rot * s for
//     scores, p * s^V for values) are the B operand, split into fp16 hi + lo
//     columns (~22 significant bits) and pre-scaled by 2^(F - p) so the
//     product is code * factor * 2^(F - 24);
//   * N = 8 columns = 4 query heads x {hi, lo}: all GQA heads share each
//     loaded tile;
//   * online softmax in the log2 domain; tensor-core accumulators restart at
//     every group and are added into fp32 registers on the CUDA cores.
#include <cstddef>

#include "decode_common.cuh"

namespace oscar {
namespace {

constexpr int kConsumers = 4;
constexpr int kDecThreads = (kConsumers + 1) * 32;
constexpr int kStages = 6;
constexpr int kPbStride = kGroup + 8;  // probability rows, padded against bank conflicts

struct DecSmem {
  alignas(128) uint8_t stage[kStages][kBlockBytes];
  alignas(16) float qrot[kMaxGqa][kHeadDim];            // float4 stores
  alignas(16) float pbuf[kConsumers][kMaxGqa][kPbStride];  // float2 loads
  alignas(16) float ost[kConsumers][kMaxGqa][kHeadDim];
  float qmax[kMaxGqa];
  float mst[kConsumers][kMaxGqa];
  float lst[kConsumers][kMaxGqa];
  alignas(8) uint64_t full[kStages];
  uint64_t empty[kStages];
  uint32_t issued[kStages];   // uses of each stage issued so far (producer -> consumers)
  int abort_flag;
};
static_assert(offsetof(DecSmem, qrot) % 16 == 0, "qrot must be 16-byte aligned");
static_assert(offsetof(DecSmem, pbuf) % 16 == 0, "pbuf must be 16-byte aligned");
static_assert((kPbStride * 4) % 16 == 0, "pbuf rows must keep 16-byte alignment");
static_assert(offsetof(DecSmem, full) % 8 == 0, "mbarriers must be 8-byte aligned");
static_assert(kBlockBytes % 16 == 0, "stages must stay 16-byte aligned");

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

template <int MAXS>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_int2_kernel(const __grid_constant__ DecodeParams<MAXS> p, const uint8_t* __restrict__ arena) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecSmem& S = *reinterpret_cast<DecSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t T = p.h.n_units;
  const int64_t N = p.h.n_ctas;
  const int64_t cta = blockIdx.x;
  const int64_t u0 = cta_first_unit(cta, T, N);
  const int64_t u1 = cta_first_unit(cta + 1, T, N);
  const int hkv = p.h.hkv;
  const uint8_t* blocks = arena + p.h.blocks_off;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
      S.issued[s] = 0;
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int64_t k = 0;
    int64_t u = u0;
    while (u < u1) {
      int b, j, g, ng;
      locate_unit(p, u, b, j, g, ng);
      const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
      const int64_t seg_end = row_end < u1 ? row_end : u1;
      const uint8_t* src = blocks + (((int64_t)p.seq[b].slot * hkv + j) * p.h.max_groups + g) * kBlockBytes;
      for (; u < seg_end; ++u, ++k, src += kBlockBytes) {
        const int s = (int)(k % kStages);
        if (k >= kStages) {
          if (!mbar_wait_bounded(&S.empty[s], (uint32_t)(((k / kStages) - 1) & 1), &S.abort_flag, p.h.err_word)) {
            goto drain;
          }
        }
        mbar_arrive_expect_tx(&S.full[s], kBlockBytes);
        bulk_g2s(S.stage[s], src, kBlockBytes, &S.full[s]);
        reinterpret_cast<volatile uint32_t*>(S.issued)[s] = (uint32_t)(k / kStages) + 1;
      }
    }
  drain:
    if (S.abort_flag) {
      // wait (bounded, once more) for the copies that may still be in flight
      const int64_t first = k > kStages ? k - kStages : 0;
      for (int64_t kk = first; kk < k; ++kk) {
        const int s = (int)(kk % kStages);
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(&S.full[s], (uint32_t)((kk / kStages) & 1))) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;     // row group of the mma fragments
  const int tig = lane & 3;    // thread in group
  const int hb = g >> 1;       // head of this thread's B column
  const bool want_lo = (g & 1) != 0;
  const int gqa = p.h.gqa;
  const float scale_log2 = p.h.scale_log2;

  int64_t k = 0;
  int64_t u = u0;
  while (u < u1) {
    int b, j, g0, ng;
    locate_unit(p, u, b, j, g0, ng);
    const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
    const int64_t seg_end = row_end < u1 ? row_end : u1;
    const int64_t k_begin = k;
    const int64_t k_end = k + (seg_end - u);
    const int slot = p.seq[b].slot;

    // ---- segment setup: rotate the GQA queries (warp w rotates head w)
    {
      const int h = warp;
      float qv[4] = {0.f, 0.f, 0.f, 0.f};
      if (h < gqa) {
        const uint2 raw = *reinterpret_cast<const uint2*>(p.h.q + ((int64_t)b * p.h.hq + j * gqa + h) * kHeadDim +
                                                          4 * lane);
        qv[0] = bf16_lo(raw.x);
        qv[1] = bf16_hi(raw.x);
        qv[2] = bf16_lo(raw.y);
        qv[3] = bf16_hi(raw.y);
        // channel c = 4 * lane + i: bits 0,1 in registers, bits 2..6 across lanes
        float a = qv[0] + qv[1], bq = qv[0] - qv[1], c = qv[2] + qv[3], d = qv[2] - qv[3];
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
        const float inv_sqrt_d = 0.088388347648318440550f;  // 1/sqrt(128)
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[i] *= inv_sqrt_d;
      }
      float mx = fmaxf(fmaxf(fabsf(qv[0]), fabsf(qv[1])), fmaxf(fabsf(qv[2]), fabsf(qv[3])));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      *reinterpret_cast<float4*>(&S.qrot[h][4 * lane]) = make_float4(qv[0], qv[1], qv[2], qv[3]);
      if (lane == 0) S.qmax[h] = mx;
    }
    named_bar_sync(1, kConsumers * 32);

    // per-thread constants of this segment
    const int Fk_b = range_exponent(S.qmax[hb] * (2.0f / 3.0f));     // B-column head hb
    const int Fk_s = range_exponent(S.qmax[tig] * (2.0f / 3.0f));    // score head tig
    const float kq = pow2f(24 - Fk_s);
    const float vmax = __uint_as_float(
        reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[(int64_t)slot * hkv + j]);
    const int Fv = range_exponent(vmax);
    const float kv = pow2f(24 - Fv);
    float q2[32];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c0 = 16 * ks + 2 * tig;
      const float f0 = pow2f(Fk_b - frag_p(2 * (ks & 3)));
      const float f1 = pow2f(Fk_b - frag_p(2 * (ks & 3) + 1));
      q2[4 * ks + 0] = S.qrot[hb][c0] * f0;
      q2[4 * ks + 1] = S.qrot[hb][c0 + 1] * f0;
      q2[4 * ks + 2] = S.qrot[hb][c0 + 8] * f1;
      q2[4 * ks + 3] = S.qrot[hb][c0 + 9] * f1;
    }
    const float inv2Fk_b = pow2f(-Fk_b);

    float m_run = -INFINITY;   // running max (log2 units) of head tig
    float l_run = 0.0f;        // partial sum of p over this thread's tokens
    float o_acc[8][2];         // head tig, channels 16 mt + g + 8 r
    float zacc[kVGroups];      // sum_t p_t z^V_t,gr over this thread's tokens
#pragma unroll
    for (int i = 0; i < 8; ++i) o_acc[i][0] = o_acc[i][1] = 0.0f;
#pragma unroll
    for (int i = 0; i < kVGroups; ++i) zacc[i] = 0.0f;

    for (int64_t kk = k_begin + ((warp - k_begin) % kConsumers + kConsumers) % kConsumers; kk < k_end;
         kk += kConsumers) {
      const int s = (int)(kk % kStages);
      const uint32_t use = (uint32_t)(kk / kStages);
      if (!wait_issued(&S.issued[s], use, &S.abort_flag, p.h.err_word)) continue;
      if (!mbar_wait_bounded(&S.full[s], use & 1, &S.abort_flag, p.h.err_word)) continue;
      const uint8_t* blk = S.stage[s];
      const float* ksc = reinterpret_cast<const float*>(blk + kOffKScale);
      const float* kze = reinterpret_cast<const float*>(blk + kOffKZero);
      const float* knm = reinterpret_cast<const float*>(blk + kOffKNorm);
      const float* vsz = reinterpret_cast<const float*>(blk + kOffVSZ);

      // ---- B fragments of the score contraction, and q_rot . z
      uint32_t bk[8][2];
      float qzp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) qzp[i] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c0 = 16 * ks + 2 * tig;
        const float2 s01 = *reinterpret_cast<const float2*>(ksc + c0);
        const float2 s89 = *reinterpret_cast<const float2*>(ksc + c0 + 8);
        const float2 z01 = *reinterpret_cast<const float2*>(kze + c0);
        const float2 z89 = *reinterpret_cast<const float2*>(kze + c0 + 8);
        bk[ks][0] = split_half2(q2[4 * ks] * s01.x, q2[4 * ks + 1] * s01.y, want_lo);
        bk[ks][1] = split_half2(q2[4 * ks + 2] * s89.x, q2[4 * ks + 3] * s89.y, want_lo);
        const int i0 = 2 * (ks & 3);
        qzp[i0] = fmaf(q2[4 * ks], z01.x, fmaf(q2[4 * ks + 1], z01.y, qzp[i0]));
        qzp[i0 + 1] = fmaf(q2[4 * ks + 2], z89.x, fmaf(q2[4 * ks + 3], z89.y, qzp[i0 + 1]));
      }
      float qz = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) qz = fmaf(qzp[i], pow2f(frag_p(i)), qz);
      qz += __shfl_xor_sync(0xffffffffu, qz, 1);
      qz += __shfl_xor_sync(0xffffffffu, qz, 2);
      qz *= inv2Fk_b;                                        // q_rot[hb] . z
      const float qz_s = __shfl_sync(0xffffffffu, qz, 8 * tig);  // q_rot[tig] . z

      // ---- scores: S^T[token][head x {hi, lo}] = codes x B
      float sc[16];
      {
        const uint4* kc = reinterpret_cast<const uint4*>(blk + kOffKCodes);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const uint4 w = kc[mt * 32 + lane];
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t w0 = (ks < 4) ? w.x : w.z;
            const uint32_t w1 = (ks < 4) ? w.y : w.w;
            uint32_t a0, a1, a2, a3;
            switch (ks & 3) {
              case 0: a0 = frag_extract<0>(w0); a1 = frag_extract<0>(w1); a2 = frag_extract<1>(w0); a3 = frag_extract<1>(w1); break;
              case 1: a0 = frag_extract<2>(w0); a1 = frag_extract<2>(w1); a2 = frag_extract<3>(w0); a3 = frag_extract<3>(w1); break;
              case 2: a0 = frag_extract<4>(w0); a1 = frag_extract<4>(w1); a2 = frag_extract<5>(w0); a3 = frag_extract<5>(w1); break;
              default: a0 = frag_extract<6>(w0); a1 = frag_extract<6>(w1); a2 = frag_extract<7>(w0); a3 = frag_extract<7>(w1); break;
            }
            mma_f16_16816(acc, a0, a1, a2, a3, bk[ks][0], bk[ks][1]);
          }
          const int t0 = 16 * mt + g;
          sc[2 * mt] = fmaf(acc[0] + acc[1], kq, qz_s) * knm[t0] * scale_log2;
          sc[2 * mt + 1] = fmaf(acc[2] + acc[3], kq, qz_s) * knm[t0 + 8] * scale_log2;
        }
      }

      // ---- online softmax (head tig)
      float gm = sc[0];
#pragma unroll
      for (int i = 1; i < 16; ++i) gm = fmaxf(gm, sc[i]);
      gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
      gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
      gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
      const float m_new = fmaxf(m_run, gm);
      const float alpha = exp2f(m_run - m_new);
      m_run = m_new;
      float psum = 0.0f;
      float* pb = S.pbuf[warp][tig];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float pv = exp2f(sc[i] - m_new);
        sc[i] = pv;
        psum += pv;
      }
      l_run = fmaf(l_run, alpha, psum);
#pragma unroll
      for (int gr = 0; gr < kVGroups; ++gr) zacc[gr] *= alpha;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int t0 = 16 * mt + g;
        pb[t0] = sc[2 * mt];
        pb[t0 + 8] = sc[2 * mt + 1];
        const float4 z0 = *reinterpret_cast<const float4*>(vsz + 8 * t0 + 4);
        const float4 z1 = *reinterpret_cast<const float4*>(vsz + 8 * (t0 + 8) + 4);
        zacc[0] = fmaf(sc[2 * mt], z0.x, fmaf(sc[2 * mt + 1], z1.x, zacc[0]));
        zacc[1] = fmaf(sc[2 * mt], z0.y, fmaf(sc[2 * mt + 1], z1.y, zacc[1]));
        zacc[2] = fmaf(sc[2 * mt], z0.z, fmaf(sc[2 * mt + 1], z1.z, zacc[2]));
        zacc[3] = fmaf(sc[2 * mt], z0.w, fmaf(sc[2 * mt + 1], z1.w, zacc[3]));
      }
      __syncwarp();

      // ---- P.V: O^T[channel][head x {hi, lo}] = codes^V^T x (p * s^V)
      float pacc[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) pacc[mt][0] = pacc[mt][1] = pacc[mt][2] = pacc[mt][3] = 0.0f;
      const float* pbh = S.pbuf[warp][hb];
      const float fvs = pow2f(Fv);
#pragma unroll
      for (int jh = 0; jh < 2; ++jh) {
        uint2 vw[8];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          vw[mt] = *reinterpret_cast<const uint2*>(blk + kOffVCodes + ((mt * 32 + lane) * 4 + 2 * jh) * 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ks = 4 * jh + kk;
          const int t0 = 16 * ks + 2 * tig;
          float2 pa = *reinterpret_cast<const float2*>(pbh + t0);
          float2 pq = *reinterpret_cast<const float2*>(pbh + t0 + 8);
          const float fa = fvs * pow2f(-frag_p(2 * kk));
          const float fb = fvs * pow2f(-frag_p(2 * kk + 1));
          pa.x *= fa; pa.y *= fa; pq.x *= fb; pq.y *= fb;
          const float4 sa0 = *reinterpret_cast<const float4*>(vsz + 8 * t0);
          const float4 sa1 = *reinterpret_cast<const float4*>(vsz + 8 * (t0 + 1));
          const float4 sb0 = *reinterpret_cast<const float4*>(vsz + 8 * (t0 + 8));
          const float4 sb1 = *reinterpret_cast<const float4*>(vsz + 8 * (t0 + 9));
          const float sA0[4] = {sa0.x, sa0.y, sa0.z, sa0.w};
          const float sA1[4] = {sa1.x, sa1.y, sa1.z, sa1.w};
          const float sB0[4] = {sb0.x, sb0.y, sb0.z, sb0.w};
          const float sB1[4] = {sb1.x, sb1.y, sb1.z, sb1.w};
#pragma unroll
          for (int gr = 0; gr < kVGroups; ++gr) {
            const uint32_t b0 = split_half2(pa.x * sA0[gr], pa.y * sA1[gr], want_lo);
            const uint32_t b1 = split_half2(pq.x * sB0[gr], pq.y * sB1[gr], want_lo);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int mt = 2 * gr + h2;
              uint32_t a0, a1, a2, a3;
              switch (kk) {
                case 0: a0 = frag_extract<0>(vw[mt].x); a1 = frag_extract<0>(vw[mt].y); a2 = frag_extract<1>(vw[mt].x); a3 = frag_extract<1>(vw[mt].y); break;
                case 1: a0 = frag_extract<2>(vw[mt].x); a1 = frag_extract<2>(vw[mt].y); a2 = frag_extract<3>(vw[mt].x); a3 = frag_extract<3>(vw[mt].y); break;
                case 2: a0 = frag_extract<4>(vw[mt].x); a1 = frag_extract<4>(vw[mt].y); a2 = frag_extract<5>(vw[mt].x); a3 = frag_extract<5>(vw[mt].y); break;
                default: a0 = frag_extract<6>(vw[mt].x); a1 = frag_extract<6>(vw[mt].y); a2 = frag_extract<7>(vw[mt].x); a3 = frag_extract<7>(vw[mt].y); break;
              }
              mma_f16_16816(pacc[mt], a0, a1, a2, a3, b0, b1);
            }
          }
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o_acc[mt][0] = fmaf(o_acc[mt][0], alpha, (pacc[mt][0] + pacc[mt][1]) * kv);
        o_acc[mt][1] = fmaf(o_acc[mt][1], alpha, (pacc[mt][2] + pacc[mt][3]) * kv);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }

    // ---- segment end: per-warp state -> shared memory -> CTA merge -> partial
    {
      float l = l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
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
        S.mst[warp][tig] = m_run;
        S.lst[warp][tig] = l;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float zg = zs[mt >> 1];
        S.ost[warp][tig][16 * mt + g] = o_acc[mt][0] + zg;
        S.ost[warp][tig][16 * mt + g + 8] = o_acc[mt][1] + zg;
      }
    }
    named_bar_sync(1, kConsumers * 32);
    {
      const int c = threadIdx.x;  // 0..127: channel
      const int64_t rho = (int64_t)hkv * p.seq[b].rank + j;
      float* part = p.h.partials + (cta + rho) * (int64_t)gqa * kPartialFloats;
      for (int h = 0; h < gqa; ++h) {
        float M = S.mst[0][h];
#pragma unroll
        for (int w = 1; w < kConsumers; ++w) M = fmaxf(M, S.mst[w][h]);
        float o = 0.0f, l = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
          const float mw = S.mst[w][h];
          const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - M);
          o = fmaf(f, S.ost[w][h][c], o);
          l = fmaf(f, S.lst[w][h], l);
        }
        part[h * kPartialFloats + c] = o;
        if (c == 0) {
          part[h * kPartialFloats + 128] = M;
          part[h * kPartialFloats + 129] = l;
        }
      }
    }
    named_bar_sync(1, kConsumers * 32);
    k = k_end;
    u = seg_end;
  }
}

// ---------------------------------------------------------------- combine
// One CTA per (sequence, KV head): attend the gqa query heads to the bf16
// window (unrotated q . k, the window holds raw keys), then merge the window
// state with the split-K partials: m* = max m_i, o = sum 2^(m_i - m*) o_i /
// sum 2^(m_i - m*) l_i, written as bf16.
template <int MAXS>
__global__ void __launch_bounds__(128)
    combine_kernel(const __grid_constant__ DecodeParams<MAXS> p, const uint8_t* __restrict__ arena) {
  const int b = blockIdx.x / p.h.hkv;
  const int j = blockIdx.x % p.h.hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const DecodeSeq sq = p.seq[b];
  const int hkv = p.h.hkv, gqa = p.h.gqa;
  const int ng = units_of_len(sq.len, p.h.bf16_mode);
  const int wlen = p.h.bf16_mode ? 0 : (sq.len % kGroup);
  const int64_t T = p.h.n_units, N = p.h.n_ctas;
  for (int h = warp; h < gqa; h += 4) {
    const int qh = j * gqa + h;
    float M = -INFINITY, L = 0.0f;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    if (wlen > 0) {
      const uint2 qr = *reinterpret_cast<const uint2*>(p.h.q + ((int64_t)b * p.h.hq + qh) * kHeadDim + 4 * lane);
      const float q0 = bf16_lo(qr.x), q1 = bf16_hi(qr.x), q2 = bf16_lo(qr.y), q3 = bf16_hi(qr.y);
      const uint16_t* wk = reinterpret_cast<const uint16_t*>(
          arena + p.h.windows_off + ((int64_t)sq.slot * hkv + j) * kWindowBytes);
      const uint16_t* wv = wk + kGroup * kHeadDim;
      for (int t = 0; t < wlen; ++t) {
        const uint2 kr = *reinterpret_cast<const uint2*>(wk + t * kHeadDim + 4 * lane);
        float d = q0 * bf16_lo(kr.x) + q1 * bf16_hi(kr.x) + q2 * bf16_lo(kr.y) + q3 * bf16_hi(kr.y);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        const float s = d * p.h.scale_log2;
        const float Mn = fmaxf(M, s);
        const float a = exp2f(M - Mn);
        const float pt = exp2f(s - Mn);
        const uint2 vr = *reinterpret_cast<const uint2*>(wv + t * kHeadDim + 4 * lane);
        o[0] = fmaf(o[0], a, pt * bf16_lo(vr.x));
        o[1] = fmaf(o[1], a, pt * bf16_hi(vr.x));
        o[2] = fmaf(o[2], a, pt * bf16_lo(vr.y));
        o[3] = fmaf(o[3], a, pt * bf16_hi(vr.y));
        L = fmaf(L, a, pt);
        M = Mn;
      }
    }
    if (ng > 0) {
      const int64_t rho = (int64_t)hkv * sq.rank + j;
      const int64_t U = sq.ubase + (int64_t)j * ng;
      const int64_t first = cta_of_unit(U, T, N);
      const int64_t last = cta_of_unit(U + ng - 1, T, N);
      for (int64_t i = first; i <= last; ++i) {
        const float* part = p.h.partials + ((i + rho) * gqa + h) * (int64_t)kPartialFloats;
        const float mi = part[128], li = part[129];
        if (mi == -INFINITY) continue;
        const float4 oi = *reinterpret_cast<const float4*>(part + 4 * lane);
        const float Mn = fmaxf(M, mi);
        const float a = exp2f(M - Mn), bi = exp2f(mi - Mn);
        o[0] = o[0] * a + oi.x * bi;
        o[1] = o[1] * a + oi.y * bi;
        o[2] = o[2] * a + oi.z * bi;
        o[3] = o[3] * a + oi.w * bi;
        L = L * a + li * bi;
        M = Mn;
      }
    }
    const float inv = 1.0f / L;
    const uint32_t lo = f32_to_bf16_bits(o[0] * inv) | (f32_to_bf16_bits(o[1] * inv) << 16);
    const uint32_t hi = f32_to_bf16_bits(o[2] * inv) | (f32_to_bf16_bits(o[3] * inv) << 16);
    *reinterpret_cast<uint2*>(p.h.out + ((int64_t)b * p.h.hq + qh) * kHeadDim + 4 * lane) = make_uint2(lo, hi);
  }
}

}  // namespace

int decode_int2_ctas_per_sm() { return 2; }

int num_sms(int device) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  return n;
}

template <int MAXS>
cudaError_t launch_decode_int2(const DecodeParams<MAXS>& p, const uint8_t* arena, cudaStream_t stream,
                               cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (p.h.n_units <= 0) return cudaSuccess;
  const int smem = (int)sizeof(DecSmem);
  cudaError_t e = cudaFuncSetAttribute(decode_int2_kernel<MAXS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (ev_start) cudaEventRecord(ev_start, stream);
  decode_int2_kernel<MAXS><<<p.h.n_ctas, kDecThreads, smem, stream>>>(p, arena);
  e = cudaGetLastError();
  if (ev_stop) cudaEventRecord(ev_stop, stream);
  return e;
}

template <int MAXS>
cudaError_t launch_combine(const DecodeParams<MAXS>& p, const uint8_t* arena, cudaStream_t stream) {
  combine_kernel<MAXS><<<p.h.n_seqs * p.h.hkv, 128, 0, stream>>>(p, arena);
  return cudaGetLastError();
}

template cudaError_t launch_decode_int2<kDecodeSeqsSmall>(const DecodeParams<kDecodeSeqsSmall>&, const uint8_t*,
                                                          cudaStream_t, cudaEvent_t, cudaEvent_t);
template cudaError_t launch_decode_int2<kDecodeSeqsLarge>(const DecodeParams<kDecodeSeqsLarge>&, const uint8_t*,
                                                          cudaStream_t, cudaEvent_t, cudaEvent_t);
template cudaError_t launch_combine<kDecodeSeqsSmall>(const DecodeParams<kDecodeSeqsSmall>&, const uint8_t*,
                                                      cudaStream_t);
template cudaError_t launch_combine<kDecodeSeqsLarge>(const DecodeParams<kDecodeSeqsLarge>&, const uint8_t*,
                                                      cudaStream_t);

}  // namespace oscar
