// INT2 split-K decode attention over the packed OScaR cache (sm_103a), and
// the log-sum-exp combine kernel that also attends to the bf16 window.
//
// Score of a quantised token t for query q (OScaR abstract and ai-papers.net
// "OScaRの提案手法": keys are stored rotated by H_d and divided by their norm):
//   s_t = n_t * sum_c (H_d q)_c (code_tc s_c + z_c) * scale
//       = n_t * (sum_c code_tc (q_rot_c s_c) + sum_c q_rot_c z_c) * scale.
// Output: o = sum_t p_t (code^V_tc s^V_t,gr(c) + z^V_t,gr(c)) / sum_t p_t.
//
// Kernel structure (persistent CTAs, 2 per SM; 4 consumer warps + 1 helper):
//   * helper warp, lane 0: streams whole 13,824-byte group blocks (codes,
//     scales, zeros, norms of K and V) into a 6-stage shared-memory ring with
//     1-D bulk copies (cp.async.bulk + mbarrier transaction counts), 5 groups
//     ahead of the consumers;
//   * helper warp, all lanes: per segment it rotates the GQA queries (FWHT
//     over the lanes); per group it builds the B operand of the score
//     contraction, q_rot * s split into fp16 hi + lo columns and pre-scaled,
//     plus q_rot . z, into the stage's aux record;
//   * consumer warp w takes tokens 32w..32w+31 of every group and runs both
//     contractions with mma.sync m16n8k16: the 2-bit codes are the A operand,
//     taken straight from the packed words with one AND each (an fp16
//     subnormal code * 2^(p - 24)); the fp32 factors are the B operand split
//     into hi + lo fp16 columns (~22 significant bits) pre-scaled by 2^(F - p),
//     so each product is code * factor * 2^(F - 24); for P.V the hi/lo split
//     is shared between partner lanes (one shuffle);
//   * N = 8 columns = 4 query heads x {hi, lo}: all GQA heads share each tile;
//   * online softmax in the log2 domain per warp; tensor-core accumulators
//     restart at every group and are added into fp32 registers; every warp
//     waits on every stage in ring order, so the mbarrier parity test is exact.
#include <cstddef>

#include "decode_common.cuh"

namespace oscar {
namespace {

constexpr int kConsumers = 4;                  // consumer warps; warp w takes tokens 32w..32w+31
constexpr int kDecThreads = (kConsumers + 1) * 32;
constexpr int kStages = 6;
constexpr int kPbStride = 32 + 4;              // probability rows (4 heads x 32 tokens), padded

// Per-stage data the helper warp prepares for the consumers.
struct GroupAux {
  uint4 bk[4][32];       // score B fragments: {bk[2i][0], bk[2i][1], bk[2i+1][0], bk[2i+1][1]} per lane
  float qz[kMaxGqa];     // (H_d q_h) . z of the group, per query head
  float kq[kMaxGqa];     // 2^(24 - F_h): undoes the operand pre-scaling of head h
  float fv;              // 2^Fv: pre-scaling of the value-side operand
  float kv;              // 2^(24 - Fv)
  float pad[2];
};

struct DecSmem {
  alignas(128) uint8_t stage[kStages][kBlockBytes];
  alignas(16) GroupAux aux[kStages];
  alignas(16) float qrot[kMaxGqa][kHeadDim];               // helper: rotated queries of the segment
  alignas(16) float pbuf[kConsumers][kMaxGqa][kPbStride];  // consumer-private probabilities
  alignas(16) float ost[kConsumers][kMaxGqa][kHeadDim];
  float qmax[kMaxGqa];
  float mst[kConsumers][kMaxGqa];
  float lst[kConsumers][kMaxGqa];
  alignas(8) uint64_t full[kStages];
  uint64_t ready[kStages];
  uint64_t empty[kStages];
  int abort_flag;
};
static_assert(offsetof(DecSmem, aux) % 16 == 0, "aux must be 16-byte aligned");
static_assert(sizeof(GroupAux) % 16 == 0, "aux entries must stay 16-byte aligned");
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

template <int I>
__device__ __forceinline__ void extract4(uint32_t w0, uint32_t w1, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                         uint32_t& a3) {
  a0 = frag_extract<I>(w0);
  a1 = frag_extract<I>(w1);
  a2 = frag_extract<I + 1>(w0);
  a3 = frag_extract<I + 1>(w1);
}

// A fragment (k-step with ks & 3 == KK) from the two words of rows g, g+8.
template <int KK>
__device__ __forceinline__ void frag_a(uint32_t w0, uint32_t w1, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                       uint32_t& a3) {
  extract4<2 * KK>(w0, w1, a0, a1, a2, a3);
}

// Consumer work on tokens 32w .. 32w + 31 of one group block.  WQ = w & 1
// fixes which k-steps (tokens) of the P.V product this warp owns:
// ks = 2w, 2w + 1, i.e. kk = 2 WQ, 2 WQ + 1 within j = w >> 1.
struct ConsumerState {
  float m_run;
  float l_run;
  float o_acc[8][2];
  float zacc[kVGroups];
};

template <int WQ>
__device__ __forceinline__ void consume_group(const uint8_t* __restrict__ blk, const GroupAux& aux, int warp,
                                              int lane, float scale_log2, float* __restrict__ pbw,
                                              ConsumerState& st) {
  const int g = lane >> 2, tig = lane & 3;
  const int hb = g >> 1;
  const bool want_lo = (g & 1) != 0;
  const float* knm = reinterpret_cast<const float*>(blk + kOffKNorm);
  const float* vsz = reinterpret_cast<const float*>(blk + kOffVSZ);

  // ---- scores of tokens 16 mt + g (+8), mt = 2 warp + {0, 1}, head tig
  uint32_t bk[8][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = aux.bk[i][lane];
    bk[2 * i][0] = v.x;
    bk[2 * i][1] = v.y;
    bk[2 * i + 1][0] = v.z;
    bk[2 * i + 1][1] = v.w;
  }
  const float qz = aux.qz[tig];
  const float kq = aux.kq[tig];
  float sc[4];
  const uint4* kc = reinterpret_cast<const uint4*>(blk + kOffKCodes);
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int mt = 2 * warp + h2;
    const uint4 w = kc[mt * 32 + lane];
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t a0, a1, a2, a3;
    frag_a<0>(w.x, w.y, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[0][0], bk[0][1]);
    frag_a<1>(w.x, w.y, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[1][0], bk[1][1]);
    frag_a<2>(w.x, w.y, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[2][0], bk[2][1]);
    frag_a<3>(w.x, w.y, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[3][0], bk[3][1]);
    frag_a<0>(w.z, w.w, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[4][0], bk[4][1]);
    frag_a<1>(w.z, w.w, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[5][0], bk[5][1]);
    frag_a<2>(w.z, w.w, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[6][0], bk[6][1]);
    frag_a<3>(w.z, w.w, a0, a1, a2, a3); mma_f16_16816(acc, a0, a1, a2, a3, bk[7][0], bk[7][1]);
    const int t0 = 16 * mt + g;
    sc[2 * h2] = fmaf(acc[0] + acc[1], kq, qz) * knm[t0] * scale_log2;
    sc[2 * h2 + 1] = fmaf(acc[2] + acc[3], kq, qz) * knm[t0 + 8] * scale_log2;
  }

  // ---- online softmax over this warp's 32 tokens (head tig)
  float gm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
  gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
  const float m_new = fmaxf(st.m_run, gm);
  const float alpha = exp2f(st.m_run - m_new);
  st.m_run = m_new;
  float psum = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    sc[i] = exp2f(sc[i] - m_new);
    psum += sc[i];
  }
  st.l_run = fmaf(st.l_run, alpha, psum);
#pragma unroll
  for (int gr = 0; gr < kVGroups; ++gr) st.zacc[gr] *= alpha;
  float* pbt = pbw + tig * kPbStride;
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int tl = 16 * h2 + g;              // token index within the warp's 32
    const int t0 = 32 * warp + tl;
    pbt[tl] = sc[2 * h2];
    pbt[tl + 8] = sc[2 * h2 + 1];
    const float4 z0 = *reinterpret_cast<const float4*>(vsz + 8 * t0 + 4);
    const float4 z1 = *reinterpret_cast<const float4*>(vsz + 8 * (t0 + 8) + 4);
    st.zacc[0] = fmaf(sc[2 * h2], z0.x, fmaf(sc[2 * h2 + 1], z1.x, st.zacc[0]));
    st.zacc[1] = fmaf(sc[2 * h2], z0.y, fmaf(sc[2 * h2 + 1], z1.y, st.zacc[1]));
    st.zacc[2] = fmaf(sc[2 * h2], z0.z, fmaf(sc[2 * h2 + 1], z1.z, st.zacc[2]));
    st.zacc[3] = fmaf(sc[2 * h2], z0.w, fmaf(sc[2 * h2 + 1], z1.w, st.zacc[3]));
  }
  __syncwarp();

  // ---- P.V over this warp's two k-steps: O^T[channel][head x {hi, lo}]
  float pacc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) pacc[mt][0] = pacc[mt][1] = pacc[mt][2] = pacc[mt][3] = 0.0f;
  const int jh = warp >> 1;
  uint2 vw[8];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
    vw[mt] = *reinterpret_cast<const uint2*>(blk + kOffVCodes + ((mt * 32 + lane) * 4 + 2 * jh) * 4);
  const float* pbh = pbw + hb * kPbStride;
#pragma unroll
  for (int kk2 = 0; kk2 < 2; ++kk2) {
    constexpr int dummy = 0;
    (void)dummy;
    const int kk = 2 * WQ + kk2;               // ks & 3
    const int tl = 16 * kk2 + 2 * tig + (want_lo ? 8 : 0);   // this lane's two tokens (within the warp's 32)
    const int t = 32 * warp + tl;
    // lanes g even hold tokens +0,+1 (b0 half), g odd hold +8,+9 (b1 half); the
    // partner lane (g xor 1) covers the other half of the same column pair
    const float fsc = aux.fv * pow2f(-frag_p(2 * kk + (want_lo ? 1 : 0)));
    const float2 pp = *reinterpret_cast<const float2*>(pbh + tl);
    const float p0 = pp.x * fsc, p1 = pp.y * fsc;
    const float4 s0 = *reinterpret_cast<const float4*>(vsz + 8 * t);
    const float4 s1 = *reinterpret_cast<const float4*>(vsz + 8 * (t + 1));
    const float sA[4] = {s0.x, s0.y, s0.z, s0.w};
    const float sB[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int gr = 0; gr < kVGroups; ++gr) {
      const float x0 = p0 * sA[gr], x1 = p1 * sB[gr];
      const uint32_t hi = pack_half2(x0, x1);
      const uint32_t lo = pack_half2(x0 - half_lo_to_float(hi), x1 - half_hi_to_float(hi));
      const uint32_t send = want_lo ? hi : lo;
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 4);
      const uint32_t b0 = want_lo ? recv : hi;
      const uint32_t b1 = want_lo ? lo : recv;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int mt = 2 * gr + h2;
        uint32_t a0, a1, a2, a3;
        if (WQ == 0) {
          if (kk2 == 0) frag_a<0>(vw[mt].x, vw[mt].y, a0, a1, a2, a3);
          else frag_a<1>(vw[mt].x, vw[mt].y, a0, a1, a2, a3);
        } else {
          if (kk2 == 0) frag_a<2>(vw[mt].x, vw[mt].y, a0, a1, a2, a3);
          else frag_a<3>(vw[mt].x, vw[mt].y, a0, a1, a2, a3);
        }
        mma_f16_16816(pacc[mt], a0, a1, a2, a3, b0, b1);
      }
    }
  }
  const float kv = aux.kv;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    st.o_acc[mt][0] = fmaf(st.o_acc[mt][0], alpha, (pacc[mt][0] + pacc[mt][1]) * kv);
    st.o_acc[mt][1] = fmaf(st.o_acc[mt][1], alpha, (pacc[mt][2] + pacc[mt][3]) * kv);
  }
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
  const int64_t nloc = u1 - u0;
  const int hkv = p.h.hkv;
  const int gqa = p.h.gqa;
  const uint8_t* blocks = arena + p.h.blocks_off;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.ready[s], 32);          // every helper lane arrives after its writes
      mbar_init(&S.empty[s], kConsumers);
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ============================================================ helper warp
    const int g = lane >> 2, tig = lane & 3, hb = g >> 1;
    const bool want_lo = (g & 1) != 0;
    // lane 0: bulk copy of local unit k into its stage
    int64_t iss_u = u0;
    int iss_b = 0, iss_j = 0, iss_g = 0, iss_ng = 1;
    int64_t iss_k = 0;
    auto issue_next = [&]() {
      if (iss_k >= nloc) return;
      if (iss_k == 0 || iss_g >= iss_ng) locate_unit(p, iss_u, iss_b, iss_j, iss_g, iss_ng);
      const int s = (int)(iss_k % kStages);
      if (iss_k >= kStages)
        mbar_wait_bounded(&S.empty[s], (uint32_t)(((iss_k / kStages) - 1) & 1), &S.abort_flag, p.h.err_word);
      if (!S.abort_flag) {
        const uint8_t* src =
            blocks + (((int64_t)p.seq[iss_b].slot * hkv + iss_j) * p.h.max_groups + iss_g) * kBlockBytes;
        mbar_arrive_expect_tx(&S.full[s], kBlockBytes);
        bulk_g2s(S.stage[s], src, kBlockBytes, &S.full[s]);
      }
      ++iss_k;
      ++iss_u;
      ++iss_g;
    };
    if (lane == 0)
      for (int i = 0; i < kStages - 1; ++i) issue_next();

    float q2[32];
    float inv2F = 1.0f;
    float kq_h[kMaxGqa];
    float fv = 1.0f, kv = 1.0f;
    int64_t k = 0;
    int64_t u = u0;
    while (u < u1) {
      int b, j, g0, ng;
      locate_unit(p, u, b, j, g0, ng);
      const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
      const int64_t seg_end = row_end < u1 ? row_end : u1;
      // ---- segment setup: rotate the gqa queries (4 channels per lane)
      for (int h = 0; h < kMaxGqa; ++h) {
        float qv[4] = {0.f, 0.f, 0.f, 0.f};
        if (h < gqa) {
          const uint2 raw = *reinterpret_cast<const uint2*>(p.h.q + ((int64_t)b * p.h.hq + j * gqa + h) * kHeadDim +
                                                            4 * lane);
          qv[0] = bf16_lo(raw.x);
          qv[1] = bf16_hi(raw.x);
          qv[2] = bf16_lo(raw.y);
          qv[3] = bf16_hi(raw.y);
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
          const float inv_sqrt_d = 0.088388347648318440550f;  // 1/sqrt(128)
#pragma unroll
          for (int i = 0; i < 4; ++i) qv[i] *= inv_sqrt_d;
        }
        float mx = fmaxf(fmaxf(fabsf(qv[0]), fabsf(qv[1])), fmaxf(fabsf(qv[2]), fabsf(qv[3])));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        *reinterpret_cast<float4*>(&S.qrot[h][4 * lane]) = make_float4(qv[0], qv[1], qv[2], qv[3]);
        kq_h[h] = pow2f(24 - range_exponent(mx * (2.0f / 3.0f)));
        if (h == hb) {
          const int F = range_exponent(mx * (2.0f / 3.0f));
          inv2F = pow2f(-F);
        }
        if (lane == 0) S.qmax[h] = mx;
      }
      __syncwarp();
      {
        const int Fb = range_exponent(S.qmax[hb] * (2.0f / 3.0f));
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int c0 = 16 * ks + 2 * tig;
          const float f0 = pow2f(Fb - frag_p(2 * (ks & 3)));
          const float f1 = pow2f(Fb - frag_p(2 * (ks & 3) + 1));
          q2[4 * ks + 0] = S.qrot[hb][c0] * f0;
          q2[4 * ks + 1] = S.qrot[hb][c0 + 1] * f0;
          q2[4 * ks + 2] = S.qrot[hb][c0 + 8] * f1;
          q2[4 * ks + 3] = S.qrot[hb][c0 + 9] * f1;
        }
        const float vmax = __uint_as_float(
            reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[(int64_t)p.seq[b].slot * hkv + j]);
        const int Fv = range_exponent(vmax);
        fv = pow2f(Fv);
        kv = pow2f(24 - Fv);
      }
      // ---- per group: score operands into the stage's aux record
      for (; u < seg_end; ++u, ++k) {
        const int s = (int)(k % kStages);
        mbar_wait_bounded(&S.full[s], (uint32_t)((k / kStages) & 1), &S.abort_flag, p.h.err_word);
        const uint8_t* blk = S.stage[s];
        const float* ksc = reinterpret_cast<const float*>(blk + kOffKScale);
        const float* kze = reinterpret_cast<const float*>(blk + kOffKZero);
        GroupAux& ax = S.aux[s];
        float qzp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) qzp[i] = 0.0f;
#pragma unroll
        for (int ks2 = 0; ks2 < 4; ++ks2) {
          uint32_t r[4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ks = 2 * ks2 + e;
            const int c0 = 16 * ks + 2 * tig;
            const float2 s01 = *reinterpret_cast<const float2*>(ksc + c0);
            const float2 s89 = *reinterpret_cast<const float2*>(ksc + c0 + 8);
            const float2 z01 = *reinterpret_cast<const float2*>(kze + c0);
            const float2 z89 = *reinterpret_cast<const float2*>(kze + c0 + 8);
            r[2 * e] = split_half2(q2[4 * ks] * s01.x, q2[4 * ks + 1] * s01.y, want_lo);
            r[2 * e + 1] = split_half2(q2[4 * ks + 2] * s89.x, q2[4 * ks + 3] * s89.y, want_lo);
            const int i0 = 2 * (ks & 3);
            qzp[i0] = fmaf(q2[4 * ks], z01.x, fmaf(q2[4 * ks + 1], z01.y, qzp[i0]));
            qzp[i0 + 1] = fmaf(q2[4 * ks + 2], z89.x, fmaf(q2[4 * ks + 3], z89.y, qzp[i0 + 1]));
          }
          ax.bk[ks2][lane] = make_uint4(r[0], r[1], r[2], r[3]);
        }
        float qz = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) qz = fmaf(qzp[i], pow2f(frag_p(i)), qz);
        qz += __shfl_xor_sync(0xffffffffu, qz, 1);
        qz += __shfl_xor_sync(0xffffffffu, qz, 2);
        if ((lane & 7) == 0) ax.qz[hb] = qz * inv2F;   // lanes g = 2 hb, tig = 0
        if (lane < kMaxGqa) ax.kq[lane] = kq_h[lane < kMaxGqa ? lane : 0];
        if (lane == 0) {
          ax.fv = fv;
          ax.kv = kv;
        }
        mbar_arrive(&S.ready[s]);          // release of this lane's aux writes
        if (lane == 0) issue_next();       // refill: waits until the consumers released unit k - 1
        __syncwarp();
      }
    }
    if (lane == 0 && S.abort_flag) {
      // wait (bounded, once more) for the copies that may still be in flight
      const int64_t first = iss_k > kStages ? iss_k - kStages : 0;
      for (int64_t kk = first; kk < iss_k; ++kk) {
        const int s = (int)(kk % kStages);
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(&S.full[s], (uint32_t)((kk / kStages) & 1))) break;
      }
    }
    return;
  }

  // ============================================================== consumers
  const int g = lane >> 2;
  const int tig = lane & 3;
  const float scale_log2 = p.h.scale_log2;
  float* pbw = &S.pbuf[warp][0][0];

  int64_t k = 0;
  int64_t u = u0;
  while (u < u1) {
    int b, j, g0, ng;
    locate_unit(p, u, b, j, g0, ng);
    const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
    const int64_t seg_end = row_end < u1 ? row_end : u1;
    ConsumerState st;
    st.m_run = -INFINITY;
    st.l_run = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) st.o_acc[i][0] = st.o_acc[i][1] = 0.0f;
#pragma unroll
    for (int i = 0; i < kVGroups; ++i) st.zacc[i] = 0.0f;

    for (; u < seg_end; ++u, ++k) {
      const int s = (int)(k % kStages);
      const uint32_t par = (uint32_t)((k / kStages) & 1);
      const bool ok = mbar_wait_bounded(&S.ready[s], par, &S.abort_flag, p.h.err_word) &&
                      mbar_wait_bounded(&S.full[s], par, &S.abort_flag, p.h.err_word);
      if (ok) {
        if (warp & 1)
          consume_group<1>(S.stage[s], S.aux[s], warp, lane, scale_log2, pbw, st);
        else
          consume_group<0>(S.stage[s], S.aux[s], warp, lane, scale_log2, pbw, st);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }

    // ---- segment end: per-warp state -> shared memory -> CTA merge -> partial
    {
      float l = st.l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      float zs[kVGroups];
#pragma unroll
      for (int gr = 0; gr < kVGroups; ++gr) {
        float z = st.zacc[gr];
        z += __shfl_xor_sync(0xffffffffu, z, 4);
        z += __shfl_xor_sync(0xffffffffu, z, 8);
        z += __shfl_xor_sync(0xffffffffu, z, 16);
        zs[gr] = z;
      }
      if (g == 0) {
        S.mst[warp][tig] = st.m_run;
        S.lst[warp][tig] = l;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float zg = zs[mt >> 1];
        S.ost[warp][tig][16 * mt + g] = st.o_acc[mt][0] + zg;
        S.ost[warp][tig][16 * mt + g + 8] = st.o_acc[mt][1] + zg;
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
  }
}

// ---------------------------------------------------------------- combine
// One CTA per (sequence, KV head), 128 threads.  For each of the gqa query
// heads: attend to the bf16 window (unrotated q . k: the window holds raw
// keys), then merge the window state with the row's split-K partials:
// m* = max m_i, o = sum 2^(m_i - m*) o_i / sum 2^(m_i - m*) l_i, written as
// bf16.  The partial maxima are read by all threads at once and the weighted
// sum runs with independent loads per thread (thread = channel), so the
// merge costs a few memory latencies, not one per partial.
constexpr int kCombineMaxPartials = 2048;

template <int MAXS>
__global__ void __launch_bounds__(128)
    combine_kernel(const __grid_constant__ DecodeParams<MAXS> p, const uint8_t* __restrict__ arena) {
  __shared__ float wts[kCombineMaxPartials + 1];
  __shared__ float red[2][4];
  __shared__ float win_m[kMaxGqa], win_l[kMaxGqa];
  __shared__ __align__(16) float win_o[kMaxGqa][kHeadDim];
  const int b = blockIdx.x / p.h.hkv;
  const int j = blockIdx.x % p.h.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DecodeSeq sq = p.seq[b];
  const int hkv = p.h.hkv, gqa = p.h.gqa;
  const int ng = units_of_len(sq.len, p.h.bf16_mode);
  const int wlen = p.h.bf16_mode ? 0 : (sq.len % kGroup);
  const int64_t T = p.h.n_units, N = p.h.n_ctas;

  // ---- window attention: warp h handles query head h (4 channels per lane)
  for (int h = warp; h < gqa; h += 4) {
    float M = -INFINITY, L = 0.0f;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    if (wlen > 0) {
      const int qh = j * gqa + h;
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
    *reinterpret_cast<float4*>(&win_o[h][4 * lane]) = make_float4(o[0], o[1], o[2], o[3]);
    if (lane == 0) {
      win_m[h] = M;
      win_l[h] = L;
    }
  }
  __syncthreads();

  // ---- merge with the partials of this row
  int64_t first = 0, count = 0, rho = 0;
  if (ng > 0) {
    rho = (int64_t)hkv * sq.rank + j;
    const int64_t U = sq.ubase + (int64_t)j * ng;
    first = cta_of_unit(U, T, N);
    count = cta_of_unit(U + ng - 1, T, N) - first + 1;
    if (count > kCombineMaxPartials) count = kCombineMaxPartials;  // cannot happen: count <= N
  }
  for (int h = 0; h < gqa; ++h) {
    const float* base = p.h.partials + ((first + rho) * gqa + h) * (int64_t)kPartialFloats;
    const int64_t stride = (int64_t)gqa * kPartialFloats;
    // maximum over partials and window
    float mx = (tid == 0) ? win_m[h] : -INFINITY;
    for (int64_t i = tid; i < count; i += 128) mx = fmaxf(mx, base[i * stride + 128]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[0][warp] = mx;
    __syncthreads();
    const float Mx = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
    // weights and normaliser
    float lsum = 0.0f;
    for (int64_t i = tid; i < count; i += 128) {
      const float mi = base[i * stride + 128];
      const float w = (mi == -INFINITY) ? 0.0f : exp2f(mi - Mx);
      wts[i] = w;
      lsum = fmaf(w, base[i * stride + 129], lsum);
    }
    if (tid == 0) {
      const float w = (win_m[h] == -INFINITY) ? 0.0f : exp2f(win_m[h] - Mx);
      wts[kCombineMaxPartials] = w;
      lsum = fmaf(w, win_l[h], lsum);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (lane == 0) red[1][warp] = lsum;
    __syncthreads();
    const float Lt = red[1][0] + red[1][1] + red[1][2] + red[1][3];
    // weighted sum: thread = channel, independent loads across partials
    float acc = wts[kCombineMaxPartials] * win_o[h][tid];
    int64_t i = 0;
    for (; i + 4 <= count; i += 4) {
      const float x0 = base[(i + 0) * stride + tid];
      const float x1 = base[(i + 1) * stride + tid];
      const float x2 = base[(i + 2) * stride + tid];
      const float x3 = base[(i + 3) * stride + tid];
      acc = fmaf(wts[i], x0, acc);
      acc = fmaf(wts[i + 1], x1, acc);
      acc = fmaf(wts[i + 2], x2, acc);
      acc = fmaf(wts[i + 3], x3, acc);
    }
    for (; i < count; ++i) acc = fmaf(wts[i], base[i * stride + tid], acc);
    const float ov = acc / Lt;
    p.h.out[((int64_t)b * p.h.hq + j * gqa + h) * kHeadDim + tid] = (uint16_t)f32_to_bf16_bits(ov);
    __syncthreads();   // wts / red reused by the next head
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
  static bool attr_done[64] = {};
  cudaError_t e = ensure_smem_attr(decode_int2_kernel<MAXS>, smem, attr_done);
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
