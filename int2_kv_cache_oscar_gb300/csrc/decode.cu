// INT2 split-K decode attention over the packed OScaR cache (sm_103a), and
// the log-sum-exp combine kernel that also attends to the bf16 window.
//
// Score of a quantised token t for query q (OScaR abstract and ai-papers.net
// "OScaRの提案手法": keys are stored rotated by H_d and divided by their norm):
//   s_t = n_t * sum_c (H_d q)_c (code_tc s_c + z_c) * scale
//       = n_t * (sum_c code_tc (q_rot_c s_c) + sum_c q_rot_c z_c) * scale.
// Output: o = sum_t p_t (code^V_tc s^V_t,gr(c) + z^V_t,gr(c)) / sum_t p_t.
//
// Kernel structure (persistent CTAs, 2 per SM; 4 consumer warps + 1 producer
// warp):
//   * the producer streams whole group blocks (codes, scales, zeros, norms of
//     K and V; 13,824 bytes, or 11,008 with float16 metadata) into a 7-stage
//     (8-stage) shared-memory ring with 1-D bulk copies (cp.async.bulk +
//     mbarrier transaction counts) and publishes how many uses of each stage
//     it has issued, so that a consumer waits on a stage's barrier only for a
//     phase that exists (no parity aliasing);
//   * the grid is a programmatic dependent of the kernel before it: the
//     producer fills the ring with blocks of settled groups (ones no running
//     kernel can be writing; the host tracks appends) before the grid
//     dependency wait, so back-to-back steps overlap one step's ring fill
//     with the previous step's combine; everything else waits;
//   * each consumer warp takes every 4th group and runs both contractions on
//     the tensor cores with mma.sync m16n8k16: the 2-bit codes are the A
//     operand, taken straight from the packed words with one AND each (an
//     fp16 subnormal code * 2^(p - 24)); the fp32 factors (q_rot * s for
//     scores, p * s^V for values) are the B operand, split into fp16 hi + lo
//     columns (~22 significant bits) and pre-scaled by 2^(F - p) so the
//     product is code * factor * 2^(F - 24); partner lanes (hi column, lo
//     column of one head) each split half of the pairs and swap halves;
//   * N = 8 columns = 4 query heads x {hi, lo}: all GQA heads share each
//     loaded tile; the score k-steps run over 4 independent m-tile chains;
//   * online softmax in the log2 domain; tensor-core accumulators restart at
//     every group and are added into fp32 registers on the CUDA cores.
#include <cstddef>

#include "decode_common.cuh"

namespace oscar {
namespace {

constexpr int kConsumers = 4;
constexpr int kDecThreads = (kConsumers + 1) * 32;
constexpr int kCtasPerSm = 2;
// Ring stages filled before the grid dependency wait.  Back-to-back 128K
// steps (CUDA graph): 1, 2, 3, 4, 7 stages -> 30.1, 30.0, 30.2, 30.6, 31.8 us
// (31.3 us without the early fill); more stages crowd the previous kernel's
// own loads.
constexpr int kPreWaitStages = 2;
constexpr int kPbStride = kGroup + 16;  // probability rows (see pb_col)

// Ring geometry by metadata width: 7 stages of 13,824 B, or 8 of 11,008 B
// (float16 metadata), two CTAs per SM either way.
template <bool M16>
struct Ring {
  static constexpr int kStages = M16 ? 8 : 7;
  static constexpr int kStageBytes = Blk<M16>::kBytes;
};

static_assert(kConsumers < Ring<false>::kStages && kConsumers < Ring<true>::kStages, "one stage step per block");
static_assert(kPreWaitStages <= Ring<false>::kStages && kPreWaitStages <= Ring<true>::kStages &&
                  kConsumers <= Ring<false>::kStages && kConsumers <= Ring<true>::kStages,
              "the pre-wait fill uses each stage once (no free-slot waits)");

template <bool M16>
struct DecSmemT {
  static constexpr int kStages = Ring<M16>::kStages;
  alignas(128) uint8_t stage[kStages][Ring<M16>::kStageBytes];
  alignas(16) float qrot[kMaxGqaInt2][kHeadDim];          // float4 stores
  alignas(16) float4 q2t[2][4][32];                       // per-lane scaled query values, [head set][i/4][lane]
  // consumer-private probabilities; at a segment end each warp's region holds
  // its output rows ([head][channel]) for the CTA merge instead
  alignas(16) float pbuf[kConsumers][kMaxGqa][kPbStride];
  float qmax[kMaxGqaInt2];
  float mst[kConsumers][kMaxGqa];
  float lst[kConsumers][kMaxGqa];
  alignas(8) uint64_t full[kStages];
  uint64_t empty[kStages];
  uint32_t issued[kStages];   // uses of each stage issued so far (producer -> consumers)
  uint64_t qready;            // consumers have requested their first queries (-> producer)
  int abort_flag;
};
static_assert(kPbStride >= kHeadDim, "output rows must fit in the probability rows");
static_assert((kPbStride * 4) % 16 == 0, "pbuf rows must keep 16-byte alignment");
static_assert(offsetof(DecSmemT<false>, qrot) % 16 == 0 && offsetof(DecSmemT<true>, qrot) % 16 == 0,
              "qrot must be 16-byte aligned");
static_assert(offsetof(DecSmemT<false>, pbuf) % 16 == 0 && offsetof(DecSmemT<true>, pbuf) % 16 == 0,
              "pbuf must be 16-byte aligned");
static_assert(offsetof(DecSmemT<false>, full) % 8 == 0 && offsetof(DecSmemT<true>, full) % 8 == 0,
              "mbarriers must be 8-byte aligned");
static_assert(kBlockBytes % 128 == 0 && kBlockBytes16 % 128 == 0, "stages must stay 128-byte aligned");
static_assert(kCtasPerSm * (sizeof(DecSmemT<false>) + 1024) <= 233472 &&
                  kCtasPerSm * (sizeof(DecSmemT<true>) + 1024) <= 233472,
              "two CTAs per SM");


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
// The lo column holds the negated remainders, hi - x (exact in float32, one
// mixed-precision subtraction each with the fp16 operand taken in place), so
// a contraction's value is its hi column minus its lo column.
__device__ __forceinline__ void split_exchange(float x0, float x1, bool lo_lane, uint32_t& b0, uint32_t& b1) {
  const uint32_t hi = pack_half2(x0, x1);
  float r0, r1;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tsub.rn.f32.f16 %0, l, %3;\n\tsub.rn.f32.f16 %1, h, %4;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "r"(hi), "f"(x0), "f"(x1));
  const uint32_t lo = pack_half2(r0, r1);
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

// Waits until the kernels this grid depends on have completed and their
// writes are visible (returns at once when it was launched without a
// programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <int MAXS, bool M16, bool PAIRS>
__global__ void __launch_bounds__(kDecThreads, kCtasPerSm)
    decode_int2_kernel(const __grid_constant__ DecodeParams<MAXS> p, const uint8_t* __restrict__ arena) {
  using DecSmem = DecSmemT<M16>;
  using B = Blk<M16>;
  using MR = Meta<M16>;
  constexpr int kStages = DecSmem::kStages;
  constexpr int kStageBytes = B::kBytes;
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
      mbar_init(&S.empty[s], PAIRS ? 2 : 1);   // the warps that read each block
      S.issued[s] = 0;
    }
    mbar_init(&S.qready, kConsumers);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int64_t k = 0;
    int64_t u = u0;
    // Use k of the ring: stage ks = k mod kStages, its use ku = k / kStages,
    // both kept incrementally.  (Failure-path test: the copy of one unit of
    // CTA 0 is never issued, so the phase its consumer waits for never
    // completes.)
    int ks = 0;
    uint32_t ku = 0;
    auto issue = [&](const uint8_t* src) {
      if (!(cta == 0 && k == p.h.fault_unit)) {
        mbar_arrive_expect_tx(&S.full[ks], kStageBytes);
        bulk_g2s(S.stage[ks], src, kStageBytes, &S.full[ks]);
      }
      reinterpret_cast<volatile uint32_t*>(S.issued)[ks] = ku + 1;
      if (++ks == kStages) {
        ks = 0;
        ++ku;
      }
    };
    // Ring fill before the grid dependency wait: blocks of settled groups
    // (no kernel that may still run can be writing them), kPreWaitStages at
    // most.  Launched as a programmatic dependent, this grid starts while the
    // previous kernel finishes, and these copies overlap its tail.
    // a CTA with at most one unit per consumer fills all of them
    const int64_t pre = (u1 - u0) <= kConsumers ? kConsumers : kPreWaitStages;
    while (u < u1 && k < pre) {
      int b, j, g, ng;
      locate_unit(p, u, b, j, g, ng);
      const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
      const int64_t seg_end = row_end < u1 ? row_end : u1;
      const int settled = p.seq[b].settled;
      const uint8_t* src = blocks + (((int64_t)p.seq[b].slot * hkv + j) * p.h.max_groups + g) * kStageBytes;
      for (; u < seg_end && k < pre && g < settled; ++u, ++k, ++g, src += kStageBytes) issue(src);
      if (u < seg_end) break;         // an unsettled group (or the ring is full)
    }
    grid_dependency_wait();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!mbar_wait_bounded(&S.qready, 0, &S.abort_flag, p.h.err_word, p.h.spin_limit)) goto drain;
    while (u < u1) {
      int b, j, g, ng;
      locate_unit(p, u, b, j, g, ng);
      const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
      const int64_t seg_end = row_end < u1 ? row_end : u1;
      const uint8_t* src = blocks + (((int64_t)p.seq[b].slot * hkv + j) * p.h.max_groups + g) * kStageBytes;
      for (; u < seg_end; ++u, ++k, src += kStageBytes) {
        if (ku > 0) {   // the stage's previous use has been released
          if (!mbar_wait_bounded(&S.empty[ks], (ku - 1) & 1, &S.abort_flag, p.h.err_word, p.h.spin_limit)) {
            goto drain;
          }
        }
        issue(src);
      }
    }
  drain:
    if (S.abort_flag) {
      // wait (bounded, once more) for the copies that may still be in flight
      const int64_t first = k > kStages ? k - kStages : 0;
      for (int64_t kk = first; kk < k; ++kk) {
        const int s = (int)(kk % kStages);
        for (uint32_t i = 0; i < p.h.spin_limit; ++i)
          if (mbar_try_wait(&S.full[s], (uint32_t)((kk / kStages) & 1))) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;     // row group of the mma fragments
  const int tig = lane & 3;    // thread in group
  const int hb = g >> 1;       // head of this lane's B column
  const int half = g & 1;      // 0: hi column lane (computes b0 pairs), 1: lo column lane (b1 pairs)
  const bool lo_lane = half != 0;
  const int gqa = p.h.gqa;
  const float scale_log2 = p.h.scale_log2;
  // Up to 4 query heads: each warp takes every 4th block for all heads.  5 to
  // 8 (PAIRS): warps 2 i and 2 i + 1 read the same blocks (every 2nd) for head
  // sets 0-3 and 4-7, so the cache is streamed once for all of them.
  constexpr bool pairs = PAIRS;
  const int hs = pairs ? (warp & 1) : 0;          // head set of this warp
  const int h0 = kMaxGqa * hs;                    // its first query head
  const int cw = pairs ? (warp >> 1) : warp;      // block stream of this warp
  const int ncw = pairs ? kConsumers / 2 : kConsumers;

  // The queries, the value-scale maxima and the workspace are outputs of the
  // kernels before this one: wait for them.  Every CTA of this persistent grid
  // is resident from the start, so the dependent combine may be scheduled now:
  // its CTAs take SMs as these exit and attend to the window meanwhile (its
  // own grid dependency wait still waits for this whole grid).  Triggering
  // only after the wait keeps every kernel before this one complete by the
  // time a dependent of the combine starts.
  grid_dependency_wait();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // The query rows and value-scale maxima of this CTA's first two segments
  // are requested before the producer's copies past the ring fill (it waits
  // on qready): requested after them they would queue behind every CTA's
  // copies.
  uint2 qpre0 = make_uint2(0u, 0u), qpre1 = make_uint2(0u, 0u);
  uint32_t vpre0 = 0u, vpre1 = 0u;
  {
    int64_t uu = u0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (uu < u1) {
        int b, j, gg, ng;
        locate_unit(p, uu, b, j, gg, ng);
        uint2 qr = make_uint2(0u, 0u);
        if (warp < gqa)
          qr = *reinterpret_cast<const uint2*>(p.h.q + ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + warp) * kHeadDim + 4 * lane);
        const uint32_t vr = reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[(int64_t)p.seq[b].slot * hkv + j];
        if (i == 0) { qpre0 = qr; vpre0 = vr; } else { qpre1 = qr; vpre1 = vr; }
        const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
        uu = row_end < u1 ? row_end : u1;
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&S.qready);

  int64_t k = 0;
  int64_t u = u0;
  int seg_idx = 0;
  while (u < u1) {
    int b, j, g0, ng;
    locate_unit(p, u, b, j, g0, ng);
    const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
    const int64_t seg_end = row_end < u1 ? row_end : u1;
    const int64_t k_begin = k;
    const int64_t k_end = k + (seg_end - u);
    const int slot = p.seq[b].slot;

    // ---- segment setup: rotate the GQA queries (warp w rotates heads w and w + 4)
    for (int h = warp; h < (pairs ? kMaxGqaInt2 : kMaxGqa); h += kConsumers) {
      float qv[4] = {0.f, 0.f, 0.f, 0.f};
      if (h < gqa) {
        const uint2 raw = h == warp && seg_idx == 0   ? qpre0
                          : h == warp && seg_idx == 1 ? qpre1
                                                       : *reinterpret_cast<const uint2*>(
                                                             p.h.q + ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + h) * kHeadDim + 4 * lane);
        qv[0] = bf16_lo(raw.x);
        qv[1] = bf16_hi(raw.x);
        qv[2] = bf16_lo(raw.y);
        qv[3] = bf16_hi(raw.y);
        // channel c = 4 * lane + i: bits 0,1 in registers, bits 2..6 across lanes
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
      if (lane == 0) S.qmax[h] = mx;
    }
    named_bar_sync(1, kConsumers * 32);

    // per-lane constants of this segment
    const int Fk_b = range_exponent(S.qmax[h0 + hb] * (2.0f / 3.0f));     // B-column head h0 + hb
    const int Fk_s = range_exponent(S.qmax[h0 + tig] * (2.0f / 3.0f));    // score head h0 + tig
    const float kqs = pow2f(24 - Fk_s) * scale_log2;
    const float inv2Fk_b = pow2f(-Fk_b);
    const float vmax = __uint_as_float(
        seg_idx == 0   ? vpre0
        : seg_idx == 1 ? vpre1
                       : reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[(int64_t)slot * hkv + j]);
    const int Fv = range_exponent(vmax);
    const float fv = pow2f(Fv);
    const float kv = pow2f(24 - Fv);
    // q2 table: this lane's 16 query values (its half of each k-step's
    // channel pairs) times 2^(F - p); the same for every warp of a head set,
    // written by warp hs
    if (warp == hs) {
      float q2[16];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c = 16 * ks + 2 * tig + 8 * half;
        const int pp = half ? frag_p(2 * (ks & 3) + 1) : frag_p(2 * (ks & 3));
        const float f = pow2f(Fk_b - pp);
        q2[2 * ks] = S.qrot[h0 + hb][c] * f;
        q2[2 * ks + 1] = S.qrot[h0 + hb][c + 1] * f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) S.q2t[hs][i][lane] = make_float4(q2[4 * i], q2[4 * i + 1], q2[4 * i + 2], q2[4 * i + 3]);
    }
    named_bar_sync(1, kConsumers * 32);

    // bit-position weights of this lane's k-rows: 2^p for the score zero term,
    // 2^(Fv - p) for the value factors
    float zwk[4], fsc[4];
    // lane-constant parts of the swizzled shared-memory columns (token bit 3
    // is fixed for every access below): probability rows (pb_col) and the
    // float32 value scale / zero rows (vmeta_row), each relative to its
    // 16-token block
    const int pbs0 = g ^ (8 * ((tig >> 1) & 1));                      // row tig, token g
    const int pbs1 = (g + 8) ^ (8 * ((tig >> 1) & 1));                // row tig, token g + 8
    const int pbl = (2 * tig + 8 * half) ^ (8 * ((hb >> 1) & 1));     // row hb, tokens 2 tig + 8 half, + 1
    const int vsl0 = 16 * (2 * tig + 8 * half + half);                // bytes: token 2 tig + 8 half
    const int vsl1 = 16 * (2 * tig + 8 * half + 1 - half);            //        token 2 tig + 8 half + 1
    const int vzl0 = 16 * g, vzl1 = 16 * ((g + 8) ^ 1);               //        tokens g, g + 8
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int pp = half ? frag_p(2 * kk + 1) : frag_p(2 * kk);
      zwk[kk] = pow2f(pp);
      fsc[kk] = fv * pow2f(-pp);
    }

    float m_run = -INFINITY;   // running max (log2 units) of head tig
    float l_run = 0.0f;        // partial sum of p over this lane's tokens
    float2 o_acc[8];           // head tig, channels 16 mt + g (.x) and + 8 (.y), times 2^(Fv - 24)
    float2 zacc[kVGroups / 2]; // sum_t p_t z^V_t,gr over this lane's tokens, value groups (0, 1) and (2, 3)
#pragma unroll
    for (int i = 0; i < 8; ++i) o_acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < kVGroups / 2; ++i) zacc[i] = make_float2(0.0f, 0.0f);

    const int64_t kk0 = k_begin + ((cw - k_begin) % ncw + ncw) % ncw;
    int s_next = (int)(kk0 % kStages);               // stage and use of the next block, kept
    uint32_t use_next = (uint32_t)(kk0 / kStages);   // incrementally (ncw < kStages)
    for (int64_t kk = kk0; kk < k_end; kk += ncw) {
      const int s = s_next;
      const uint32_t use = use_next;
      s_next += ncw;
      if (s_next >= kStages) {
        s_next -= kStages;
        ++use_next;
      }
      if (!wait_issued(&S.issued[s], use, &S.abort_flag, p.h.err_word, p.h.spin_limit)) continue;
      if (!mbar_wait_bounded(&S.full[s], use & 1, &S.abort_flag, p.h.err_word, p.h.spin_limit)) continue;
      const uint8_t* blk = S.stage[s];
      const uint8_t* ksc = blk + B::kKScale;
      const uint8_t* kze = blk + B::kKZero;
      const uint8_t* knm = blk + B::kKNorm;
      const uint8_t* vsc = blk + B::kVScale;
      const uint8_t* vze = blk + B::kVZero;

      // ---- B fragments of the score contraction, and q_rot . z
      uint32_t bk[8][2];
      float2 qzc[4];   // per k-step class (ks & 3): sum of q2 * z over this lane's channel pairs
#pragma unroll
      for (int i = 0; i < 4; ++i) qzc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 q4 = S.q2t[hs][i][lane];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ks = 2 * i + e;
          const float2 qq = e ? make_float2(q4.z, q4.w) : make_float2(q4.x, q4.y);
          const int c = 16 * ks + 2 * tig + 8 * half;
          const float2 s2 = MR::two(ksc, c);
          const float2 z2 = MR::two(kze, c);
          const float2 x = __fmul2_rn(qq, s2);
          split_exchange(x.x, x.y, lo_lane, bk[ks][0], bk[ks][1]);
          qzc[ks & 3] = __ffma2_rn(qq, z2, qzc[ks & 3]);
        }
      }
      float qz = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) qz = fmaf(qzc[i].x + qzc[i].y, zwk[i], qz);
      qz += __shfl_xor_sync(0xffffffffu, qz, 1);
      qz += __shfl_xor_sync(0xffffffffu, qz, 2);
      qz += __shfl_xor_sync(0xffffffffu, qz, 4);
      qz *= inv2Fk_b;                                                          // q_rot[hb] . z
      const float qzs = __shfl_sync(0xffffffffu, qz, 8 * tig) * scale_log2;   // head tig, log2 units

      // ---- scores: S^T[token][head x {hi, lo}] = codes x B, 8 independent chains
      float2 sc[8];   // tokens 16 mt + g (.x) and + 8 (.y), head tig
      {
        const uint4* kc = reinterpret_cast<const uint4*>(blk + kOffKCodes);
        const float2 kq2 = make_float2(kqs, kqs), qz2 = make_float2(qzs, qzs);
#pragma unroll
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
            const float2 a = make_float2(acc[m][0] - acc[m][1], acc[m][2] - acc[m][3]);
            sc[mt] = __fmul2_rn(__ffma2_rn(a, kq2, qz2), make_float2(MR::one(knm, t0), MR::one(knm, t0 + 8)));
          }
        }
      }

      // ---- online softmax (head tig)
      float gm = fmaxf(sc[0].x, sc[0].y);
#pragma unroll
      for (int i = 1; i < 8; ++i) asm("max.f32 %0, %0, %1, %2;" : "+f"(gm) : "f"(sc[i].x), "f"(sc[i].y));
      gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
      gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
      gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
      const float m_new = fmaxf(m_run, gm);
      const float alpha = fast_exp2(m_run - m_new);
      m_run = m_new;
      const float2 neg_m = make_float2(-m_new, -m_new);
      float2 psum = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 d = __fadd2_rn(sc[i], neg_m);
        sc[i] = make_float2(fast_exp2(d.x), fast_exp2(d.y));
        psum = __fadd2_rn(psum, sc[i]);
      }
      l_run = fmaf(l_run, alpha, psum.x + psum.y);
#pragma unroll
      for (int i = 0; i < kVGroups / 2; ++i) zacc[i] = __fmul2_rn(zacc[i], make_float2(alpha, alpha));
      float* pb = S.pbuf[warp][tig];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int t0 = 16 * mt + g;
        pb[16 * mt + pbs0] = sc[mt].x;
        pb[16 * mt + pbs1] = sc[mt].y;
        float4 z0, z1;
        if constexpr (M16) {
          z0 = MR::v4(vze, t0);
          z1 = MR::v4(vze, t0 + 8);
        } else {
          z0 = *reinterpret_cast<const float4*>(vze + 256 * mt + vzl0);
          z1 = *reinterpret_cast<const float4*>(vze + 256 * mt + vzl1);
        }
        const float2 px = make_float2(sc[mt].x, sc[mt].x), py = make_float2(sc[mt].y, sc[mt].y);
        zacc[0] = __ffma2_rn(px, make_float2(z0.x, z0.y), __ffma2_rn(py, make_float2(z1.x, z1.y), zacc[0]));
        zacc[1] = __ffma2_rn(px, make_float2(z0.z, z0.w), __ffma2_rn(py, make_float2(z1.z, z1.w), zacc[1]));
      }
      __syncwarp();

      // ---- P.V: O^T[channel][head x {hi, lo}] = codes^V^T x (p * s^V); each
      // k-step's factors are built once and feed all 8 channel m-tiles
      {
        const float* pbh = S.pbuf[warp][hb];
        float pacc[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) pacc[mt][0] = pacc[mt][1] = pacc[mt][2] = pacc[mt][3] = 0.0f;
#pragma unroll
        for (int jh = 0; jh < 2; ++jh) {
          uint2 vw[8];
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
            vw[mt] = *reinterpret_cast<const uint2*>(blk + B::kVCodes + vword_off(mt, jh, lane));
#pragma unroll
          for (int kk2 = 0; kk2 < 4; ++kk2) {
            const int t = 16 * (4 * jh + kk2) + 2 * tig + 8 * half;   // this lane's two tokens
            const float2 pr = __fmul2_rn(*reinterpret_cast<const float2*>(pbh + 16 * (4 * jh + kk2) + pbl),
                                         make_float2(fsc[kk2], fsc[kk2]));
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
        const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          o_acc[mt] = __ffma2_rn(o_acc[mt], al2, make_float2(pacc[mt][0] - pacc[mt][1], pacc[mt][2] - pacc[mt][3]));
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
        float z = (gr & 1) ? zacc[gr >> 1].y : zacc[gr >> 1].x;
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
        S.pbuf[warp][tig][16 * mt + pbs0] = fmaf(o_acc[mt].x, kv, zg);
        S.pbuf[warp][tig][16 * mt + pbs1] = fmaf(o_acc[mt].y, kv, zg);
      }
    }
    named_bar_sync(1, kConsumers * 32);
    {
      const int64_t rho = (int64_t)hkv * p.seq[b].rank + j;
      float* part = p.h.partials + (cta + rho) * (int64_t)gqa * kPartialFloats;
      for (int idx = threadIdx.x; idx < gqa * kHeadDim; idx += kConsumers * 32) {
        const int h = idx >> 7;
        const int c = idx & (kHeadDim - 1);
        const int hw = h & (kMaxGqa - 1);   // the head's row in its warps' state
        const int w0 = pairs ? (h >> 2) : 0, dw = pairs ? 2 : 1;   // the warps of its head set
        float M = -INFINITY;
        for (int w = w0; w < kConsumers; w += dw) M = fmaxf(M, S.mst[w][hw]);
        float o = 0.0f, l = 0.0f;
        for (int w = w0; w < kConsumers; w += dw) {
          const float mw = S.mst[w][hw];
          const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - M);
          o = fmaf(f, S.pbuf[w][hw][pb_col(hw, c)], o);
          l = fmaf(f, S.lst[w][hw], l);
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
    ++seg_idx;
  }
}

// ---------------------------------------------------------------- combine
// One CTA per (sequence, KV head), 128 threads per query head (thread = one
// (head, channel) output).  It is launched as a programmatic dependent of the
// main kernel, which allows that at its start: combine CTAs take SMs as main
// CTAs exit and attend to the window (which the main kernel never reads) while
// the rest of the main grid drains; griddepcontrol.wait then guards every read
// of the partials.  Bulk copies stage the bf16 window rows (keys then values)
// and then the row's split-K partial records (contiguous slots) in shared
// memory; everything after that runs from shared memory:
//   window: the 4 warps of head h score 32 window tokens each (lane = token,
//           rotated 16-byte chunk order against bank conflicts); thread
//           (h, c) then sums p_t v_t;
//   merge:  m* = max(m_window, m_i), o = (sum 2^(m_i - m*) o_i) /
//           (sum 2^(m_i - m*) l_i), written as bf16.
constexpr int kCombineThreads = 128 * kMaxGqaInt2;   // launched with 128 x gqa
constexpr int kCombinePartBytes = 96 * 1024;   // at most this many bytes of partial records per chunk
constexpr int kCombineSmem = kWindowBytes + kCombinePartBytes;   // largest launch
constexpr int kCombineMaxChunk = kCombinePartBytes / (kPartialFloats * 4);

template <int MAXS>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const __grid_constant__ DecodeParams<MAXS> p, const uint8_t* __restrict__ arena) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // dynamic shared memory, sized per launch: window keys [wrows][128], window
  // values [wrows][128] (bf16), then a chunk of partial records
  const int wrows = p.h.comb_wrows;
  uint16_t* wk = reinterpret_cast<uint16_t*>(smem_raw);
  uint16_t* wv = wk + wrows * kHeadDim;
  float* part = reinterpret_cast<float*>(smem_raw + 2 * wrows * kHeadDim * 2);
  __shared__ __align__(16) float qs[kMaxGqaInt2][kHeadDim];
  __shared__ float pw[kMaxGqaInt2][kGroup];                             // window probabilities
  __shared__ float wts[kMaxGqaInt2][kCombineMaxChunk];
  __shared__ float red[kMaxGqaInt2][2][4];
  __shared__ float win_m[kMaxGqaInt2];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;

  const int b = blockIdx.x / p.h.hkv;
  const int j = blockIdx.x % p.h.hkv;
  const int tid = threadIdx.x;
  const int h = tid >> 7;            // query head within the group
  const int c = tid & 127;           // channel
  const int wih = c >> 5;            // warp within the head
  const int lane = tid & 31;
  const DecodeSeq sq = p.seq[b];
  const int hkv = p.h.hkv, gqa = p.h.gqa;
  const bool active = h < gqa;
  const int ng = units_of_len(sq.len, p.h.bf16_mode);
  const int wlen = p.h.bf16_mode ? 0 : (sq.len % kGroup);
  // fused append: the newest window row comes from the input (the host only
  // fuses when no group closes, so wlen >= 1); the others from the arena
  const bool fused = p.h.k_new != nullptr;
  const int wstored = fused ? wlen - 1 : wlen;
  const int64_t T = p.h.n_units, N = p.h.n_ctas;
  int64_t first = 0, count = 0, rho = 0;
  if (ng > 0) {
    rho = (int64_t)hkv * sq.rank + j;
    const int64_t U = sq.ubase + (int64_t)j * ng;
    first = cta_of_unit(U, T, N);
    count = cta_of_unit(U + ng - 1, T, N) - first + 1;
  }
  const int rec_bytes = gqa * kPartialFloats * 4;          // one slot: gqa records
  const int per_chunk = p.h.comb_part_bytes / rec_bytes;
  const int64_t nchunks = (count + per_chunk - 1) / per_chunk;

  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  qs[h][c] = active ? __uint_as_float((uint32_t)p.h.q[((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + h) * kHeadDim + c] << 16)
                    : 0.0f;
  if (fused && tid < 32) {
    // the new token: 16 x 16 bytes of K (tid < 16) and of V, into shared row
    // wlen - 1 and into the arena window slot it occupies from now on (the
    // main kernel never reads windows; the bulk copy below reads rows < wlen - 1)
    const int part = tid >> 4, chunk = tid & 15;
    const uint16_t* src = (part ? p.h.v_new : p.h.k_new) + ((int64_t)b * hkv + j) * kHeadDim + 8 * chunk;
    const uint4 val = *reinterpret_cast<const uint4*>(src);
    uint16_t* srow = (part ? wv : wk) + (wlen - 1) * kHeadDim;
    *reinterpret_cast<uint4*>(srow + 8 * chunk) = val;
    uint16_t* arow = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(arena) + p.h.windows_off +
                                                 ((int64_t)sq.slot * hkv + j) * kWindowBytes) +
                     part * kGroup * kHeadDim + (wlen - 1) * kHeadDim;
    *reinterpret_cast<uint4*>(arow + 8 * chunk) = val;
  }
  __syncthreads();
  // phase 0 of the barrier: the stored window rows
  if (tid == 0) {
    const uint32_t wbytes = (uint32_t)wstored * kHeadDim * 2;
    if (wbytes > 0) {
      mbar_arrive_expect_tx(&bar, 2 * wbytes);
      const uint8_t* wsrc = arena + p.h.windows_off + ((int64_t)sq.slot * hkv + j) * kWindowBytes;
      bulk_g2s(wk, wsrc, wbytes, &bar);
      bulk_g2s(wv, wsrc + kGroup * kHeadDim * 2, wbytes, &bar);
    } else {
      mbar_arrive(&bar);
    }
  }
  mbar_wait_bounded(&bar, 0, &abort_flag, p.h.err_word);

  // ---- window attention: warp wih of head h scores tokens 32 wih + lane
  float mxw = -INFINITY;
  float scw = -INFINITY;
  if (active) {
    const int t = 32 * wih + lane;
    if (t < wlen) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int ch = (i + lane) & 15;                       // rotated 16-byte chunk
        const uint4 kv4 = *reinterpret_cast<const uint4*>(wk + t * kHeadDim + 8 * ch);
        const float4 qa = *reinterpret_cast<const float4*>(&qs[h][8 * ch]);
        const float4 qb = *reinterpret_cast<const float4*>(&qs[h][8 * ch + 4]);
        a0 = fmaf(qa.x, bf16_lo(kv4.x), a0); a1 = fmaf(qa.y, bf16_hi(kv4.x), a1);
        a0 = fmaf(qa.z, bf16_lo(kv4.y), a0); a1 = fmaf(qa.w, bf16_hi(kv4.y), a1);
        a0 = fmaf(qb.x, bf16_lo(kv4.z), a0); a1 = fmaf(qb.y, bf16_hi(kv4.z), a1);
        a0 = fmaf(qb.z, bf16_lo(kv4.w), a0); a1 = fmaf(qb.w, bf16_hi(kv4.w), a1);
      }
      scw = (a0 + a1) * p.h.scale_log2;
    }
    mxw = scw;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mxw = fmaxf(mxw, __shfl_xor_sync(0xffffffffu, mxw, off));
    if (lane == 0) red[h][0][wih] = mxw;
  }
  __syncthreads();
  if (active) {
    const float M = fmaxf(fmaxf(red[h][0][0], red[h][0][1]), fmaxf(red[h][0][2], red[h][0][3]));
    const int t = 32 * wih + lane;
    const float pt = (t < wlen) ? exp2f(scw - M) : 0.0f;
    pw[h][t] = pt;
    float ls = pt;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    if (lane == 0) red[h][1][wih] = ls;
    if (c == 0) win_m[h] = (wlen > 0) ? M : -INFINITY;
  }
  __syncthreads();
  float Mh = -INFINITY, Lh = 0.0f, Oh = 0.0f;
  if (active) {
    Mh = win_m[h];
    Lh = red[h][1][0] + red[h][1][1] + red[h][1][2] + red[h][1][3];
    float o0 = 0.f, o1 = 0.f;
    int t = 0;
    for (; t + 2 <= wlen; t += 2) {
      o0 = fmaf(pw[h][t], __uint_as_float((uint32_t)wv[t * kHeadDim + c] << 16), o0);
      o1 = fmaf(pw[h][t + 1], __uint_as_float((uint32_t)wv[(t + 1) * kHeadDim + c] << 16), o1);
    }
    if (t < wlen) o0 = fmaf(pw[h][t], __uint_as_float((uint32_t)wv[t * kHeadDim + c] << 16), o0);
    Oh = o0 + o1;
  }

  // ---- merge: window state + partial records, chunk by chunk (heads in parallel);
  // chunk ck arrives on phase ck + 1 of the barrier
  grid_dependency_wait();            // the main kernel's partials are complete and visible
  // The next decode's main kernel may start now (it copies only blocks of
  // settled groups before its own wait, and every kernel before this one has
  // completed).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int64_t ck = 0; ck < nchunks; ++ck) {
    const int64_t c0 = ck * per_chunk;
    const int n = (int)((count - c0) < per_chunk ? (count - c0) : per_chunk);
    if (ck > 0) __syncthreads();                     // everyone done with the previous chunk
    if (tid == 0) {
      mbar_arrive_expect_tx(&bar, (uint32_t)(n * rec_bytes));
      bulk_g2s(part, p.h.partials + (first + rho + c0) * (int64_t)gqa * kPartialFloats, (uint32_t)(n * rec_bytes),
               &bar);
    }
    mbar_wait_bounded(&bar, (uint32_t)((ck + 1) & 1), &abort_flag, p.h.err_word);
    float mx = -INFINITY;
    if (active)
      for (int i = c; i < n; i += 128) mx = fmaxf(mx, part[(i * gqa + h) * kPartialFloats + 128]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (active && lane == 0) red[h][0][wih] = mx;
    __syncthreads();
    float Mn = Mh;
    if (active) {
      const float Mc = fmaxf(fmaxf(red[h][0][0], red[h][0][1]), fmaxf(red[h][0][2], red[h][0][3]));
      Mn = fmaxf(Mh, Mc);
    }
    float lsum = 0.0f;
    if (active)
      for (int i = c; i < n; i += 128) {
        const float mi = part[(i * gqa + h) * kPartialFloats + 128];
        const float w = (mi == -INFINITY) ? 0.0f : exp2f(mi - Mn);
        wts[h][i] = w;
        lsum = fmaf(w, part[(i * gqa + h) * kPartialFloats + 129], lsum);
      }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (active && lane == 0) red[h][1][wih] = lsum;
    __syncthreads();
    if (active) {
      const float Lc = red[h][1][0] + red[h][1][1] + red[h][1][2] + red[h][1][3];
      const float a = (Mh == -INFINITY) ? 0.0f : exp2f(Mh - Mn);
      float acc0 = Oh * a, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
      int i = 0;
      for (; i + 4 <= n; i += 4) {
        acc0 = fmaf(wts[h][i], part[((i + 0) * gqa + h) * kPartialFloats + c], acc0);
        acc1 = fmaf(wts[h][i + 1], part[((i + 1) * gqa + h) * kPartialFloats + c], acc1);
        acc2 = fmaf(wts[h][i + 2], part[((i + 2) * gqa + h) * kPartialFloats + c], acc2);
        acc3 = fmaf(wts[h][i + 3], part[((i + 3) * gqa + h) * kPartialFloats + c], acc3);
      }
      for (; i < n; ++i) acc0 = fmaf(wts[h][i], part[(i * gqa + h) * kPartialFloats + c], acc0);
      Oh = (acc0 + acc1) + (acc2 + acc3);
      Lh = Lh * a + Lc;
      Mh = Mn;
    }
  }
  if (active) {
    const float ov = Oh / Lh;
    const int64_t oi = ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + h) * kHeadDim + c;
    if (p.h.out_f32)
      reinterpret_cast<float*>(p.h.out)[oi] = ov;
    else
      p.h.out[oi] = (uint16_t)f32_to_bf16_bits(ov);
  }
}

}  // namespace

int decode_int2_ctas_per_sm() { return kCtasPerSm; }

int num_sms(int device) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  return n;
}

template <int MAXS, bool M16, bool PAIRS>
cudaError_t launch_decode_int2_t(const DecodeParams<MAXS>& p, const uint8_t* arena, cudaStream_t stream,
                                 cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (p.h.n_units <= 0) return cudaSuccess;
  const int smem = (int)sizeof(DecSmemT<M16>);
  static bool attr_done[64] = {};
  cudaError_t e = ensure_smem_attr(decode_int2_kernel<MAXS, M16, PAIRS>, smem, attr_done);
  if (e != cudaSuccess) return e;
  if (ev_start) cudaEventRecord(ev_start, stream);
  // programmatic dependent launch: the grid may start while the previous
  // kernel in the stream finishes (see the producer's ring fill)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.h.n_ctas);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_int2_kernel<MAXS, M16, PAIRS>, p, arena);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (ev_stop) cudaEventRecord(ev_stop, stream);
  return e;
}

template <int MAXS>
cudaError_t launch_decode_int2(const DecodeParams<MAXS>& p, const uint8_t* arena, bool meta16, cudaStream_t stream,
                               cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  // more than kMaxGqa query heads per KV head: two head sets on the same blocks
  if (p.h.gqa > kMaxGqa)
    return meta16 ? launch_decode_int2_t<MAXS, true, true>(p, arena, stream, ev_start, ev_stop)
                  : launch_decode_int2_t<MAXS, false, true>(p, arena, stream, ev_start, ev_stop);
  return meta16 ? launch_decode_int2_t<MAXS, true, false>(p, arena, stream, ev_start, ev_stop)
                : launch_decode_int2_t<MAXS, false, false>(p, arena, stream, ev_start, ev_stop);
}

template <int MAXS>
cudaError_t launch_combine(const DecodeParams<MAXS>& p, const uint8_t* arena, cudaStream_t stream) {
  static bool attr_done[64] = {};
  cudaError_t e = ensure_smem_attr(combine_kernel<MAXS>, kCombineSmem, attr_done);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: may start while the main kernel drains
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.h.n_seqs * p.h.hkv);
  cfg.blockDim = dim3(128 * p.h.gqa);
  cfg.dynamicSmemBytes = (size_t)2 * p.h.comb_wrows * kHeadDim * 2 + p.h.comb_part_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, combine_kernel<MAXS>, p, arena);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template cudaError_t launch_decode_int2<kDecodeSeqsSmall>(const DecodeParams<kDecodeSeqsSmall>&, const uint8_t*,
                                                          bool, cudaStream_t, cudaEvent_t, cudaEvent_t);
template cudaError_t launch_decode_int2<kDecodeSeqsLarge>(const DecodeParams<kDecodeSeqsLarge>&, const uint8_t*,
                                                          bool, cudaStream_t, cudaEvent_t, cudaEvent_t);
template cudaError_t launch_combine<kDecodeSeqsSmall>(const DecodeParams<kDecodeSeqsSmall>&, const uint8_t*,
                                                      cudaStream_t);
template cudaError_t launch_combine<kDecodeSeqsLarge>(const DecodeParams<kDecodeSeqsLarge>&, const uint8_t*,
                                                      cudaStream_t);

}  // namespace oscar
