// BF16 reference split-K decode (sm_103a): the same persistent structure as
// the INT2 kernel over a plain bf16 K/V cache [slot][kv head][max_len][128].
// It stands in for the pages' comparator, BF16 FlashDecoding-v2 (ai-papers.net
// summary, section "実験結果"), to give the INT2/BF16 speed ratio on this GPU.
//
//   * producer warp: 2-D TMA (cp.async.bulk.tensor, 128-byte swizzle) of
//     64-token K and V tiles, two 64x64 boxes each, into a 3-stage ring;
//   * consumer warp (every 4th tile): scores S^T = K q^T on the tensor cores
//     (mma.sync m16n8k16 bf16, A = K via ldmatrix, B = q, 4 of 8 columns
//     used), online softmax in fp32 (log2 domain), then O^T = V^T P^T with
//     A = V^T via ldmatrix.trans and B = P split into bf16 hi + lo columns
//     (4 heads x {hi, lo} = 8 columns); accumulators restart every tile and
//     are added into fp32 registers.
#include <cstddef>

#include <cudaTypedefs.h>

#include "decode_common.cuh"

namespace oscar {
namespace {

constexpr int kConsumersB = 4;
constexpr int kThreadsB = (kConsumersB + 1) * 32;
constexpr int kStagesB = 3;
constexpr int kTile = 64;
constexpr int kBoxBytes = 64 * 128;            // 64 rows x 64 bf16 channels
constexpr int kStageBytesB = 4 * kBoxBytes;    // K box 0, K box 1, V box 0, V box 1
constexpr int kPbStrideB = kTile + 4;

struct Bf16Smem {
  alignas(1024) uint8_t stage[kStagesB][kStageBytesB];
  alignas(16) float pbuf[kConsumersB][kMaxGqa][kPbStrideB];
  alignas(16) float ost[kConsumersB][kMaxGqa][kHeadDim];
  float mst[kConsumersB][kMaxGqa];
  float lst[kConsumersB][kMaxGqa];
  alignas(8) uint64_t full[kStagesB];
  uint64_t empty[kStagesB];
  uint32_t issued[kStagesB];   // uses of each stage issued so far (producer -> consumers)
  int abort_flag;
};
static_assert(kStageBytesB % 1024 == 0, "128-byte-swizzled boxes need 1024-byte alignment");
static_assert(offsetof(Bf16Smem, full) % 8 == 0, "mbarriers must be 8-byte aligned");

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Byte offset of row r, 16-byte chunk ch inside a 128-byte-swizzled 64x128 B box.
__device__ __forceinline__ uint32_t swz(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

// Partner-lane bf16 hi/lo split (see the INT2 kernel): lanes g = 2h (hi
// column) and g = 2h + 1 (lo column) each split one pair and swap halves.
__device__ __forceinline__ void split_exchange_bf16(float x0, float x1, bool lo_lane, uint32_t& b0, uint32_t& b1) {
  const uint32_t hi = pack_bf16x2(x0, x1);
  const float r0 = x0 - __uint_as_float(hi << 16);
  const float r1 = x1 - __uint_as_float(hi & 0xffff0000u);
  const uint32_t lo = pack_bf16x2(r0, r1);
  const uint32_t send = lo_lane ? hi : lo;
  const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 4);
  b0 = lo_lane ? recv : hi;
  b1 = lo_lane ? lo : recv;
}

template <int MAXS>
__global__ void __launch_bounds__(kThreadsB, 2)
    decode_bf16_kernel(const __grid_constant__ DecodeParams<MAXS> p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the dynamic window is only guaranteed 16-byte aligned: round up to 1024
  Bf16Smem& S = *reinterpret_cast<Bf16Smem*>(
      smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t T = p.h.n_units;
  const int64_t N = p.h.n_ctas;
  const int64_t cta = blockIdx.x;
  const int64_t u0 = cta_first_unit(cta, T, N);
  const int64_t u1 = cta_first_unit(cta + 1, T, N);
  const int hkv = p.h.hkv;
  const int64_t max_len = p.h.max_groups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
      S.issued[s] = 0;
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Every CTA of this grid is resident from the start (persistent grid), so
  // the dependent combine may be scheduled now: its CTAs take SMs as these
  // exit and stage what does not depend on the partials; its
  // griddepcontrol.wait still waits for this whole grid to complete.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kConsumersB) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int64_t k = 0;
    int64_t u = u0;
    while (u < u1) {
      int b, j, g, ng;
      locate_unit(p, u, b, j, g, ng);
      const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
      const int64_t seg_end = row_end < u1 ? row_end : u1;
      const int64_t rowbase = ((int64_t)p.seq[b].slot * hkv + j) * max_len;
      for (; u < seg_end; ++u, ++k, ++g) {
        const int s = (int)(k % kStagesB);
        if (k >= kStagesB) {
          if (!mbar_wait_bounded(&S.empty[s], (uint32_t)(((k / kStagesB) - 1) & 1), &S.abort_flag, p.h.err_word))
            goto drain;
        }
        const int r0 = (int)(rowbase + (int64_t)g * kTile);
        mbar_arrive_expect_tx(&S.full[s], kStageBytesB);
        tma_load_2d(S.stage[s] + 0 * kBoxBytes, &tmk, 0, r0, &S.full[s]);
        tma_load_2d(S.stage[s] + 1 * kBoxBytes, &tmk, 64, r0, &S.full[s]);
        tma_load_2d(S.stage[s] + 2 * kBoxBytes, &tmv, 0, r0, &S.full[s]);
        tma_load_2d(S.stage[s] + 3 * kBoxBytes, &tmv, 64, r0, &S.full[s]);
        reinterpret_cast<volatile uint32_t*>(S.issued)[s] = (uint32_t)(k / kStagesB) + 1;
      }
    }
  drain:
    if (S.abort_flag) {
      const int64_t first = k > kStagesB ? k - kStagesB : 0;
      for (int64_t kk = first; kk < k; ++kk) {
        const int s = (int)(kk % kStagesB);
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(&S.full[s], (uint32_t)((kk / kStagesB) & 1))) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, tig = lane & 3;
  const int hb = g >> 1;
  const int half = g & 1;
  const bool lo_lane = half != 0;
  const int gqa = p.h.gqa;
  const float scale_log2 = p.h.scale_log2;
  float* pbw = &S.pbuf[warp][0][0];

  int64_t k = 0;
  int64_t u = u0;
  while (u < u1) {
    int b, j, g0, ng;
    locate_unit(p, u, b, j, g0, ng);
    const int len = p.seq[b].len;
    const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
    const int64_t seg_end = row_end < u1 ? row_end : u1;
    const int64_t k_begin = k;
    const int64_t k_end = k + (seg_end - u);

    // B operand of the score contraction: column n = g is query head g (zero beyond gqa)
    uint32_t qb[8][2];
    {
      const uint16_t* qrow = p.h.q + ((int64_t)b * p.h.hq + j * p.h.q_group + p.h.q_head0 + (g < gqa ? g : 0)) * kHeadDim;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c = 16 * ks + 2 * tig;
        qb[ks][0] = g < gqa ? *reinterpret_cast<const uint32_t*>(qrow + c) : 0u;
        qb[ks][1] = g < gqa ? *reinterpret_cast<const uint32_t*>(qrow + c + 8) : 0u;
      }
    }
    float m_run[2] = {-INFINITY, -INFINITY};   // heads 2 tig, 2 tig + 1
    float l_run[2] = {0.0f, 0.0f};
    float o_acc[8][2];                         // head tig, channels 16 mt + g (+8)
#pragma unroll
    for (int i = 0; i < 8; ++i) o_acc[i][0] = o_acc[i][1] = 0.0f;

    for (int64_t kk = k_begin + ((warp - k_begin) % kConsumersB + kConsumersB) % kConsumersB; kk < k_end;
         kk += kConsumersB) {
      const int s = (int)(kk % kStagesB);
      const uint32_t use = (uint32_t)(kk / kStagesB);
      if (!wait_issued(&S.issued[s], use, &S.abort_flag, p.h.err_word)) continue;
      if (!mbar_wait_bounded(&S.full[s], use & 1, &S.abort_flag, p.h.err_word)) continue;
      const int tile = g0 + (int)(kk - k_begin);
      const int rows = min(kTile, len - tile * kTile);
      uint8_t* st = S.stage[s];
      if (rows < kTile) {
        // rows past the sequence end hold whatever the cache has there: zero them
        for (int idx = lane; idx < (kTile - rows) * 4 * 8; idx += 32) {
          const int r = rows + idx / 32, box = (idx / 8) & 3, q = idx & 7;
          reinterpret_cast<uint4*>(st + box * kBoxBytes + r * 128)[q] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      const uint32_t kbase = smem_u32(st);
      const uint32_t vbase = kbase + 2 * kBoxBytes;

      // ---- scores S^T[token][head]
      float sc[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int box = ks >> 2;
        const int ch = 2 * (ks & 3) + (lane >> 4);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const int r = 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kbase + box * kBoxBytes + swz(r, ch), a0, a1, a2, a3);
          mma_bf16_16816(sc[mt], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        }
      }
      // ---- online softmax for heads 2 tig + e (rows past the end masked)
      float gm[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int t = 16 * mt + g + 8 * r;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v = (t < rows) ? sc[mt][2 * r + e] * scale_log2 : -INFINITY;
            sc[mt][2 * r + e] = v;
            gm[e] = fmaxf(gm[e], v);
          }
        }
      }
      float alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        gm[e] = fmaxf(gm[e], __shfl_xor_sync(0xffffffffu, gm[e], 4));
        gm[e] = fmaxf(gm[e], __shfl_xor_sync(0xffffffffu, gm[e], 8));
        gm[e] = fmaxf(gm[e], __shfl_xor_sync(0xffffffffu, gm[e], 16));
        const float m_new = fmaxf(m_run[e], gm[e]);
        alpha[e] = exp2f(m_run[e] - m_new);
        m_run[e] = m_new;
        float ps = 0.0f;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float pv = exp2f(sc[mt][2 * r + e] - m_new);
            sc[mt][2 * r + e] = pv;
            ps += pv;
          }
        }
        l_run[e] = fmaf(l_run[e], alpha[e], ps);
      }
      if (tig < 2) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int e = 0; e < 2; ++e) pbw[(2 * tig + e) * kPbStrideB + 16 * mt + g + 8 * r] = sc[mt][2 * r + e];
      }
      __syncwarp();
      // alpha of head tig (the O rows this lane owns) from lane tig >> 1
      const float al0 = __shfl_sync(0xffffffffu, alpha[0], tig >> 1);
      const float al1 = __shfl_sync(0xffffffffu, alpha[1], tig >> 1);
      const float alpha_o = (tig & 1) ? al1 : al0;

      // ---- O^T[channel][head x {hi, lo}] = V^T x P^T
      float pacc[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) pacc[mt][0] = pacc[mt][1] = pacc[mt][2] = pacc[mt][3] = 0.0f;
      const float* pbh = pbw + hb * kPbStrideB;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int t = 16 * ks + 2 * tig + 8 * half;
        const float2 pp = *reinterpret_cast<const float2*>(pbh + t);
        uint32_t b0, b1;
        split_exchange_bf16(pp.x, pp.y, lo_lane, b0, b1);
        const int r = 16 * ks + (lane & 7) + ((lane >> 4) & 1) * 8;   // token row
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int box = mt >> 2;
          const int ch = 2 * (mt & 3) + ((lane >> 3) & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vbase + box * kBoxBytes + swz(r, ch), a0, a1, a2, a3);
          mma_bf16_16816(pacc[mt], a0, a1, a2, a3, b0, b1);
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o_acc[mt][0] = fmaf(o_acc[mt][0], alpha_o, pacc[mt][0] + pacc[mt][1]);
        o_acc[mt][1] = fmaf(o_acc[mt][1], alpha_o, pacc[mt][2] + pacc[mt][3]);
      }
      if (rows < kTile) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }

    // ---- segment end: per-warp state -> shared memory -> CTA merge -> partial
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_run[e];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (g == 0 && tig < 2) {
        S.mst[warp][2 * tig + e] = m_run[e];
        S.lst[warp][2 * tig + e] = l;
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      S.ost[warp][tig][16 * mt + g] = o_acc[mt][0];
      S.ost[warp][tig][16 * mt + g + 8] = o_acc[mt][1];
    }
    named_bar_sync(1, kConsumersB * 32);
    {
      const int c = threadIdx.x;
      const int64_t rho = (int64_t)hkv * p.seq[b].rank + j;
      float* part = p.h.partials + (cta + rho) * (int64_t)gqa * kPartialFloats;
      for (int h = 0; h < gqa; ++h) {
        float M = S.mst[0][h];
#pragma unroll
        for (int w = 1; w < kConsumersB; ++w) M = fmaxf(M, S.mst[w][h]);
        float oo = 0.0f, ll = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumersB; ++w) {
          const float mw = S.mst[w][h];
          const float f = (mw == -INFINITY) ? 0.0f : exp2f(mw - M);
          oo = fmaf(f, S.ost[w][h][c], oo);
          ll = fmaf(f, S.lst[w][h], ll);
        }
        part[h * kPartialFloats + c] = oo;
        if (c == 0) {
          part[h * kPartialFloats + 128] = M;
          part[h * kPartialFloats + 129] = ll;
        }
      }
    }
    named_bar_sync(1, kConsumersB * 32);
    k = k_end;
    u = seg_end;
  }
}

// 2-D tensor map over rows of 128 bf16 channels: box = 64 channels x 64 rows,
// 128-byte swizzle.
bool encode_rows_map(CUtensorMap* map, const void* base, uint64_t rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {kHeadDim, rows};
  const cuuint64_t strides[1] = {kHeadDim * 2};
  const cuuint32_t box[2] = {64, kTile};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int decode_bf16_ctas_per_sm() { return 2; }

template <int MAXS>
cudaError_t launch_decode_bf16(const DecodeParams<MAXS>& p, const uint16_t* kc, const uint16_t* vc,
                               cudaStream_t stream, cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (p.h.n_units <= 0) return cudaSuccess;
  int max_slot = 0;
  for (int i = 0; i < p.h.n_seqs; ++i) max_slot = p.seq[i].slot > max_slot ? p.seq[i].slot : max_slot;
  const uint64_t rows = (uint64_t)(max_slot + 1) * p.h.hkv * p.h.max_groups;
  CUtensorMap tmk, tmv;
  if (!encode_rows_map(&tmk, kc, rows) || !encode_rows_map(&tmv, vc, rows)) return cudaErrorInvalidValue;
  const int smem = (int)sizeof(Bf16Smem) + 1024;   // + slack for the 1024-byte alignment of the stages
  static bool attr_done[64] = {};
  cudaError_t e = ensure_smem_attr(decode_bf16_kernel<MAXS>, smem, attr_done);
  if (e != cudaSuccess) return e;
  if (ev_start) cudaEventRecord(ev_start, stream);
  decode_bf16_kernel<MAXS><<<p.h.n_ctas, kThreadsB, smem, stream>>>(p, tmk, tmv);
  e = cudaGetLastError();
  if (ev_stop) cudaEventRecord(ev_stop, stream);
  return e;
}

template cudaError_t launch_decode_bf16<kDecodeSeqsSmall>(const DecodeParams<kDecodeSeqsSmall>&, const uint16_t*,
                                                          const uint16_t*, cudaStream_t, cudaEvent_t, cudaEvent_t);
template cudaError_t launch_decode_bf16<kDecodeSeqsLarge>(const DecodeParams<kDecodeSeqsLarge>&, const uint16_t*,
                                                          const uint16_t*, cudaStream_t, cudaEvent_t, cudaEvent_t);

}  // namespace oscar
