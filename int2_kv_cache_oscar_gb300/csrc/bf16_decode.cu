// BF16 reference split-K decode (sm_103a): the same persistent structure as
// the INT2 kernel over a plain bf16 K/V cache [slot][kv head][max_len][128].
// It stands in for the pages' comparator, BF16 FlashDecoding-v2 (ai-papers.net
// summary, section "実験結果"), to give the INT2/BF16 speed ratio on this GPU.
//
// Producer warp: 1-D bulk copies of 64-token K and V tiles (16 KB each) into
// a 3-stage ring.  Consumer warp: 8 lanes per token (16 channels each), 4
// tokens per step; fp32 dot products reduced with 3 shuffles, online softmax
// with a lazy rescale (the running max is only raised when a score exceeds it
// by more than 2^8, so p <= 256), fp32 P.V.
#include <cstddef>

#include "decode_common.cuh"

namespace oscar {
namespace {

constexpr int kConsumersB = 4;
constexpr int kThreadsB = (kConsumersB + 1) * 32;
constexpr int kStagesB = 3;
constexpr int kTile = 64;
constexpr int kTileBytes = kTile * kHeadDim * 2;

struct Bf16Smem {
  alignas(128) uint8_t k[kStagesB][kTileBytes];
  alignas(128) uint8_t v[kStagesB][kTileBytes];
  alignas(16) float ost[kConsumersB][kMaxGqa][kHeadDim];
  float mst[kConsumersB][kMaxGqa];
  float lst[kConsumersB][kMaxGqa];
  alignas(8) uint64_t full[kStagesB];
  uint64_t empty[kStagesB];
  uint32_t issued[kStagesB];   // uses of each stage issued so far (producer -> consumers)
  int abort_flag;
};
static_assert(offsetof(Bf16Smem, v) % 16 == 0, "bulk-copy destinations must be 16-byte aligned");
static_assert(offsetof(Bf16Smem, full) % 8 == 0, "mbarriers must be 8-byte aligned");

__device__ __forceinline__ void unpack8(const uint4 u, float* x) {
  x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

// 16 bf16 of one row chunk; lanes with sw = 1 read the upper 16 bytes first so
// that the 8 lanes of a token hit 8 distinct bank groups.
__device__ __forceinline__ void load16(const uint8_t* src, int sw, float* x) {
  const uint4* r = reinterpret_cast<const uint4*>(src);
  const uint4 c0 = r[sw], c1 = r[sw ^ 1];
  const uint4 lo = sw ? c1 : c0, hi = sw ? c0 : c1;
  unpack8(lo, &x[0]);
  unpack8(hi, &x[8]);
}

template <int MAXS>
__global__ void __launch_bounds__(kThreadsB, 2)
    decode_bf16_kernel(const __grid_constant__ DecodeParams<MAXS> p, const uint16_t* __restrict__ kc,
                       const uint16_t* __restrict__ vc) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Bf16Smem& S = *reinterpret_cast<Bf16Smem*>(smem_raw);
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

  if (warp == kConsumersB) {
    if (lane != 0) return;
    int64_t k = 0;
    int64_t u = u0;
    while (u < u1) {
      int b, j, g, ng;
      locate_unit(p, u, b, j, g, ng);
      const int len = p.seq[b].len;
      const int64_t row_end = p.seq[b].ubase + (int64_t)(j + 1) * ng;
      const int64_t seg_end = row_end < u1 ? row_end : u1;
      const int64_t rowbase = ((int64_t)p.seq[b].slot * hkv + j) * max_len;
      for (; u < seg_end; ++u, ++k, ++g) {
        const int s = (int)(k % kStagesB);
        if (k >= kStagesB) {
          if (!mbar_wait_bounded(&S.empty[s], (uint32_t)(((k / kStagesB) - 1) & 1), &S.abort_flag, p.h.err_word))
            goto drain;
        }
        const int rows = min(kTile, len - g * kTile);
        const uint32_t bytes = (uint32_t)rows * kHeadDim * 2;
        mbar_arrive_expect_tx(&S.full[s], 2 * bytes);
        const int64_t off = (rowbase + (int64_t)g * kTile) * kHeadDim;
        bulk_g2s(S.k[s], kc + off, bytes, &S.full[s]);
        bulk_g2s(S.v[s], vc + off, bytes, &S.full[s]);
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

  const int ts = lane >> 3;   // token slot 0..3
  const int cq = lane & 7;    // channels 16 cq .. 16 cq + 15
  const int sw = (cq >> 2) & 1;  // read order of the two 16-byte halves (bank spread)
  const int gqa = p.h.gqa;

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

    float qf[kMaxGqa][16];
#pragma unroll
    for (int h = 0; h < kMaxGqa; ++h) {
      if (h < gqa) {
        const uint4* q4 = reinterpret_cast<const uint4*>(p.h.q + ((int64_t)b * p.h.hq + j * gqa + h) * kHeadDim +
                                                         16 * cq);
        unpack8(q4[0], &qf[h][0]);
        unpack8(q4[1], &qf[h][8]);
#pragma unroll
        for (int i = 0; i < 16; ++i) qf[h][i] *= p.h.scale_log2;
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) qf[h][i] = 0.0f;
      }
    }
    float m[kMaxGqa], l[kMaxGqa], o[kMaxGqa][16];
#pragma unroll
    for (int h = 0; h < kMaxGqa; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) o[h][i] = 0.0f;
    }

    for (int64_t kk = k_begin + ((warp - k_begin) % kConsumersB + kConsumersB) % kConsumersB; kk < k_end;
         kk += kConsumersB) {
      const int s = (int)(kk % kStagesB);
      const uint32_t use = (uint32_t)(kk / kStagesB);
      if (!wait_issued(&S.issued[s], use, &S.abort_flag, p.h.err_word)) continue;
      if (!mbar_wait_bounded(&S.full[s], use & 1, &S.abort_flag, p.h.err_word)) continue;
      const int tile = g0 + (int)(kk - k_begin);
      const int rows = min(kTile, len - tile * kTile);
      const uint8_t* ktile = S.k[s];
      const uint8_t* vtile = S.v[s];
      for (int it = 0; it < kTile / 4; ++it) {
        const int t = 4 * it + ts;
        if (4 * it >= rows) break;                 // warp-uniform
        const bool valid = t < rows;
        const int tr = valid ? t : rows - 1;
        float kx[16];
        load16(ktile + tr * 256 + 32 * cq, sw, kx);
        float sc[kMaxGqa];
#pragma unroll
        for (int h = 0; h < kMaxGqa; ++h) {
          float d = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) d = fmaf(qf[h][i], kx[i], d);
          d += __shfl_xor_sync(0xffffffffu, d, 1);
          d += __shfl_xor_sync(0xffffffffu, d, 2);
          d += __shfl_xor_sync(0xffffffffu, d, 4);
          sc[h] = d;
        }
        if (valid) {
          float vx[16];
          load16(vtile + tr * 256 + 32 * cq, sw, vx);
#pragma unroll
          for (int h = 0; h < kMaxGqa; ++h) {
            if (sc[h] > m[h] + 8.0f) {
              const float a = exp2f(m[h] - sc[h]);
              m[h] = sc[h];
              l[h] *= a;
#pragma unroll
              for (int i = 0; i < 16; ++i) o[h][i] *= a;
            }
            const float pt = exp2f(sc[h] - m[h]);
            l[h] += pt;
#pragma unroll
            for (int i = 0; i < 16; ++i) o[h][i] = fmaf(pt, vx[i], o[h][i]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }

    // ---- merge the 4 token slots of the warp, then the CTA
#pragma unroll
    for (int h = 0; h < kMaxGqa; ++h) {
      float M = fmaxf(m[h], __shfl_xor_sync(0xffffffffu, m[h], 8));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
      const float a = (m[h] == -INFINITY) ? 0.0f : exp2f(m[h] - M);
      float lh = l[h] * a;
      lh += __shfl_xor_sync(0xffffffffu, lh, 8);
      lh += __shfl_xor_sync(0xffffffffu, lh, 16);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float x = o[h][i] * a;
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        o[h][i] = x;
      }
      if (ts == 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) S.ost[warp][h][16 * cq + i] = o[h][i];
      }
      if (lane == 0) {
        S.mst[warp][h] = M;
        S.lst[warp][h] = lh;
      }
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
  }  // this CTA's partials are written: let the dependent combine launch
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

int decode_bf16_ctas_per_sm() { return 2; }

template <int MAXS>
cudaError_t launch_decode_bf16(const DecodeParams<MAXS>& p, const uint16_t* kc, const uint16_t* vc,
                               cudaStream_t stream, cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (p.h.n_units <= 0) return cudaSuccess;
  const int smem = (int)sizeof(Bf16Smem);
  static bool attr_done[64] = {};
  cudaError_t e = ensure_smem_attr(decode_bf16_kernel<MAXS>, smem, attr_done);
  if (e != cudaSuccess) return e;
  if (ev_start) cudaEventRecord(ev_start, stream);
  decode_bf16_kernel<MAXS><<<p.h.n_ctas, kThreadsB, smem, stream>>>(p, kc, vc);
  e = cudaGetLastError();
  if (ev_stop) cudaEventRecord(ev_stop, stream);
  return e;
}

template cudaError_t launch_decode_bf16<kDecodeSeqsSmall>(const DecodeParams<kDecodeSeqsSmall>&, const uint16_t*,
                                                          const uint16_t*, cudaStream_t, cudaEvent_t, cudaEvent_t);
template cudaError_t launch_decode_bf16<kDecodeSeqsLarge>(const DecodeParams<kDecodeSeqsLarge>&, const uint16_t*,
                                                          const uint16_t*, cudaStream_t, cudaEvent_t, cudaEvent_t);

}  // namespace oscar
