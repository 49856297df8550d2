// OScaR compression kernel (sm_103a): quantise every 128-token group that
// fills during an append, and copy the remaining tokens into the bf16 window.
//
// Method ("OScaR", arXiv 2605.19660 Abstract; ai-papers.net summary, section
// "OScaRの提案手法"): Canalized Rotation (normalised Walsh-Hadamard H_d) of
// every key, then Omni-Token Scaling (store the token's L2 norm, divide the
// token by it), then per-channel asymmetric INT2 over the group's 128 tokens.
// Values: per-token asymmetric INT2 over 32-channel groups (KIVI convention
// cited in the qiita.com NOVA-KV article).
//
// One CTA = one (group, KV head), 256 threads; the thread pair (2t, 2t+1)
// owns token t, each thread 64 of its channels.
//   1. V: per 32-channel group min/max, s = (max-min)/3, z = min, codes; codes
//      go to shared memory (transposed), s/z to the block.
//   2. K: unnormalised fast Walsh-Hadamard transform, H_d = Hu / sqrt(128):
//      6 butterfly stages in registers, the 7th across the thread pair;
//      n_t = sqrt(|Hu k|^2 / 128); k_hat = Hu k / |Hu k| (= H_d k / n_t).
//   3. Per-channel min/max of k_hat over the 128 tokens (shared memory,
//      16-token slices, then 8 slices).
//   4. Codes of k_hat, packed straight into the fragment-order words.
//   5. Coalesced 16-byte stores of both code matrices.
#include <cstddef>

#include "common.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int kQThreads = 256;   // two threads per token: channels [0, 64) and [64, 128)
constexpr int kKhStride = 132;   // floats per k_hat row in shared memory (padding vs bank conflicts)
constexpr int kVbStride = 144;   // bytes per value-code row (channel) in shared memory
constexpr int kKrawOffset = 128 * kKhStride * 4 - 128 * 256;   // raw K rows at the end of the k_hat buffer

struct QuantSmem {
  alignas(16) float kh[kGroup * kKhStride];          // k_hat[t][c]; float4 stores / loads
  alignas(16) uint8_t vb[kHeadDim * kVbStride + 16];  // value codes [channel][permuted token]; uint4 loads
  alignas(16) float4 rmin[8][kHeadDim / 4];          // per 16-token slice: channel minima
  alignas(16) float4 rmax[8][kHeadDim / 4];          // per 16-token slice: channel maxima
  alignas(16) uint32_t kw[1024];                     // key code words, fragment order; uint4 loads
  alignas(16) float2 kp[kHeadDim + 4];               // per-channel (1/s, z), see kp_index
  float red[kQThreads / 32];
};
static_assert(offsetof(QuantSmem, vb) % 16 == 0 && offsetof(QuantSmem, kw) % 16 == 0, "alignment");
static_assert((kKhStride * 4) % 16 == 0 && kVbStride % 16 == 0, "rows must keep 16-byte alignment");

// Round-half-even code of x against (inv = 1/s, z): v = fl32(fl32(x - z) * inv)
// (the product is rounded before the integer rounding, as the decision rule
// specifies);
// x >= z and x <= max keep v in [0, 3] (s == 0 gives inv = 0, v = 0), so no
// clamp is needed; the magic constant 1.5 * 2^23 leaves rne(v) in the low
// mantissa bits.
__device__ __forceinline__ uint32_t int2_code(float x, float inv, float z) {
  const float v = __fmul_rn(x - z, inv);   // rounded product; never contracted into the add
  return __float_as_uint(v + 12582912.0f) & 3u;
}

// Byte offset of value-code row (channel) c: rows of the upper 64 channels are
// shifted by 16 bytes so that the two threads of a token (one per channel
// half) store into different banks.
__device__ __forceinline__ int vb_row(int c) { return c * kVbStride + ((c >> 6) << 4); }

// Index of channel c in the (1/s, z) table: the upper half is shifted by 4
// entries (32 bytes) for the same reason.
__device__ __forceinline__ int kp_index(int c) { return c + ((c >> 6) << 2); }

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Position of token/col c inside its 16-byte packing chunk of the byte
// staging area: chunk (tig, j), byte ((kk * 4) + hf + 2 e).
__device__ __forceinline__ int vb_perm(int c) {
  const int ks = c >> 4, j = ks >> 2, kk = ks & 3, hf = (c >> 3) & 1, tig = (c >> 1) & 3, e = c & 1;
  return ((tig * 2 + j) * 4 + kk) * 4 + hf + 2 * e;
}

__device__ __forceinline__ void load64(const uint16_t* src, float (&x)[64]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 u = __ldg(s + i);
    x[8 * i + 0] = bf16_lo(u.x);
    x[8 * i + 1] = bf16_hi(u.x);
    x[8 * i + 2] = bf16_lo(u.y);
    x[8 * i + 3] = bf16_hi(u.y);
    x[8 * i + 4] = bf16_lo(u.z);
    x[8 * i + 5] = bf16_hi(u.z);
    x[8 * i + 6] = bf16_lo(u.w);
    x[8 * i + 7] = bf16_hi(u.w);
  }
}

template <int CAP>
__global__ void __launch_bounds__(kQThreads, 2)
    quantize_append_kernel(const __grid_constant__ QuantPlan<CAP> plan, uint8_t* __restrict__ arena,
                           const uint16_t* __restrict__ kin, const uint16_t* __restrict__ vin) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  QuantSmem& S = *reinterpret_cast<QuantSmem*>(smem_raw);
  const int head = blockIdx.y;
  const int tid = threadIdx.x;
  const QuantTask T = plan.t[blockIdx.x];
  const int hkv = plan.hkv;
  const int64_t sh = (int64_t)T.slot * hkv + head;
  uint8_t* win = arena + plan.windows_off + sh * kWindowBytes;
  uint16_t* win_k = reinterpret_cast<uint16_t*>(win);
  uint16_t* win_v = win_k + kGroup * kHeadDim;

  if (T.kind == 0) {
    uint8_t* blk = arena + plan.blocks_off + (sh * plan.max_groups + T.group) * (int64_t)kBlockBytes;
    const int t = tid >> 1;          // token of the group
    const int half = tid & 1;        // channels [64 half, 64 half + 64)
    const bool from_win = t < T.n_win;
    const int64_t row = (int64_t)T.in_row + (t - T.n_win);
    const uint16_t* ksrc = (from_win ? win_k + t * kHeadDim : kin + (row * hkv + head) * kHeadDim) + 64 * half;
    const uint16_t* vsrc = (from_win ? win_v + t * kHeadDim : vin + (row * hkv + head) * kHeadDim) + 64 * half;

    // raw K rows (bf16, 256 B each) -> upper half of the k_hat buffer, in
    // flight while the values are processed; chunk i of a thread's 128 bytes
    // is stored at slot (i + t) mod 8 so that a warp's 16-byte accesses
    // spread over all bank groups
    uint8_t* kraw = reinterpret_cast<uint8_t*>(S.kh) + kKrawOffset;
#pragma unroll
    for (int i = 0; i < 8; ++i) cp_async16(kraw + t * 256 + 128 * half + 16 * ((i + t) & 7), ksrc + 8 * i);
    asm volatile("cp.async.commit_group;" ::: "memory");

    // ---- values: per-token INT2 over this thread's two 32-channel groups
    float smax = 0.0f;
    {
      float x[64];
      load64(vsrc, x);
      const int pt = vb_perm(t);
      float sv[2], zv[2];
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
        float mn = x[32 * g2], mx = x[32 * g2];
#pragma unroll
        for (int i = 1; i < kVGroup; ++i) {
          mn = fminf(mn, x[32 * g2 + i]);
          mx = fmaxf(mx, x[32 * g2 + i]);
        }
        const float sc = (mx - mn) / 3.0f;
        const float inv = sc > 0.0f ? 1.0f / sc : 0.0f;
        sv[g2] = sc;
        zv[g2] = mn;
        smax = fmaxf(smax, sc);
        const int gi = 2 * half + g2;
#pragma unroll
        for (int i = 0; i < kVGroup; ++i)
          S.vb[vb_row(gi * kVGroup + i) + pt] = (uint8_t)int2_code(x[32 * g2 + i], inv, mn);
      }
      *reinterpret_cast<float2*>(blk + kOffVSZ + 32 * t + 8 * half) = make_float2(sv[0], sv[1]);
      *reinterpret_cast<float2*>(blk + kOffVSZ + 32 * t + 16 + 8 * half) = make_float2(zv[0], zv[1]);
    }

    // ---- keys: rotation (6 butterfly stages in registers + 1 across the
    // thread pair), norm, unit vector
    float x[64];
    cp_async_wait_all();
    __syncthreads();                   // every thread's raw K row is in shared memory
    {
      const uint4* s4 = reinterpret_cast<const uint4*>(kraw + t * 256 + 128 * half);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 u = s4[(i + t) & 7];   // 16-byte chunks rotated by token: 8 bank groups per warp
        x[8 * i + 0] = bf16_lo(u.x);
        x[8 * i + 1] = bf16_hi(u.x);
        x[8 * i + 2] = bf16_lo(u.y);
        x[8 * i + 3] = bf16_hi(u.y);
        x[8 * i + 4] = bf16_lo(u.z);
        x[8 * i + 5] = bf16_hi(u.z);
        x[8 * i + 6] = bf16_lo(u.w);
        x[8 * i + 7] = bf16_hi(u.w);
      }
    }
    __syncthreads();                   // raw rows read before k_hat rows overwrite them
#pragma unroll
    for (int hb = 0; hb < 6; ++hb) {
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        const int h = 1 << hb;
        const int j = ((n >> hb) << (hb + 1)) | (n & (h - 1));
        const float a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float y = __shfl_xor_sync(0xffffffffu, x[i], 1);   // the partner's channel i + 64 or i - 64
      x[i] = half ? y - x[i] : x[i] + y;
    }
    float sq[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) sq[i] = x[i] * x[i] + x[i + 32] * x[i + 32];
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
      for (int i = 0; i < w; ++i) sq[i] += sq[i + w];
    }
    const float ss = sq[0] + __shfl_xor_sync(0xffffffffu, sq[0], 1);
    const float norm = sqrtf(ss * (1.0f / kHeadDim));
    const float rinv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) x[i] *= rinv;
    if (half == 0) reinterpret_cast<float*>(blk + kOffKNorm)[t] = norm;
    {
      float4* dst = reinterpret_cast<float4*>(&S.kh[t * kKhStride + 64 * half]);
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
    if ((tid & 31) == 0) S.red[tid >> 5] = smax;
    __syncthreads();

    // ---- per-channel key parameters: 16-token slices of 4 channels, then 8 slices
    {
      const int cq = tid & 31, ts = tid >> 5;
      float4 mn = *reinterpret_cast<const float4*>(&S.kh[(16 * ts) * kKhStride + 4 * cq]);
      float4 mx = mn;
#pragma unroll
      for (int r = 1; r < 16; ++r) {
        const float4 v = *reinterpret_cast<const float4*>(&S.kh[(16 * ts + r) * kKhStride + 4 * cq]);
        mn.x = fminf(mn.x, v.x); mn.y = fminf(mn.y, v.y); mn.z = fminf(mn.z, v.z); mn.w = fminf(mn.w, v.w);
        mx.x = fmaxf(mx.x, v.x); mx.y = fmaxf(mx.y, v.y); mx.z = fmaxf(mx.z, v.z); mx.w = fmaxf(mx.w, v.w);
      }
      S.rmin[ts][cq] = mn;
      S.rmax[ts][cq] = mx;
    }
    __syncthreads();
    if (tid < kHeadDim) {
      const int c = tid;
      const float* rmn = reinterpret_cast<const float*>(S.rmin);
      const float* rmx = reinterpret_cast<const float*>(S.rmax);
      float mn = rmn[c], mx = rmx[c];
#pragma unroll
      for (int ts = 1; ts < 8; ++ts) {
        mn = fminf(mn, rmn[ts * kHeadDim + c]);
        mx = fmaxf(mx, rmx[ts * kHeadDim + c]);
      }
      const float sc = (mx - mn) / 3.0f;
      S.kp[kp_index(c)] = make_float2(sc > 0.0f ? 1.0f / sc : 0.0f, mn);
      reinterpret_cast<float*>(blk + kOffKScale)[c] = sc;
      reinterpret_cast<float*>(blk + kOffKZero)[c] = mn;
    }
    __syncthreads();

    // ---- key codes of token t, channels of half: the 4 fragment words with j = half
    {
      const int mt = t >> 4, g = t & 7, r = (t >> 3) & 1;
#pragma unroll
      for (int tig = 0; tig < 4; ++tig) {
        uint32_t w = 0;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 16 * kk + 8 * hf + 2 * tig + e;    // channel 64 half + i
              const float2 pq = S.kp[kp_index(64 * half + i)];
              w |= int2_code(x[i], pq.x, pq.y) << (16 * e + 4 * kk + 2 * hf);
            }
          }
        }
        S.kw[((mt * 32 + 4 * g + tig) * 4) + 2 * half + r] = w;
      }
    }
    __syncthreads();

    // ---- coalesced stores of both code matrices (256 x 16 B each)
    {
      const int u = tid;
      reinterpret_cast<uint4*>(blk + kOffKCodes)[u] = reinterpret_cast<const uint4*>(S.kw)[u];
      const int mt = u >> 5, lane = u & 31, g = lane >> 2, tig = lane & 3;
      uint32_t wv[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int rowc = 16 * mt + g + 8 * r;
          const uint4 b = *reinterpret_cast<const uint4*>(&S.vb[vb_row(rowc) + (tig * 2 + j) * 16]);
          const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
          uint32_t w = 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t y = (bw[kk] | (bw[kk] >> 6)) & 0x000F000Fu;
            w |= y << (4 * kk);
          }
          wv[2 * j + r] = w;
        }
      }
      reinterpret_cast<uint4*>(blk + kOffVCodes)[u] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
    if (tid == 0) {
      float m = S.red[0];
#pragma unroll
      for (int i = 1; i < kQThreads / 32; ++i) m = fmaxf(m, S.red[i]);
      atomicMax(reinterpret_cast<unsigned int*>(arena + kMetaHeader) + sh, __float_as_uint(m));
    }
    if (T.tail_count <= 0) return;
    // the window reads above completed before the first __syncthreads
  }

  // ---- window append: rows tail_in_row.. -> window slots (tail_pos + i) mod 128
  {
    const int count = T.tail_count;
    for (int idx = tid; idx < count * 16; idx += kQThreads) {
      const int i = idx >> 4, q = idx & 15;
      const int64_t row = (int64_t)T.tail_in_row + i;
      const int slot = (T.tail_pos + i) & (kGroup - 1);
      const uint4* ks = reinterpret_cast<const uint4*>(kin + (row * hkv + head) * kHeadDim);
      const uint4* vs = reinterpret_cast<const uint4*>(vin + (row * hkv + head) * kHeadDim);
      reinterpret_cast<uint4*>(win_k + slot * kHeadDim)[q] = __ldg(ks + q);
      reinterpret_cast<uint4*>(win_v + slot * kHeadDim)[q] = __ldg(vs + q);
    }
  }
}

template <int CAP>
cudaError_t launch_quantize(const QuantPlan<CAP>& plan, uint8_t* arena, const uint16_t* k, const uint16_t* v,
                            cudaStream_t stream) {
  if (plan.n_tasks <= 0) return cudaSuccess;
  const int smem = (int)sizeof(QuantSmem);
  static bool attr_done[64] = {};
  cudaError_t e = ensure_smem_attr(quantize_append_kernel<CAP>, smem, attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid(plan.n_tasks, plan.hkv);
  quantize_append_kernel<CAP><<<grid, kQThreads, smem, stream>>>(plan, arena, k, v);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_small(const QuantPlan<kQuantPlanSmall>& plan, uint8_t* arena, const uint16_t* k,
                                  const uint16_t* v, cudaStream_t stream) {
  return launch_quantize(plan, arena, k, v, stream);
}

cudaError_t launch_quantize_large(const QuantPlan<kQuantPlanLarge>& plan, uint8_t* arena, const uint16_t* k,
                                  const uint16_t* v, cudaStream_t stream) {
  return launch_quantize(plan, arena, k, v, stream);
}

}  // namespace oscar
