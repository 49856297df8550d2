// Chunked-prefill attention over the packed OScaR cache: the launch of the
// tcgen05 history kernel (prefill_tc.cu) and, when the history is split into
// parts, the merge of their per-row records.
#include <cstddef>

#include "common.cuh"
#include "launch.h"

namespace oscar {
namespace {

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
  cudaError_t e = launch_prefill_tc(p, arena, M16, stream);
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
