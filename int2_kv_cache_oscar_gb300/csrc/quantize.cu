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
// owns token t, each thread 64 of its channels (128 bytes of the key row and
// of the value row, read with 32-byte loads when the inputs allow).
//   1. V: per 32-channel group min/max (on packed bf16 pairs: exact), s =
//      (max-min)/3, z = min, codes; codes go to shared memory (transposed,
//      four channels per byte), s/z to the block.  The key row is already
//      being loaded into registers.
//   2. K: unnormalised fast Walsh-Hadamard transform, H_d = Hu / sqrt(128):
//      6 butterfly stages in registers (the first as the bf16 words are
//      widened, with mixed-precision adds; the others packed f32x2), the 7th
//      across the thread pair with shuffles of half the values (after it each thread
//      holds channels [32 half, + 32) and [64 + 32 half, + 32));
//      n_t = sqrt(|Hu k|^2 / 128); k_hat = Hu k / |Hu k| (= H_d k / n_t).
//   3. Per-channel min/max of k_hat over the 128 tokens (shared memory,
//      16-token slices, then 8 slices).
//   4. Codes of k_hat, packed straight into the fragment-order words and
//      stored; the value code words are stored in V order from the staged
//      bytes after the first barrier.
// A code is round_half_even((x - z) / s) of the stored s and z, clamped.
// Key codes: fl32(x - z) * fl32(1/s) rounded once to the nearest integer by
// a fused multiply-add with 1.5 * 2^23; with the fp32 k_hat, quotients within
// a few ulp of a tie are rare (about 1e-7 of the benchmark keys' codes, always
// inside the 1e-3-step boundary window).  Value codes: bf16 values make exact
// ties, and quotients a hair off a tie, common (about 1e-4 of the codes), so
// the value decision is made exact there, see value_coefficients.  The packed
// f32x2 operations round each lane exactly like the scalar ones.
#include <cstddef>

#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int kQThreads = 256;   // two threads per token: channels [0, 64) and [64, 128)
constexpr int kVbStride = 144;   // bytes per value-code row (4 channels) in shared memory
constexpr int kVbRows = kHeadDim / 4;
constexpr float kMagic = 12582912.0f;                          // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;

struct QuantSmem {
  alignas(16) float kh[kGroup * kHeadDim];           // k_hat[t][4 kh_slot(t, c / 4) + c % 4]; float4 stores / loads
  alignas(16) uint8_t vb[kVbRows * kVbStride + 16];  // value codes [channel / 4][permuted token]; uint4 loads
  alignas(16) float4 rmin[8][kHeadDim / 4];          // per 16-token slice: channel minima
  alignas(16) float4 rmax[8][kHeadDim / 4];          // per 16-token slice: channel maxima
  alignas(16) float4 kq[kHeadDim / 2 + 4];           // per channel pair (1/s, 1/s', -z, -z'), see kq_index
  uint32_t red[2][kQThreads / 32];   // per warp: largest value scale, largest |value zero| (float bits)
};
static_assert(offsetof(QuantSmem, vb) % 16 == 0, "alignment");
static_assert(offsetof(QuantSmem, kq) % 16 == 0, "alignment");
static_assert(kVbStride % 16 == 0, "rows must keep 16-byte alignment");

// Physical float4 slot of float4 column q (channels 4q .. 4q + 3) of k_hat
// row t.  The 8 threads of a quarter warp (tokens t .. t + 3, both threads of
// each) store columns 8 h + i and 16 + 8 h + i (thread h of the pair): the
// XOR sends them to 8 different bank groups.  It only permutes slots within
// aligned groups of 8, so a warp reading a whole row stays conflict-free.
__device__ __forceinline__ int kh_slot(int t, int q) { return q ^ (((t & 3) << 1) | ((q >> 3) & 1)); }

// Entry of channel pair (c, c + 1) in the key-parameter table: every 32
// channels shift by one more entry (16 bytes), so that the two threads of a
// token (channels c and c + 32 at the same step) read different banks.
__device__ __forceinline__ int kq_index(int c) { return (c >> 1) + (c >> 5); }

// Value decisions.  With d = x - z (exact: x, z and max - min are bf16
// values, or the float16 zero, in float32) and r = fl32(1/s), the quotient
// P = d r, evaluated as below, is within 4 2^-24 P of d / s (the roundings
// of r, of the coefficient b and of the two multiply-adds).  That decides
// every code except where d / s is within that distance of a boundary
// j + 1/2, and bf16 values put d / s there in two ways:
//   * exactly on the tie (2 d = (2j + 1) s): half to even, i.e. down at 0.5
//     and 2.5, up at 1.5;
//   * a hair off it, when 6 d = (2j + 1) (max - min) and s = fl32((max -
//     min) / 3) is rounded: then d / s = (j + 1/2) (max - min) / (3 s) sits
//     on the side opposite to the rounding of s, at most 2.5 2^-24 away
//     (only j = 1 occurs: at j = 0, 2 the same d makes (max - min) / 3 exact).
// Each group's decision therefore evaluates P' = a d^2 + b d + c (two
// multiply-adds) and rounds P' to the nearest integer:
//   * s == (max - min) / 3 exactly, or float16 parameters (whose ties do not
//     come from the rounding of s): P' = P - kappa (P - 1)(P - 2), which moves
//     0.5 and 2.5 down by 3 kappa / 4 and 1.5 up by kappa / 4 (2.6 times the
//     evaluation error there) and everything else by at most 2 kappa;
//   * s rounded up / down: P' = P (1 -+ lambda), which moves the near-ties at
//     1.5 to their side by 1.5 lambda (more than the evaluation error plus
//     their distance from the tie) and everything else by at most 3 lambda.
// Quotients that are neither ties nor near-ties but lie within 2 kappa of a
// boundary can still round to the wrong side; on the benchmark values that
// is 1 value code in 1.4e8 (CPU emulation), inside the boundary window.
constexpr float kTieKappa = 0x1p-18f;
constexpr float kTieLambda = 0x1p-20f;

// Coefficients (a, b, c) of a value group's decision polynomial from its
// range max - min (exact), stored scale s and r = 1/s (0 when s == 0: every
// code is then 0).  sign_from_range: the stored s is the float32 (max - min)
// / 3, whose rounding direction is the sign of 3 s - (max - min), exact as
// one multiply-add.
__device__ __forceinline__ float3 value_coefficients(float range, float s, float r, bool sign_from_range) {
  int sg = 0;
  if (sign_from_range) {
    const float e = __fmaf_rn(3.0f, s, -range);
    sg = (e > 0.0f) - (e < 0.0f);
  }
  if (sg == 0)
    return make_float3(__fmul_rn(__fmul_rn(r, r), -kTieKappa), __fmul_rn(r, 1.0f + 3.0f * kTieKappa),
                       -2.0f * kTieKappa);
  return make_float3(0.0f, __fmul_rn(r, sg > 0 ? 1.0f - kTieLambda : 1.0f + kTieLambda), 0.0f);
}

// Value decisions of a pair: the float bits of fl32(P') + 1.5 * 2^23, i.e.
// 0x4B400000 + code.  For float32 parameters P' lies in [-2 kappa, 3 (1 +
// 2 lambda)], so the code is the low byte without a clamp.  The magic add
// cannot merge with the multiply-add before it.
__device__ __forceinline__ uint2 value_code_bits2(float2 d, float2 a, float2 b, float2 c) {
  const float2 u = __ffma2_rn(a, d, b);
  const float2 p = __ffma2_rn(u, d, c);
  const float2 y = __fadd2_rn(p, make_float2(kMagic, kMagic));
  return make_uint2(__float_as_uint(y.x), __float_as_uint(y.y));
}

// Key decisions of a pair, one rounding each: the float bits of
// fl32(fl32(x - z) * inv + 1.5 * 2^23) = 0x4B400000 + code (see above).
__device__ __forceinline__ uint2 code_bits2_fma(float2 x, float2 inv, float2 negz) {
  const float2 d = __fadd2_rn(x, negz);
  const float2 c = __ffma2_rn(d, inv, make_float2(kMagic, kMagic));
  return make_uint2(__float_as_uint(c.x), __float_as_uint(c.y));
}

// Code 0..3 from the float bits of a decision, clamped: in the float16
// metadata layout the rounded zero and scale can move a value by up to
// |z| 2^-12 / s outside [0, 3] (the method's rule clamps).
__device__ __forceinline__ uint32_t clamped_code(uint32_t bits) {
  const int c = (int)(bits - kMagicBits);
  return (uint32_t)min(max(c, 0), 3);
}

// The float16 that the 16-bit metadata layout stores for x (nearest even).
__device__ __forceinline__ float to_half_value(float x) { return __half2float(__float2half_rn(x)); }

// Byte offset of value-code row q (channels 4q .. 4q + 3, code of channel
// 4q + i in bits 2i, 2i + 1 of each byte): rows of the upper 64 channels are
// shifted by 16 bytes so that the two threads of a token (one per channel
// half) store into different banks.
__device__ __forceinline__ int vb_row(int q) { return q * kVbStride + ((q >> 4) << 4); }

// Position of token/col c inside its 16-byte packing chunk of the byte
// staging area: chunk (tig, j), byte ((kk * 4) + hf + 2 e).
__device__ __forceinline__ int vb_perm(int c) {
  const int ks = c >> 4, j = ks >> 2, kk = ks & 3, hf = (c >> 3) & 1, tig = (c >> 1) & 3, e = c & 1;
  return ((tig * 2 + j) * 4 + kk) * 4 + hf + 2 * e;
}

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Mixed-precision adds and multiply-adds (sm_100 and later) take a bf16
// operand, widen it exactly and round the float32 result once.
// (lo + hi, lo - hi) of the two bf16 values of a word: the first Hadamard
// stage straight from the packed input.
__device__ __forceinline__ float2 bf16_pair_butterfly(uint32_t u) {
  float s, d;
  asm("{\n\t.reg .b16 lo, hi, m1;\n\t.reg .f32 lf;\n\tmov.b32 {lo, hi}, %2;\n\tmov.b16 m1, 0xBF80;\n\t"
      "add.rn.f32.bf16 lf, lo, 0f80000000;\n\t"    // -0 + lo: lo widened
      "add.rn.f32.bf16 %0, hi, lf;\n\t"
      "fma.rn.f32.bf16 %1, hi, m1, lf;\n\t}"       // lo - hi
      : "=f"(s), "=f"(d)
      : "r"(u));
  return make_float2(s, d);
}
// (lo + c, hi + c) of the two bf16 values of a word.
__device__ __forceinline__ float2 bf16x2_add(uint32_t u, float c) {
  float a, b;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, lo, %3;\n\t"
      "add.rn.f32.bf16 %1, hi, %3;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(u), "f"(c));
  return make_float2(a, b);
}

// Three-input float32 minimum / maximum (one instruction on sm_100 and later)
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float4 fmin3(float4 a, float4 b, float4 c) {
  return make_float4(fmin3(a.x, b.x, c.x), fmin3(a.y, b.y, c.y), fmin3(a.z, b.z, c.z), fmin3(a.w, b.w, c.w));
}
__device__ __forceinline__ float4 fmax3(float4 a, float4 b, float4 c) {
  return make_float4(fmax3(a.x, b.x, c.x), fmax3(a.y, b.y, c.y), fmax3(a.z, b.z, c.z), fmax3(a.w, b.w, c.w));
}

// a * m + c on the integer multiply-add path (m is opaque to the compiler, so
// the packing below stays off the shift / logic pipe)
__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
  return d;
}

// 32 bytes from global memory (32-byte aligned p), read once: each load of
// the pair's two threads fills whole 32-byte sectors.
__device__ __forceinline__ void ld_row32(const void* p, uint4& lo, uint4& hi) {
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
      : "l"(p));
}

// Sum of (0x4B400000 << shift) over the shifts of one key-code word
// (16 e + 4 kk + 2 hf), modulo 2^32: the float bits' constant part,
// subtracted once per word.
__host__ __device__ constexpr uint32_t key_word_magic() {
  uint32_t m = 0;
  for (int kk = 0; kk < 4; ++kk)
    for (int hf = 0; hf < 2; ++hf)
      for (int e = 0; e < 2; ++e) m += kMagicBits << (16 * e + 4 * kk + 2 * hf);
  return m;
}

template <int CAP, bool M16>
__global__ void __launch_bounds__(kQThreads, 2)
    quantize_append_kernel(const __grid_constant__ QuantPlan<CAP> plan, uint8_t* __restrict__ arena,
                           const uint16_t* __restrict__ kin, const uint16_t* __restrict__ vin) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  QuantSmem& S = *reinterpret_cast<QuantSmem*>(smem_raw);
  const int head = blockIdx.y;
  const int tid = threadIdx.x;
  // 1 << 2i for the packing multiply-adds; the zero term keeps them opaque
  const uint32_t zero = (uint32_t)tid >> 31;
  const uint32_t p4 = 4u | zero, p16 = 16u | zero, p64 = 64u | zero;
  const PackedTask T = plan.t[blockIdx.x];
  const int hkv = plan.hkv;
  const int64_t sh = (int64_t)T.slot() * hkv + head;
  uint8_t* win = arena + plan.windows_off + sh * kWindowBytes;
  uint16_t* win_k = reinterpret_cast<uint16_t*>(win);
  uint16_t* win_v = win_k + kGroup * kHeadDim;

  if (T.kind() == 0) {
    using B = Blk<M16>;
    uint8_t* blk = arena + plan.blocks_off + (sh * plan.max_groups + T.group()) * (int64_t)B::kBytes;
    const int t = tid >> 1;          // token of the group
    const int half = tid & 1;        // channels [64 half, 64 half + 64)
    const bool from_win = t < T.n_win();
    const int64_t row = (int64_t)T.in_row() + (t - T.n_win());
    const uint16_t* ksrc = (from_win ? win_k + t * kHeadDim : kin + (row * hkv + head) * kHeadDim) + 64 * half;
    const uint16_t* vsrc = (from_win ? win_v + t * kHeadDim : vin + (row * hkv + head) * kHeadDim) + 64 * half;

    // this thread's half key row (64 bf16), in flight while the values are
    // processed; thread 1 of the pair holds its two 32-channel halves swapped
    uint4 kr[8];
    {
      const uint4* ks4 = reinterpret_cast<const uint4*>(ksrc);
      if (plan.wide) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ld_row32(ks4 + 2 * (i ^ (2 * half)), kr[2 * i], kr[2 * i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) kr[i] = __ldg(ks4 + (i ^ (4 * half)));
      }
    }

    // ---- values: per-token INT2 over this thread's two 32-channel groups
    float smax = 0.0f, zabs = 0.0f;   // largest value scale and |value zero| of this thread's groups
    {
      uint4 vr[8];
      const uint4* vs4 = reinterpret_cast<const uint4*>(vsrc);
      if (plan.wide) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ld_row32(vs4 + 2 * i, vr[2 * i], vr[2 * i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) vr[i] = __ldg(vs4 + i);
      }
      const int pt = vb_perm(t);
      float sv[2], zv[2];
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
        const uint4* w4 = vr + 4 * g2;
        uint32_t mn2 = w4[0].x, mx2 = w4[0].x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t ws[4] = {w4[i].x, w4[i].y, w4[i].z, w4[i].w};
#pragma unroll
          for (int e = (i == 0 ? 1 : 0); e < 4; ++e) {
            mn2 = bf16x2_min(mn2, ws[e]);
            mx2 = bf16x2_max(mx2, ws[e]);
          }
        }
        const float mn = fminf(bf16_lo(mn2), bf16_hi(mn2));
        const float mx = fmaxf(bf16_lo(mx2), bf16_hi(mx2));
        float sc = (mx - mn) / 3.0f;
        float zq = mn;
        if constexpr (M16) {     // decide against the stored (rounded) parameters
          sc = to_half_value(sc);
          zq = to_half_value(mn);
        }
        const float inv = sc > 0.0f ? 1.0f / sc : 0.0f;
        sv[g2] = sc;
        zv[g2] = zq;
        smax = fmaxf(smax, sc);
        zabs = fmaxf(zabs, fabsf(zq));
        const int gi = 2 * half + g2;
        const float3 co = value_coefficients(mx - mn, sc, inv, !M16);
        const float2 ca = make_float2(co.x, co.x), cb = make_float2(co.y, co.y), cc = make_float2(co.z, co.z);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t ws[4] = {w4[i].x, w4[i].y, w4[i].z, w4[i].w};
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {   // channels gi*32 + 8i + 4qq .. + 3
            const uint2 c01 = value_code_bits2(bf16x2_add(ws[2 * qq], -zq), ca, cb, cc);
            const uint2 c23 = value_code_bits2(bf16x2_add(ws[2 * qq + 1], -zq), ca, cb, cc);
            uint32_t b;
            if constexpr (M16) {
              b = clamped_code(c01.x) | (clamped_code(c01.y) << 2) | (clamped_code(c23.x) << 4) |
                  (clamped_code(c23.y) << 6);
            } else {
              // low byte: the codes (the float bits' constant part has a zero low byte)
              b = imad(c23.y, p64, imad(c23.x, p16, imad(c01.y, p4, c01.x)));
            }
            S.vb[vb_row(gi * 8 + 2 * i + qq) + pt] = (uint8_t)b;
          }
        }
      }
      if constexpr (M16) {   // s[t][0..3] and z[t][0..3], float16 (exact: already rounded)
        *reinterpret_cast<uint32_t*>(blk + B::kVScale + 8 * t + 4 * half) = pack_half2(sv[0], sv[1]);
        *reinterpret_cast<uint32_t*>(blk + B::kVZero + 8 * t + 4 * half) = pack_half2(zv[0], zv[1]);
      } else {
        const int vr = 16 * vmeta_row(t) + 8 * half;
        *reinterpret_cast<float2*>(blk + kOffVScale + vr) = make_float2(sv[0], sv[1]);
        *reinterpret_cast<float2*>(blk + kOffVZero + vr) = make_float2(zv[0], zv[1]);
      }
    }

    // ---- keys: rotation (6 butterfly stages in registers + 1 across the
    // thread pair), norm, unit vector.  x[i] holds channels 64 half + 2 i',
    // + 1 with i' = i (thread 0) or i ^ 16 (thread 1: halves swapped).
    // stage h = 1 (within each pair) as the words are widened
    float2 x[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[4 * i + 0] = bf16_pair_butterfly(kr[i].x);
      x[4 * i + 1] = bf16_pair_butterfly(kr[i].y);
      x[4 * i + 2] = bf16_pair_butterfly(kr[i].z);
      x[4 * i + 3] = bf16_pair_butterfly(kr[i].w);
    }
    // stages h = 2 .. 16: pairs (i, i + h/2) of float2, the same in both layouts
#pragma unroll
    for (int hb = 0; hb < 4; ++hb) {
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int h = 1 << hb;
        const int j = ((n >> hb) << (hb + 1)) | (n & (h - 1));
        const float2 a = x[j], b = x[j + h];
        x[j] = __fadd2_rn(a, b);
        x[j + h] = __fadd2_rn(a, make_float2(-b.x, -b.y));
      }
    }
    // stage h = 32 (pairs (j, j + 16)), in thread 1 with the roles swapped:
    // x[j] = b - a (minus the difference, in the slot of channel c + 32) and
    // x[j + 16] = a + b, so both layouts stay as they are
    const float2 sg = half ? make_float2(-1.0f, -1.0f) : make_float2(1.0f, 1.0f);
    const float2 nsg = make_float2(-sg.x, -sg.y);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 a = x[j], b = x[j + 16];
      x[j] = __ffma2_rn(b, sg, a);
      x[j + 16] = __ffma2_rn(b, nsg, a);
    }
    // stage h = 64 across the thread pair: each thread sends x[16 .. 31] and
    // keeps x[0 .. 15]; the pairs (channel c, c + 64) meet as
    //   thread 0: own a_c (c < 32),       received b_c       -> a + b, a - b
    //   thread 1: own -b_c (c in 32..63), received a_c       -> a + b, a - b
    // after which x[k] holds channels 32 half + 2k, + 1 and x[k + 16]
    // channels 64 + 32 half + 2k, + 1 in both threads.
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float2 own = x[k];
      const float2 rcv = make_float2(__shfl_xor_sync(0xffffffffu, x[k + 16].x, 1),
                                     __shfl_xor_sync(0xffffffffu, x[k + 16].y, 1));
      x[k] = __ffma2_rn(own, sg, rcv);
      x[k + 16] = __ffma2_rn(rcv, nsg, own);
    }
    float* krow = &S.kh[t * kHeadDim];
    float2 sq2 = make_float2(0.0f, 0.0f), sq2b = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      sq2 = __ffma2_rn(x[i], x[i], sq2);
      sq2b = __ffma2_rn(x[i + 1], x[i + 1], sq2b);
    }
    const float sq = (sq2.x + sq2.y) + (sq2b.x + sq2b.y);
    const float ss = sq + __shfl_xor_sync(0xffffffffu, sq, 1);   // the same sum in both threads
    float norm, rinv;
    if (ss >= 0x1p-100f && ss <= 0x1p+100f) {
      norm = sqrtf(ss * (1.0f / kHeadDim));
      rinv = 1.0f / sqrtf(ss);
    } else {
      // a zero token, or squares that under- or overflowed (both threads of
      // the pair): the norm of Hu k from Hu k scaled by 2^-e, exact in two
      // power-of-two steps, with m = max |Hu k| < 2^e
      const unsigned pair = 3u << (tid & 30);
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) m = fmaxf(m, fmaxf(fabsf(x[i].x), fabsf(x[i].y)));
      m = fmaxf(m, __shfl_xor_sync(pair, m, 1));
      int e = 0;
      if (m > 0.0f) frexpf(m, &e);
      const int e1 = -e / 2;
      const float2 f1 = make_float2(ldexpf(1.0f, e1), ldexpf(1.0f, e1));
      const float2 f2 = make_float2(ldexpf(1.0f, -e - e1), ldexpf(1.0f, -e - e1));
      float2 a2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = __fmul2_rn(__fmul2_rn(x[i], f1), f2);
        a2 = __ffma2_rn(x[i], x[i], a2);
      }
      float s2 = a2.x + a2.y;
      s2 += __shfl_xor_sync(pair, s2, 1);
      norm = ldexpf(sqrtf(s2 * (1.0f / kHeadDim)), e);
      rinv = s2 > 0.0f ? 1.0f / sqrtf(s2) : 0.0f;   // k_hat = (Hu k 2^-e) / |Hu k 2^-e|
    }
    // scalar rounded products: the k_hat in registers (code decisions) is the
    // k_hat stored below (parameters), and its packed subtraction in
    // code_bits2 cannot be fused with this multiply
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = make_float2(__fmul_rn(x[i].x, rinv), __fmul_rn(x[i].y, rinv));
    if (half == 0) {
      if constexpr (M16)
        reinterpret_cast<__half*>(blk + B::kKNorm)[t] = __float2half_rn(norm);
      else
        reinterpret_cast<float*>(blk + kOffKNorm)[t] = norm;
    }
    {
      float4* dst = reinterpret_cast<float4*>(krow);
#pragma unroll
      for (int i = 0; i < 16; ++i) {     // float4 column 8 half + i (i < 8) or 8 + 8 half + i
        const int q = (i < 8 ? 8 * half : 8 + 8 * half) + i;
        dst[kh_slot(t, q)] = make_float4(x[2 * i].x, x[2 * i].y, x[2 * i + 1].x, x[2 * i + 1].y);
      }
    }
#pragma unroll
    {   // non-negative floats order as their bit patterns
      const uint32_t sm = __reduce_max_sync(0xffffffffu, __float_as_uint(smax));
      const uint32_t zm = __reduce_max_sync(0xffffffffu, __float_as_uint(zabs));
      if ((tid & 31) == 0) {
        S.red[0][tid >> 5] = sm;
        S.red[1][tid >> 5] = zm;
      }
    }
    __syncthreads();

    // ---- value code words, V order (the staged bytes are complete)
    {
      const int u = tid;
      const int mt = u >> 5, lane = u & 31, g = lane >> 2, tig = lane & 3;
      uint32_t wv[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int rowc = 16 * mt + g + 8 * r;
          const int sh = 2 * (rowc & 3);                 // this channel's bits in each byte
          const uint4 b = *reinterpret_cast<const uint4*>(&S.vb[vb_row(rowc >> 2) + (tig * 2 + j) * 16]);
          const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
          uint32_t w = 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t cw = (bw[kk] >> sh) & 0x03030303u;
            const uint32_t y = (cw | (cw >> 6)) & 0x000F000Fu;
            w |= y << (4 * kk);
          }
          wv[2 * j + r] = w;
        }
      }
      *reinterpret_cast<uint2*>(blk + B::kVCodes + vword_off(mt, 0, lane)) = make_uint2(wv[0], wv[1]);
      *reinterpret_cast<uint2*>(blk + B::kVCodes + vword_off(mt, 1, lane)) = make_uint2(wv[2], wv[3]);
    }

    // ---- per-channel key parameters: 16-token slices of 4 channels, then 8 slices
    {
      const int cq = tid & 31, ts = tid >> 5;
      const float4* rows = reinterpret_cast<const float4*>(&S.kh[(16 * ts) * kHeadDim]);
      const float4 v0 = rows[kh_slot(0, cq)], v1 = rows[(kHeadDim / 4) + kh_slot(1, cq)];
      float4 mn = fmin3(v0, v1, rows[2 * (kHeadDim / 4) + kh_slot(2, cq)]);
      float4 mx = fmax3(v0, v1, rows[2 * (kHeadDim / 4) + kh_slot(2, cq)]);
#pragma unroll
      for (int r = 3; r < 15; r += 2) {    // rows 3 .. 14 in pairs, then row 15
        const float4 a = rows[r * (kHeadDim / 4) + kh_slot(r, cq)];
        const float4 b = rows[(r + 1) * (kHeadDim / 4) + kh_slot(r + 1, cq)];
        mn = fmin3(mn, a, b);
        mx = fmax3(mx, a, b);
      }
      {
        const float4 a = rows[15 * (kHeadDim / 4) + kh_slot(15, cq)];
        mn = make_float4(fminf(mn.x, a.x), fminf(mn.y, a.y), fminf(mn.z, a.z), fminf(mn.w, a.w));
        mx = make_float4(fmaxf(mx.x, a.x), fmaxf(mx.y, a.y), fmaxf(mx.z, a.z), fmaxf(mx.w, a.w));
      }
      S.rmin[ts][cq] = mn;
      S.rmax[ts][cq] = mx;
    }
    __syncthreads();
    if (tid < kHeadDim) {
      const int c = tid;
      const float* rmn = reinterpret_cast<const float*>(S.rmin);
      const float* rmx = reinterpret_cast<const float*>(S.rmax);
      float mn = fminf(rmn[c], rmn[kHeadDim + c]), mx = fmaxf(rmx[c], rmx[kHeadDim + c]);
#pragma unroll
      for (int ts = 2; ts < 8; ts += 2) {
        mn = fmin3(mn, rmn[ts * kHeadDim + c], rmn[(ts + 1) * kHeadDim + c]);
        mx = fmax3(mx, rmx[ts * kHeadDim + c], rmx[(ts + 1) * kHeadDim + c]);
      }
      float sc = (mx - mn) / 3.0f;
      if constexpr (M16) {     // decide against the stored (rounded) parameters
        sc = to_half_value(sc);
        mn = to_half_value(mn);
      }
      float* kqf = reinterpret_cast<float*>(&S.kq[kq_index(c)]);
      kqf[c & 1] = sc > 0.0f ? 1.0f / sc : 0.0f;
      kqf[2 + (c & 1)] = -mn;
      if constexpr (M16) {
        reinterpret_cast<__half*>(blk + B::kKScale)[c] = __float2half_rn(sc);
        reinterpret_cast<__half*>(blk + B::kKZero)[c] = __float2half_rn(mn);
      } else {
        reinterpret_cast<float*>(blk + kOffKScale)[c] = sc;
        reinterpret_cast<float*>(blk + kOffKZero)[c] = mn;
      }
    }
    __syncthreads();

    // ---- key codes of token t: this thread's channels fill half of each of
    // the token's fragment words (j = 0: channels [32 half, + 32), slots kk =
    // 2 half, 2 half + 1; j = 1: channels [64 + 32 half, + 32)); the pair
    // swaps halves so that thread `half` completes the 4 words with j = half
    {
      const int mt = t >> 4, g = t & 7, r = (t >> 3) & 1;
      uint32_t wa[4] = {0u, 0u, 0u, 0u}, wb[4] = {0u, 0u, 0u, 0u};   // j = 0, j = 1, per tig; bits as if half = 0
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int tig = k & 3, hf = (k >> 2) & 1, kkl = k >> 3;
        const int sft = 4 * kkl + 2 * hf;
        const float4 pa = S.kq[kq_index(32 * half + 2 * k)];
        const float4 pb = S.kq[kq_index(64 + 32 * half + 2 * k)];
        const uint2 ca = code_bits2_fma(x[k], make_float2(pa.x, pa.y), make_float2(pa.z, pa.w));
        const uint2 cb = code_bits2_fma(x[k + 16], make_float2(pb.x, pb.y), make_float2(pb.z, pb.w));
        if constexpr (M16) {
          wa[tig] |= (clamped_code(ca.x) << sft) | (clamped_code(ca.y) << (16 + sft));
          wb[tig] |= (clamped_code(cb.x) << sft) | (clamped_code(cb.y) << (16 + sft));
        } else {
          wa[tig] += (ca.x << sft) + (ca.y << (16 + sft));
          wb[tig] += (cb.x << sft) + (cb.y << (16 + sft));
        }
      }
      const int up = 8 * half;   // slots kk = 2, 3 of the words
      uint32_t* kcodes = reinterpret_cast<uint32_t*>(blk + kOffKCodes);
#pragma unroll
      for (int tig = 0; tig < 4; ++tig) {
        const uint32_t keep = (half ? wb[tig] : wa[tig]) << up;
        const uint32_t send = (half ? wa[tig] : wb[tig]) << up;
        const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 1);
        const uint32_t w = M16 ? (keep | got) : (keep + got - key_word_magic());
        kcodes[((mt * 32 + 4 * g + tig) * 4) + 2 * half + r] = w;
      }
    }
    if (tid < 2) {   // the (slot, head)'s largest value scale (decode) and |value zero| (prefill)
      uint32_t m = S.red[tid][0];
#pragma unroll
      for (int i = 1; i < kQThreads / 32; ++i) m = max(m, S.red[tid][i]);
      atomicMax(reinterpret_cast<unsigned int*>(arena + (tid == 0 ? (int64_t)kMetaHeader : plan.zmax_off)) + sh, m);
    }
    if (T.tail_count() <= 0) return;
    // the window reads above completed before the first __syncthreads
  }

  // ---- window append: rows tail_in_row.. -> window slots (tail_pos + i) mod 128
  {
    const int count = T.tail_count();
    for (int idx = tid; idx < count * 16; idx += kQThreads) {
      const int i = idx >> 4, q = idx & 15;
      const int64_t row = (int64_t)T.tail_in_row() + i;
      const int slot = (T.tail_pos_mod() + i) & (kGroup - 1);
      const uint4* ks = reinterpret_cast<const uint4*>(kin + (row * hkv + head) * kHeadDim);
      const uint4* vs = reinterpret_cast<const uint4*>(vin + (row * hkv + head) * kHeadDim);
      reinterpret_cast<uint4*>(win_k + slot * kHeadDim)[q] = __ldg(ks + q);
      reinterpret_cast<uint4*>(win_v + slot * kHeadDim)[q] = __ldg(vs + q);
    }
  }
}

template <int CAP, bool M16>
cudaError_t launch_quantize(const QuantPlan<CAP>& plan, uint8_t* arena, const uint16_t* k, const uint16_t* v,
                            cudaStream_t stream) {
  if (plan.n_tasks <= 0) return cudaSuccess;
  const int smem = (int)sizeof(QuantSmem);
  static bool attr_done[64] = {};
  cudaError_t e = ensure_smem_attr(quantize_append_kernel<CAP, M16>, smem, attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid(plan.n_tasks, plan.hkv);
  quantize_append_kernel<CAP, M16><<<grid, kQThreads, smem, stream>>>(plan, arena, k, v);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_small(const QuantPlan<kQuantPlanSmall>& plan, uint8_t* arena, const uint16_t* k,
                                  const uint16_t* v, bool meta16, cudaStream_t stream) {
  return meta16 ? launch_quantize<kQuantPlanSmall, true>(plan, arena, k, v, stream)
                : launch_quantize<kQuantPlanSmall, false>(plan, arena, k, v, stream);
}

cudaError_t launch_quantize_large(const QuantPlan<kQuantPlanLarge>& plan, uint8_t* arena, const uint16_t* k,
                                  const uint16_t* v, bool meta16, cudaStream_t stream) {
  return meta16 ? launch_quantize<kQuantPlanLarge, true>(plan, arena, k, v, stream)
                : launch_quantize<kQuantPlanLarge, false>(plan, arena, k, v, stream);
}

}  // namespace oscar
