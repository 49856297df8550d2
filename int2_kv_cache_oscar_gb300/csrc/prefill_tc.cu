// Chunked-prefill attention over the packed OScaR cache on the 5th-generation
// tensor cores (sm_103a tcgen05): the queries of a new chunk attend to every
// token already in the cache (its quantised groups and its bf16 window; no
// mask, the cache precedes the chunk), and each output row also gets its
// log-sum-exp.  Scores and outputs follow the decode path (OScaR abstract;
// ai-papers.net "OScaRの提案手法"): s_t = n_t (H_d q) . (code_t s + z) * scale
// for quantised tokens, q . k_t * scale for window tokens, o = softmax(s) .
// v_hat with v_hat = code s^V + z^V.
//
// A CTA takes 128 (query, head) rows of one KV head (M = 128; TMEM lane =
// row) and a range of the history's groups, each group (and the window) as
// two half-steps of 64 tokens; 13 warps:
//   * builders (warps 8-11): expand the packed codes into exact fp16 B
//     operands in shared memory (no-swizzle K-major core matrices), a token
//     half at a time, as soon as the MMA that read that half last is done:
//     scores B[token][channel] = code * S_i(c) and values B[channel][token] =
//     code * S_i^V(t, group), where S_1 + S_2 is the scale split into two
//     9-significant-bit pieces (code * S_i, code <= 3, is exact in fp16);
//     extra B rows carry the key and value zeros (hi + lo fp16).  The window's
//     keys are rotated like the query (H k_t) and split into fp16 hi + lo in
//     the places of the two pieces.  The first builder also streams the group
//     blocks through a ring of bulk copies;
//   * MMA issuer (warp 12): one thread issues every tcgen05.mma;
//   * rows (warps 0-7; warps w and w + 4 share TMEM lanes 32 (w & 3) ..,
//     thread = row, each warp group a 32-token chunk of every half): online
//     softmax over the scores read from TMEM; P (hi + lo) goes to TMEM (two
//     buffers) as the A operand of P.V; the output accumulator stays in TMEM
//     and is rescaled only when a row's maximum grows by more than 8 (log2
//     units; P stays below 2^8).
// Products per half-step (M = 128 rows, K = 16 per MMA; Qhi, P in TMEM, Qlo
// in shared memory):
//   scores  S[0, 144) = Qhi [B1 | zero | B2],  S[0, 80) += Qlo [B1 | zero]
//   values  [O | Z] += Phi [V1 | zero] + Plo [V1 | zero],  O += Phi V2
// dropping only the products of two low parts (relative 2^-20).  Each row
// thread reads S1 + S2 and the zero-term column; Z is the value-zero term
// sum_t p_t z^V(t) per value group.  The scores of half-step j + 1 are
// issued as soon as the rows have read those of j, the P.V of j once they
// have written its P, so the tensor cores work while the rows do.  The window
// comes last; its P.V is on bf16 operands (V exact; P as bf16 hi + lo).  With
// a workspace the history is split into parts (grid.z), each writing per-row
// records (o unnormalised, m, l) that the merge kernel combines.
#include <cstddef>

#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int kTcRows = 128;
constexpr int kTcThreads = 13 * 32;
constexpr int kTcStages = 3;
constexpr int kN1 = 80;                  // key piece-1 rows of a token half: 64 tokens + 16 zero rows
constexpr int kNK = kN1 + 64;            // key B rows of a token half: then the 64 tokens' piece 2
constexpr int kKBytes = kNK * kHeadDim * 2;
constexpr int kNV1 = kHeadDim + 16;      // value B rows of piece 1: 128 channels + the zero rows
constexpr int kV1Bytes = kNV1 * kGroup * 2;
constexpr int kVBytes = kHeadDim * kGroup * 2;       // value B piece 2: 128 channel rows x 128 tokens
constexpr uint32_t kLboK = (kNK / 8) * 128;          // B: core matrices adjacent along K
constexpr uint32_t kLboV1 = (kNV1 / 8) * 128;
constexpr uint32_t kLboV = (kHeadDim / 8) * 128;
constexpr uint32_t kSbo = 128;                       // core matrices adjacent along M / N
// TMEM columns (512 allocated)
constexpr uint32_t kTQ = 0;        // rotated q * 2^F: hi fp16 pairs [0, 64) (lo in shared memory)
constexpr uint32_t kTS = 64;       // scores of one half-step [64, 208): piece 1 (+ zero term) [0, 80), piece 2 [80, 144)
constexpr uint32_t kTP = 208;      // P of half-steps j (buffer j & 1): [208, 272), [272, 336)
constexpr uint32_t kTO = 336;      // output accumulator [336, 464), then the value-zero sums [464, 480)
constexpr uint32_t kTZ = kTO + kHeadDim;
constexpr uint32_t kTCols = 512;
constexpr float kRescaleLog2 = 8.0f;

// TMEM column of the P pairs of k-step ks of a half (tokens 16 ks .. + 15)
// in P buffer pb, hi or lo: each 32-token chunk c becomes [hi of its two
// k-steps | lo of its two k-steps] in the chunk's own 32 columns.
__host__ __device__ constexpr uint32_t p_col(int pb, int ks, bool lo) {
  return kTP + 64 * pb + 32 * (ks >> 1) + (lo ? 16 : 0) + 8 * (ks & 1);
}

struct TcSmem {
  alignas(1024) uint8_t kb[2][kKBytes];               // key B of token half h
  alignas(1024) uint8_t v1[kV1Bytes];                 // value B piece 1 (+ zero rows)
  alignas(1024) uint8_t v2[kVBytes];                  // value B piece 2
  alignas(1024) uint8_t qlo[kTcRows * kHeadDim * 2];  // A: the rows' rotated q * 2^F, fp16 lo part
  alignas(128) uint8_t stage[kTcStages][kBlockBytes];
  // key norms per step, three deep: the keys of step k + 1 are built while
  // the rows may still be on step k - 1's second half
  float nrm[3][kGroup];
  alignas(16) uint16_t s1[kHeadDim], s2[kHeadDim];    // key-scale pieces (fp16) per channel
  alignas(16) uint16_t w1[kVGroups][kGroup], w2[kVGroups][kGroup];   // value-scale pieces [group][token]
  float wmax[4];                                      // per builder warp: max |k| (window), |z^V| (groups)
  int fw;                                             // the window keys carry 2^fw
  int gz;                                             // the value-zero rows carry 2^gz
  float fexp[kTcRows];                                // 2^-(F_row + 2) * scale_log2
  float pmax[2][2][kTcRows];                          // row maxima of the two token chunks (by half-step parity)
  float lpart[kTcRows];                               // the second warp group's sum of p
  alignas(8) uint64_t full[kTcStages];
  uint64_t sdone[2], odone[2];   // scores / P.V of token half h done (one phase per step)
  // counts, monotonic (a waiter may fall a phase behind): key / value halves
  // built (2 k + h + 1), row warps done reading the scores / writing P (8 per half-step)
  uint32_t kready, vready, sread, pcount;
  uint32_t nissued[kTcStages];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(TcSmem) + 1024 <= 232448, "one CTA per SM");
static_assert(offsetof(TcSmem, stage) % 128 == 0 && offsetof(TcSmem, full) % 8 == 0, "alignment");
static_assert(offsetof(TcSmem, v2) == offsetof(TcSmem, v1) + kV1Bytes && kV1Bytes + kVBytes >= kTcRows * kHeadDim * 4,
              "q staging fits in the value buffers");

// Bounded wait that backs off: a few immediate polls, then short sleeps, so
// that waiting warps leave issue slots and shared-memory bandwidth to the
// working ones (every role here waits for microseconds at a time).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* err) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (i >= 4) __nanosleep(i < 64 ? 32 : 128);
  }
  *abort_flag = 1;
  if (err != nullptr) atomicOr(err, kErrTimeout);
  return false;
}

// Bounded wait until a count published by another role exceeds n (then the
// writes before the count are visible), with the same back-off.
__device__ __forceinline__ bool tc_wait_count(const uint32_t* cnt, uint32_t n, volatile int* abort_flag,
                                              uint32_t* err) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (*reinterpret_cast<const volatile uint32_t*>(cnt) > n) {
      __threadfence_block();
      return true;
    }
    if (*abort_flag) return false;
    if (i >= 4) __nanosleep(i < 64 ? 32 : 128);
  }
  *abort_flag = 1;
  if (err != nullptr) atomicOr(err, kErrTimeout);
  return false;
}

// Publish count n (after this thread's barrier with the writers).
__device__ __forceinline__ void publish(uint32_t* cnt, uint32_t n) {
  __threadfence_block();
  *reinterpret_cast<volatile uint32_t*>(cnt) = n;
}

__device__ __forceinline__ float tc_pow2(int e) {
  e = max(-126, min(127, e));
  return __uint_as_float((uint32_t)(127 + e) << 23);
}

__device__ __forceinline__ float tc_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of element (row, k) of a no-swizzle K-major operand with
// `rows` rows: core matrix (row / 8, k / 8) of 8 rows x 16 bytes at
// ((k / 8) * (rows / 8) + row / 8) * 128.
__device__ __forceinline__ int canon(int row, int k, int rows) {
  return ((k >> 3) * (rows >> 3) + (row >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

// Shared-memory matrix descriptor (tcgen05): start, leading (K) and stride
// (M / N) byte offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B fp16 (bf16 when
// bf16 is set), both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_f16(int n, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(kTcRows >> 4) << 24);
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
               :: "r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)acc) : "memory");
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc) : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tfence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tfence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void async_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                 "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                 "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}

__device__ __forceinline__ void tld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}

__device__ __forceinline__ void tst16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                  "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
               : "memory");
}

__device__ __forceinline__ void tld2(uint32_t taddr, uint32_t (&r)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
}

__device__ __forceinline__ void tst32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
               "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                  "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
                  "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
                  "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
               : "memory");
}

// Named barrier counted per thread (the builders' first thread leaves its
// warp's path while it waits to issue the value products).
__device__ __forceinline__ void bar_sync_threads(int id, int n) {
  asm volatile("barrier.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void tld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tst_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// x rounded to 9 significant bits (nearest, ties away), as a float.
__device__ __forceinline__ float round9(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7f800000u) == 0u) return 0.0f;   // zero and float32 subnormals: below every fp16 piece
  u = (u + 0x4000u) & ~0x7fffu;
  return __uint_as_float(u);
}

// The two fp16 pieces of x (x = S1 + S2 up to 2^-19 relative; each piece has
// at most 9 significant bits, so code * piece is exact in fp16).
__device__ __forceinline__ void pieces(float x, uint16_t& h1, uint16_t& h2) {
  const float a = round9(x);
  const float b = round9(x - a);
  h1 = __half_as_ushort(__float2half_rn(a));
  h2 = __half_as_ushort(__float2half_rn(b));
}

// fp16 codes of a pair: the two 2-bit fields at bit s and 16 + s of w, as
// exact fp16 integers 0..3.
__device__ __forceinline__ __half2 code_pair(uint32_t w, int s) {
  const uint32_t x = ((w >> s) & 0x00030003u) | 0x64006400u;   // 1024 + code
  return __hsub2(*reinterpret_cast<const __half2*>(&x), __floats2half2_rn(1024.0f, 1024.0f));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// hi + lo fp16 (or bf16) of a pair of floats.
__device__ __forceinline__ void split2(float x0, float x1, bool bf16, uint32_t& hi, uint32_t& lo) {
  if (bf16) {
    const uint32_t h0 = f32_to_bf16_bits(x0), h1 = f32_to_bf16_bits(x1);
    hi = h0 | (h1 << 16);
    lo = f32_to_bf16_bits(x0 - __uint_as_float(h0 << 16)) | (f32_to_bf16_bits(x1 - __uint_as_float(h1 << 16)) << 16);
  } else {
    hi = pack_half2(x0, x1);
    lo = pack_half2(x0 - half_lo_to_float(hi), x1 - half_hi_to_float(hi));
  }
}

// hi + lo of a pair of P values (x0 in the low half) for the A operand of
// P.V: hi is x with its mantissa cut to the target width (exact in fp16 for
// x >= 2^-14, and in bf16), lo = x - hi (exact in float), each pair converted
// with one packed cvt.
__device__ __forceinline__ void split_p(float x0, float x1, bool bf16, uint32_t& hi, uint32_t& lo) {
  const uint32_t m = bf16 ? 0xFFFF0000u : 0xFFFFE000u;
  const float h0 = __uint_as_float(__float_as_uint(x0) & m), h1 = __uint_as_float(__float_as_uint(x1) & m);
  const float r0 = x0 - h0, r1 = x1 - h1;
  if (bf16) {
    hi = (__float_as_uint(h0) >> 16) | (__float_as_uint(h1) & 0xFFFF0000u);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(r1), "f"(r0));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(h1), "f"(h0));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(r1), "f"(r0));
  }
}

// fp16 hi + lo of a pair of P values (x0 in the low half): hi rounded to
// nearest, lo the remainder x - hi (exact in float: one mixed-precision
// multiply-add per value with the fp16 hi taken in place) rounded to fp16.
__device__ __forceinline__ void split_p16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(x1), "f"(x0));
  float r0, r1;
  asm("{\n\t.reg .b16 l, h, m1;\n\tmov.b32 {l, h}, %2;\n\tmov.b16 m1, 0xBC00;\n\t"
      "fma.rn.f32.f16 %0, l, m1, %3;\n\tfma.rn.f32.f16 %1, h, m1, %4;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "r"(hi), "f"(x0), "f"(x1));
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(r1), "f"(r0));
}

// Normalised Walsh-Hadamard transform of a 128-vector held by one warp (lane
// = elements 4 lane .. + 3): two stages in registers, five across lanes.
__device__ __forceinline__ void fwht128_warp(float (&v)[4], int lane) {
  const float a = v[0] + v[1], bq = v[0] - v[1], c = v[2] + v[3], d = v[2] - v[3];
  v[0] = a + c;
  v[2] = a - c;
  v[1] = bq + d;
  v[3] = bq - d;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, v[i], o);
      v[i] = upper ? other - v[i] : v[i] + other;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] *= 0.088388347648318440550f;   // 1/sqrt(128)
}

template <bool M16>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p, const uint8_t* __restrict__ arena) {
  using B = Blk<M16>;
  using MR = Meta<M16>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the dynamic window (descriptors address 16-byte units)
  TcSmem& S = *reinterpret_cast<TcSmem*>(smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.y;                 // KV head
  const int part = blockIdx.z;
  const int g_begin = (int)(((int64_t)part * p.ng) / p.n_parts);
  const int g_end = (int)(((int64_t)(part + 1) * p.ng) / p.n_parts);
  const int ng = g_end - g_begin;
  const int wlen = part == p.n_parts - 1 ? p.wlen : 0;
  const int nsteps = ng + (wlen > 0 ? 1 : 0);   // the window is the last step
  const int nh = 2 * nsteps;                    // half-steps
  const uint8_t* blocks = arena + p.blocks_off +
                          (((int64_t)p.slot * p.hkv + j) * p.max_groups + g_begin) * (int64_t)B::kBytes;
  const float vmax = __uint_as_float(
      reinterpret_cast<const uint32_t*>(arena + kMetaHeader)[(int64_t)p.slot * p.hkv + j]);
  int Gv;   // value pieces carry 2^Gv: 3 vmax 2^Gv <= 8
  {
    int e = 0;
    if (vmax > 0.0f) frexpf(3.0f * vmax, &e);
    Gv = vmax > 0.0f ? min(3 - e, 64) : 0;
  }

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&S.full[s], 1);
      S.nissued[s] = 0;
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&S.sdone[h], 1);
      mbar_init(&S.odone[h], 1);
    }
    S.kready = 0;
    S.vready = 0;
    S.sread = 0;
    S.pcount = 0;
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(smem_u32(&S.tmem_base)),
                 "r"(kTCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // ---- q rows: rotate (warp-cooperative FWHT, lanes = 4 channels) into the
  // staging area, then each row thread stores its row into TMEM
  float* qst = reinterpret_cast<float*>(S.v1);                    // [128][128] rotated q * 2^F (v1, v2)
  for (int r = warp; r < kTcRows; r += kTcThreads / 32) {
    const int row = blockIdx.x * kTcRows + r;
    uint2 raw = make_uint2(0u, 0u);
    if (row < p.rows) {
      const int qi = row / p.gqa, h = j * p.gqa + row % p.gqa;
      raw = *reinterpret_cast<const uint2*>(p.q + ((int64_t)qi * p.hq + h) * kHeadDim + 4 * lane);
    }
    float qv[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    fwht128_warp(qv, lane);
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fabsf(qv[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int F = 0;
    if (mx > 0.0f) {
      int e;
      frexpf(mx, &e);   // mx < 2^e
      F = 15 - e;
    }
    const float f = tc_pow2(F);
    *reinterpret_cast<float4*>(qst + r * kHeadDim + 4 * lane) = make_float4(qv[0] * f, qv[1] * f, qv[2] * f, qv[3] * f);
    if (lane == 0) S.fexp[r] = tc_pow2(-(F + 2)) * p.scale_log2;
  }
  tfence_before();
  __syncthreads();
  tfence_after();
  const uint32_t tmem = S.tmem_base;
  if (warp < 4) {
    // row thread r stores its hi fp16 pairs into its lane, the lo pairs
    // into the shared-memory A operand (no-swizzle K-major, row r)
    const int r = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t hi[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        uint32_t lo[4];   // channels 2 (c0 + i) .. + 7: one 16-byte row of a core matrix
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = qst[r * kHeadDim + 2 * (c0 + i + e)], x1 = qst[r * kHeadDim + 2 * (c0 + i + e) + 1];
          split2(x0, x1, false, hi[i + e], lo[e]);
        }
        *reinterpret_cast<uint4*>(S.qlo + canon(r, 2 * (c0 + i), kTcRows)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      tst32(lane_base + kTQ + c0, hi);
    }
    tst_wait();
    async_fence();   // the lo part is read by the tensor cores
  }
  tfence_before();
  __syncthreads();   // the staging area is free again
  tfence_after();

  if (warp == 12) {
    // ============================================================ MMA issuer
    // One thread issues every tcgen05.mma: the scores of half-step j + 1 as
    // soon as the rows have read those of j (one score buffer), the P.V of j
    // once they have written its P.  An issue blocks while the MMA queue is
    // full, so this thread does nothing else.
    if (lane == 0) {
      // every operand address is fixed: descriptors and TMEM columns are set
      // up once, and each half-step's MMAs are one unrolled sequence (an MMA
      // issue stalls this thread for its own latency, so nothing else sits
      // between them)
      const uint32_t idK = idesc_f16(kNK, false), idK1 = idesc_f16(kN1, false);
      const uint32_t idO = idesc_f16(kHeadDim, false), idOZ = idesc_f16(kNV1, false), idOW = idesc_f16(kHeadDim, true);
      const uint64_t dK0 = sdesc(smem_u32(S.kb[0]), kLboK, kSbo), dK1 = sdesc(smem_u32(S.kb[1]), kLboK, kSbo);
      const uint64_t dQ = sdesc(smem_u32(S.qlo), (kTcRows / 8) * 128, kSbo);   // Qlo: A, 128 rows
      const uint64_t dV1 = sdesc(smem_u32(S.v1), kLboV1, kSbo), dV2 = sdesc(smem_u32(S.v2), kLboV, kSbo);
      const uint32_t tS = tmem + kTS, tO = tmem + kTO, tQ = tmem + kTQ;
      uint32_t n_sd[2] = {0u, 0u}, n_od[2] = {0u, 0u};   // commits issued to each barrier
      // scores of half-step j: S[0, 144) = Qhi . [B1 | zero | B2] (Qhi from
      // TMEM), S[0, 80) += Qlo . [B1 | zero] (Qlo from shared memory); the
      // window's B1 + B2 are H k_t 2^fw as fp16 hi + lo
      auto issue_scores = [&](int jj) {
        const int h = jj & 1;
        if (!tc_wait_count(&S.kready, (uint32_t)jj, &S.abort_flag, p.err_word)) return false;
        tfence_after();
        const uint64_t dk = h ? dK1 : dK0;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          mma_ts(tS, tQ + 8 * ks, dk + (uint64_t)((2 * ks * kLboK) >> 4), idK, ks > 0);
          mma_ss(tS, dQ + (uint64_t)((2 * ks * (kTcRows / 8) * 128) >> 4), dk + (uint64_t)((2 * ks * kLboK) >> 4), idK1,
                 true);
        }
        mma_commit(&S.sdone[h]);
        ++n_sd[h];
        return true;
      };
      // P.V of half-step j (its 64 tokens are the K dimension):
      // [O | Z] += Phi V1 + Plo V1 (N = 144: the zero rows give Z), O += Phi V2
      // (window: O += (Phi + Plo) V, bf16, N = 128)
      auto issue_pv = [&](int jj) {
        const int h = jj & 1;
        if (!tc_wait_count(&S.vready, (uint32_t)jj, &S.abort_flag, p.err_word)) return false;
        tfence_after();
        const uint32_t tP = tmem + p_col(jj & 1, 0, false);
        const uint64_t v1 = dV1 + (uint64_t)((8 * h * kLboV1) >> 4), v2 = dV2 + (uint64_t)((8 * h * kLboV) >> 4);
        const bool first = jj == 0;
        if ((jj >> 1) == ng) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t ah = tP + 32 * (ks >> 1) + 8 * (ks & 1);
            const uint64_t ko = (uint64_t)((2 * ks * kLboV1) >> 4);
            mma_ts(tO, ah, v1 + ko, idOW, !first || ks > 0);
            mma_ts(tO, ah + 16, v1 + ko, idOW, true);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t ah = tP + 32 * (ks >> 1) + 8 * (ks & 1);
            const uint64_t ko1 = (uint64_t)((2 * ks * kLboV1) >> 4), ko2 = (uint64_t)((2 * ks * kLboV) >> 4);
            mma_ts(tO, ah, v1 + ko1, idOZ, !first || ks > 0);
            mma_ts(tO, ah + 16, v1 + ko1, idOZ, true);
            mma_ts(tO, ah, v2 + ko2, idO, true);
          }
        }
        mma_commit(&S.odone[h]);
        ++n_od[h];
        return true;
      };
      bool ok = nh == 0 || issue_scores(0);
      for (int jj = 0; jj < nh && ok; ++jj) {
        if (jj + 1 < nh) {
          ok = tc_wait_count(&S.sread, (uint32_t)(8 * jj + 7), &S.abort_flag, p.err_word);   // all 8 row warps
          if (!ok) break;
          tfence_after();
          ok = issue_scores(jj + 1);
          if (!ok) break;
        }
        ok = tc_wait_count(&S.pcount, (uint32_t)(8 * jj + 7), &S.abort_flag, p.err_word);
        if (!ok) break;
        tfence_after();
        ok = issue_pv(jj);
      }
      // before TMEM is freed: the last committed MMAs have completed (bounded,
      // whatever the abort state: MMAs always complete)
      for (int q = 0; q < 4; ++q) {
        const uint32_t n = q < 2 ? n_sd[q] : n_od[q - 2];
        if (n == 0) continue;
        uint64_t* bar = q < 2 ? &S.sdone[q] : &S.odone[q - 2];
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(bar, (n - 1) & 1)) break;
      }
    }
  } else if (warp >= 8) {
    // =============================================================== builders
    // The operands are built in token halves, each as soon as the MMA that
    // last read that half is done, in the order keys(k, 0), values(k - 1, 1),
    // keys(k, 1), values(k, 0): a half-step of the rows then overlaps one key
    // half and one value half, each needed a half-step later.  Every builder
    // runs the same barriers in every task; after a wait gives up (abort) the
    // work is skipped but the control flow stays the same.
    const int b = tid - 256;     // channel (scale pieces, value codes) or token (value pieces)
    const int bt = b & 63, bh = b >> 6;   // token of a half, channel half (key codes, the window)
    const int bw = warp - 8;
    const float gv = tc_pow2(Gv);
    const bool lead = b == 0;    // also streams the group blocks
    const uint8_t* wsrc = arena + p.windows_off + ((int64_t)p.slot * p.hkv + j) * kWindowBytes;
    bool ok = true;
    // rows no build writes: key rows 66..79 of each half (64 and 65 carry the
    // zero), value rows 136..143 (128 + gr and 132 + gr carry the zeros)
    for (int i = b; i < 2 * 14 * 16; i += 128) {
      const int h = i / (14 * 16), rr = 66 + (i % (14 * 16)) / 16, kb = i % 16;
      *reinterpret_cast<uint4*>(S.kb[h] + canon(rr, 8 * kb, kNK)) = make_uint4(0u, 0u, 0u, 0u);
    }
    *reinterpret_cast<uint4*>(S.v1 + canon(136 + (b >> 4), 8 * (b & 15), kNV1)) = make_uint4(0u, 0u, 0u, 0u);
    if (lead) {
      for (int k = 0; k < ng && k < kTcStages; ++k) {
        mbar_arrive_expect_tx(&S.full[k], B::kBytes);
        bulk_g2s(S.stage[k], blocks + (int64_t)k * B::kBytes, B::kBytes, &S.full[k]);
        S.nissued[k] = 1;
      }
    }
    // 2^gz with max |z^V| 2^gz < 2^14 over the sequence's groups (the
    // quantiser records each (slot, head)'s largest |value zero|): the zero
    // sums accumulate across groups in these units
    int gz = 0;
    {
      const float zm = __uint_as_float(
          reinterpret_cast<const uint32_t*>(arena + p.zmax_off)[(int64_t)p.slot * p.hkv + j]);
      if (zm > 0.0f && zm <= 3.0e38f) {
        int e;
        frexpf(zm, &e);   // zm < 2^e
        gz = max(-100, min(14 - e, 100));
      }
      if (lead) S.gz = gz;   // read by the rows after their last half-step
    }
    const float gzf = tc_pow2(gz);
    uint32_t zk = 0u;            // key zero of channel b (x 4): fp16 hi | lo << 16
    int fw = 0;                  // the window keys carry 2^fw
    // ---- key operands of half h of step k, once the scores that read them last are done
    auto keys = [&](int k, int h) {
      const bool win = k == ng;
      const uint8_t* blk = S.stage[k % kTcStages];
      if (h == 0) ok = ok && (win || tc_wait(&S.full[k % kTcStages], (uint32_t)((k / kTcStages) & 1), &S.abort_flag, p.err_word));
      ok = ok && (k == 0 || tc_wait(&S.sdone[h], (uint32_t)((k - 1) & 1), &S.abort_flag, p.err_word));
      uint8_t* kbh = S.kb[h];
      const int t = 64 * h + bt;
      if (win) {
        if (h == 0) {
          // 2^fw with max |H k| 2^fw < 2^14 over the window (|H k|_inf <=
          // sqrt(128) max |k|), so that the rotated keys' fp16 pieces stay finite
          float mx = 0.0f;
          if (ok) {
#pragma unroll 1
            for (int tt = bt; tt < wlen; tt += 64) {
              const uint4* wk = reinterpret_cast<const uint4*>(wsrc + tt * kHeadDim * 2);
#pragma unroll 2
              for (int kb = 8 * bh; kb < 8 * bh + 8; ++kb) {
                const uint4 u = wk[kb];
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  mx = fmaxf(mx, fmaxf(__uint_as_float((w4[e] << 16) & 0x7FFF0000u), __uint_as_float(w4[e] & 0x7FFF0000u)));
              }
            }
          }
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) S.wmax[bw] = mx;
          bar_sync_threads(2, 128);
          mx = fmaxf(fmaxf(S.wmax[0], S.wmax[1]), fmaxf(S.wmax[2], S.wmax[3]));
          fw = 0;
          if (mx > 0.0f && mx <= 3.0e38f) {
            int e;
            frexpf(mx, &e);   // mx < 2^e, |H k| < 2^(e + 4)
            fw = min(10 - e, 100);   // (keys below 2^-90 are zero in fp16 either way)
          }
          if (lead) S.fw = fw;   // read by the rows once the window's scores are done
        }
        if (ok) {
          // the window keys rotated (H k, as the query), x 2^fw, as fp16 hi
          // (row t) + lo (row 80 + t) like a group's two pieces: each warp
          // takes 16 tokens of the half, lane = channels 4 lane .. + 3
          const float f = tc_pow2(fw);
#pragma unroll 1
          for (int i = 0; i < 16; ++i) {
            const int tl = 16 * bw + i, tt = 64 * h + tl;
            const uint2 raw = tt < wlen ? *reinterpret_cast<const uint2*>(wsrc + tt * kHeadDim * 2 + 8 * lane)
                                        : make_uint2(0u, 0u);
            float kv[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
            fwht128_warp(kv, lane);
            uint32_t h01, l01, h23, l23;
            split2(kv[0] * f, kv[1] * f, false, h01, l01);
            split2(kv[2] * f, kv[3] * f, false, h23, l23);
            *reinterpret_cast<uint2*>(kbh + canon(tl, 4 * lane, kNK)) = make_uint2(h01, h23);
            *reinterpret_cast<uint2*>(kbh + canon(kN1 + tl, 4 * lane, kNK)) = make_uint2(l01, l23);
          }
        }
      } else {
        if (h == 0) {
          if (ok) {
            // channel b: scale pieces (x 4), the zero (hi, lo x 4); token b:
            // its norm (read by the rows)
            pieces(MR::one(blk + B::kKScale, b) * 4.0f, S.s1[b], S.s2[b]);
            uint32_t zh, zl;
            split2(MR::one(blk + B::kKZero, b) * 4.0f, 0.0f, false, zh, zl);
            zk = (zh & 0xffffu) | (zl << 16);
            S.nrm[k % 3][b] = MR::one(blk + B::kKNorm, b);
          }
          bar_sync_threads(2, 128);    // the scale pieces are complete
        }
        if (ok) {
          *reinterpret_cast<uint16_t*>(kbh + canon(64, b, kNK)) = (uint16_t)(zk & 0xffffu);
          *reinterpret_cast<uint16_t*>(kbh + canon(65, b, kNK)) = (uint16_t)(zk >> 16);
          // token t, channels 64 bh .. + 63: the code fragment words of that
          // channel half; piece 1 to row bt, piece 2 to row 80 + bt
          const int mt = t >> 4, g = t & 7, r = (t >> 3) & 1;
          uint32_t w[4];
#pragma unroll
          for (int tig = 0; tig < 4; ++tig) {
            const uint2 q2 = *reinterpret_cast<const uint2*>(blk + kOffKCodes + (mt * 32 + 4 * g + tig) * 16 + 8 * bh);
            w[tig] = r ? q2.y : q2.x;
          }
#pragma unroll 2
          for (int kb = 8 * bh; kb < 8 * bh + 8; ++kb) {
            const int kk = (kb >> 1) & 3, hf = kb & 1;
            const uint4 p1 = *reinterpret_cast<const uint4*>(&S.s1[8 * kb]);
            const uint4 p2 = *reinterpret_cast<const uint4*>(&S.s2[8 * kb]);
            const uint32_t pa[4] = {p1.x, p1.y, p1.z, p1.w}, pb[4] = {p2.x, p2.y, p2.z, p2.w};
            uint32_t o1[4], o2[4];
#pragma unroll
            for (int tig = 0; tig < 4; ++tig) {
              const __half2 cd = code_pair(w[tig], 4 * kk + 2 * hf);
              o1[tig] = h2u(__hmul2(cd, u2h(pa[tig])));
              o2[tig] = h2u(__hmul2(cd, u2h(pb[tig])));
            }
            *reinterpret_cast<uint4*>(kbh + canon(bt, 8 * kb, kNK)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            *reinterpret_cast<uint4*>(kbh + canon(kN1 + bt, 8 * kb, kNK)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
          }
        }
      }
      async_fence();
      bar_sync_threads(2, 128);
      if (lead) publish(&S.kready, (uint32_t)(2 * k + h + 1));
    };
    // ---- value operands of half h of step k, once the P.V that read them last is done
    auto values = [&](int k, int h) {
      const bool win = k == ng;
      const uint8_t* blk = S.stage[k % kTcStages];
      if (!win && h == 0 && ok) {
        // token b: its four value scales as pieces (x 2^Gv); only builders read them
        const float4 sv = MR::v4(blk + B::kVScale, b);
        pieces(sv.x * gv, S.w1[0][b], S.w2[0][b]);
        pieces(sv.y * gv, S.w1[1][b], S.w2[1][b]);
        pieces(sv.z * gv, S.w1[2][b], S.w2[2][b]);
        pieces(sv.w * gv, S.w1[3][b], S.w2[3][b]);
      }
      ok = ok && (k == 0 || tc_wait(&S.odone[h], (uint32_t)((k - 1) & 1), &S.abort_flag, p.err_word));
      if (win) {
        if (ok) {
          // the window values transposed into B[channel][token], bf16: token
          // 64 h + bt, channels 64 bh .. + 63
          const int t = 64 * h + bt;
          const uint16_t* vrow = reinterpret_cast<const uint16_t*>(wsrc + kGroup * kHeadDim * 2 + t * kHeadDim * 2);
#pragma unroll 1
          for (int c = 64 * bh; c < 64 * bh + 64; c += 8) {
            const uint4 v8 = t < wlen ? *reinterpret_cast<const uint4*>(vrow + c) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t e4[4] = {v8.x, v8.y, v8.z, v8.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint16_t*>(S.v1 + canon(c + i, t, kNV1)) = (uint16_t)(e4[i >> 1] >> (16 * (i & 1)));
          }
        }
      } else {
        if (ok) {
          // the zero rows of token 64 h + bt (x 2^gz): 128 + gr z hi, 132 + gr z
          // lo, for value groups gr = 2 bh, 2 bh + 1
          const int t = 64 * h + bt;
          const float4 z4 = MR::v4(blk + B::kVZero, t);
          uint32_t zh0, zl0, zh1, zl1;
          split2((bh ? z4.z : z4.x) * gzf, 0.0f, false, zh0, zl0);
          split2((bh ? z4.w : z4.y) * gzf, 0.0f, false, zh1, zl1);
          *reinterpret_cast<uint16_t*>(S.v1 + canon(128 + 2 * bh, t, kNV1)) = (uint16_t)(zh0 & 0xffffu);
          *reinterpret_cast<uint16_t*>(S.v1 + canon(129 + 2 * bh, t, kNV1)) = (uint16_t)(zh1 & 0xffffu);
          *reinterpret_cast<uint16_t*>(S.v1 + canon(132 + 2 * bh, t, kNV1)) = (uint16_t)(zl0 & 0xffffu);
          *reinterpret_cast<uint16_t*>(S.v1 + canon(133 + 2 * bh, t, kNV1)) = (uint16_t)(zl1 & 0xffffu);
        }
        if (h == 0) bar_sync_threads(2, 128);    // the value-scale pieces are complete
        if (ok) {
          // channel c = b, tokens 64 h .. + 63
          const int c = b, mt = c >> 4, g = c & 7, r = (c >> 3) & 1, gr = c >> 5;
          uint32_t w[4];
#pragma unroll
          for (int tig = 0; tig < 4; ++tig) {
            const uint2 a2 = *reinterpret_cast<const uint2*>(blk + B::kVCodes + ((mt * 2 + h) * 32 + 4 * g + tig) * 8);
            w[tig] = r ? a2.y : a2.x;
          }
#pragma unroll 2
          for (int kb = 8 * h; kb < 8 * h + 8; ++kb) {
            const int kk = (kb >> 1) & 3, hf = kb & 1;
            const uint4 p1 = *reinterpret_cast<const uint4*>(&S.w1[gr][8 * kb]);
            const uint4 p2 = *reinterpret_cast<const uint4*>(&S.w2[gr][8 * kb]);
            const uint32_t pa[4] = {p1.x, p1.y, p1.z, p1.w}, pb[4] = {p2.x, p2.y, p2.z, p2.w};
            uint32_t o1[4], o2[4];
#pragma unroll
            for (int tig = 0; tig < 4; ++tig) {
              const __half2 cd = code_pair(w[tig], 4 * kk + 2 * hf);
              o1[tig] = h2u(__hmul2(cd, u2h(pa[tig])));
              o2[tig] = h2u(__hmul2(cd, u2h(pb[tig])));
            }
            *reinterpret_cast<uint4*>(S.v1 + canon(c, 8 * kb, kNV1)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            *reinterpret_cast<uint4*>(S.v2 + canon(c, 8 * kb, kHeadDim)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
          }
        }
      }
      async_fence();
      bar_sync_threads(2, 128);
      if (lead) publish(&S.vready, (uint32_t)(2 * k + h + 1));
      if (h == 1 && lead && ok && !win && k + kTcStages < ng) {
        // the block is consumed: refill its stage
        async_fence();
        const int s = k % kTcStages;
        mbar_arrive_expect_tx(&S.full[s], B::kBytes);
        bulk_g2s(S.stage[s], blocks + (int64_t)(k + kTcStages) * B::kBytes, B::kBytes, &S.full[s]);
        S.nissued[s] += 1;
      }
    };
    for (int k = 0; k <= nsteps; ++k) {
      if (k < nsteps) keys(k, 0);
      if (k > 0) values(k - 1, 1);
      if (k < nsteps) {
        keys(k, 1);
        values(k, 0);
      }
    }
  } else {
    // =================================================================== rows
    // A step (a group, or the window) is taken in two half-steps, one per
    // 64-token half; half-step j = 2 k + h.  Warps w and w + 4 share rows
    // 32 (w & 3) .. + 31 (their TMEM lanes) and split each half's tokens:
    // warp group 0 takes the first 32 and owns O and the output, group 1 the
    // other 32.  Each warp counts, for the issuer, when it has read the scores
    // of a half-step and when it has written its P.  As for the builders: the
    // same barriers in every half-step, work skipped after an abort.
    const int grp = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int row = blockIdx.x * kTcRows + r;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float fr = S.fexp[r];
    float m_used = -INFINITY, l = 0.0f;   // l: this warp group's sum of p
    bool ok = true;
    // wait for the P.V of half-step jp (bounded)
    auto pv_done = [&](int jp) {
      return tc_wait(&S.odone[jp & 1], (uint32_t)((jp >> 1) & 1), &S.abort_flag, p.err_word);
    };
    // this warp's TMEM accesses before are complete: count it for the issuer
    auto count = [&](uint32_t* c) {
      tfence_before();
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        atomicAdd(c, 1u);
      }
    };
    for (int jj = 0; jj < nh; ++jj) {
      const int k = jj >> 1, h = jj & 1;
      const bool win = k == ng;
      const int c0 = 64 * h + 32 * grp;   // this warp group's 32 tokens of the step
      // the scores of this half-step are done; norms and value zeros (groups)
      // or 2^fw (the window) are in shared memory
      ok = ok && tc_wait(&S.sdone[h], (uint32_t)((jj >> 1) & 1), &S.abort_flag, p.err_word);
      ok = ok && tc_wait_count(&S.kready, (uint32_t)(2 * k), &S.abort_flag, p.err_word);
      ok = __all_sync(0xffffffffu, ok);   // TMEM loads and stores are warp-collective
      // w_t = s_t (log2 units) for this warp group's tokens: groups n_t (S1_t +
      // S2_t + dz) fr, the window (S1_t + S2_t) fr 2^(2 - fw) (-inf past wlen)
      float w[32];
      if (ok) {
        tfence_after();
        uint32_t a[32], b2[32];
        tld32(lane_base + kTS + 32 * grp, a);
        tld32(lane_base + kTS + kN1 + 32 * grp, b2);
        if (win) {
          tld_wait();
          const float fwin = fr * tc_pow2(2 - S.fw);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            w[i] = c0 + i < wlen ? (__uint_as_float(a[i]) + __uint_as_float(b2[i])) * fwin : -INFINITY;
        } else {
          uint32_t z2[2];
          tld2(lane_base + kTS + 64, z2);
          tld_wait();
          const float dz = __uint_as_float(z2[0]) + __uint_as_float(z2[1]);
          const float4* nrm4 = reinterpret_cast<const float4*>(S.nrm[k % 3]) + (c0 >> 2);
          // w = ((s1 + s2) fr + dz fr) n
          const float2 f2 = make_float2(fr, fr), dzf2 = make_float2(dz * fr, dz * fr);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 n4 = nrm4[i >> 2];
            const float2 s01 = __fadd2_rn(make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])),
                                          make_float2(__uint_as_float(b2[i]), __uint_as_float(b2[i + 1])));
            const float2 s23 = __fadd2_rn(make_float2(__uint_as_float(a[i + 2]), __uint_as_float(a[i + 3])),
                                          make_float2(__uint_as_float(b2[i + 2]), __uint_as_float(b2[i + 3])));
            const float2 w01 = __fmul2_rn(__ffma2_rn(s01, f2, dzf2), make_float2(n4.x, n4.y));
            const float2 w23 = __fmul2_rn(__ffma2_rn(s23, f2, dzf2), make_float2(n4.z, n4.w));
            w[i] = w01.x;
            w[i + 1] = w01.y;
            w[i + 2] = w23.x;
            w[i + 3] = w23.y;
          }
        }
      }
      count(&S.sread);   // the score buffer is free for the next half-step's scores
      // pass 1: this warp group's maximum over its 32 tokens
      float mx = -INFINITY;
      if (ok) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          asm("max.f32 %0, %0, %1, %2;" : "+f"(mx) : "f"(w[i]), "f"(w[i + 1]));
        }
        S.pmax[jj & 1][grp][r] = mx;
      }
      named_bar_sync(3, 256);
      uint32_t pk[32];   // [hi pairs of the chunk (16) | lo pairs (16)]
      if (ok) {
        mx = fmaxf(mx, S.pmax[jj & 1][grp ^ 1][r]);
        // running maximum: rescale [O | Z] (TMEM, group 0) and l only when it
        // grows by > 8 (per row, the same decision in both groups; the TMEM
        // pass runs for the whole warp when any of its rows needs it, once the
        // P.V that writes O last has completed)
        const float m_new = fmaxf(m_used, mx);
        const bool need = m_new > m_used + kRescaleLog2 || m_used == -INFINITY;
        const float alpha = !need ? 1.0f : m_used == -INFINITY ? 0.0f : tc_exp2(m_used - m_new);
        if (grp == 0 && jj > 0 && __any_sync(0xffffffffu, need)) {
          const bool done = __all_sync(0xffffffffu, pv_done(jj - 1));
          if (done) {
            tfence_after();
#pragma unroll 1
            for (int o0 = 0; o0 < kHeadDim; o0 += 32) {
              uint32_t orr[32];
              tld32(lane_base + kTO + o0, orr);
              tld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
              tst32(lane_base + kTO + o0, orr);
            }
            uint32_t zr[16];
            tld16(lane_base + kTZ, zr);
            tld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) zr[i] = __float_as_uint(__uint_as_float(zr[i]) * alpha);
            tst16(lane_base + kTZ, zr);
          }
        }
        if (need) {
          l *= alpha;
          m_used = m_new;
        }
        // pass 2: p = 2^(w - m_used) <= 2^8
        const float base = m_used == -INFINITY ? 0.0f : m_used;
        const float2 nb = make_float2(-base, -base);
        float2 lsum = make_float2(0.0f, 0.0f);
        if (win) {
          const float psc = tc_pow2(Gv);    // window P.V in the value pieces' units
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 d = __fadd2_rn(make_float2(w[i], w[i + 1]), nb);
            const float2 p01 = make_float2(tc_exp2(d.x), tc_exp2(d.y));
            lsum = __fadd2_rn(lsum, p01);
            split_p(p01.x * psc, p01.y * psc, true, pk[i >> 1], pk[16 + (i >> 1)]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 d = __fadd2_rn(make_float2(w[i], w[i + 1]), nb);
            const float2 p01 = make_float2(tc_exp2(d.x), tc_exp2(d.y));
            lsum = __fadd2_rn(lsum, p01);
            split_p16(p01.x, p01.y, pk[i >> 1], pk[16 + (i >> 1)]);
          }
        }
        l += lsum.x + lsum.y;
      }
      // P goes over the P of half-step j - 2 once its P.V has read it
      bool pv_ok = true;
      if (ok && jj > 1) pv_ok = pv_done(jj - 2);
      ok = __all_sync(0xffffffffu, ok && pv_ok);
      if (ok) {
        tfence_after();
        tst32(lane_base + kTP + 64 * (jj & 1) + 32 * grp, pk);
      }
      tst_wait();
      count(&S.pcount);
    }
    // ---- the last P.V, then the rows out (group 0): o = (O 2^-Gv + Z
    // 2^-gz) / l, lse = (m + log2 l) ln 2 (the TMEM loads for the whole warp,
    // the stores for rows that exist)
    if (grp == 1) S.lpart[r] = l;
    ok = ok && (nh == 0 || pv_done(nh - 1));
    ok = __all_sync(0xffffffffu, ok);
    named_bar_sync(3, 256);
    if (grp == 0 && ok) {
      tfence_after();
      l += S.lpart[r];
      float zs[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // sum p z^V per value group (no groups: none)
      {
        uint32_t zr[16];
        tld16(lane_base + kTZ, zr);
        tld_wait();
        const float izf = tc_pow2(-S.gz);
        if (ng > 0) {
#pragma unroll
          for (int gr = 0; gr < 4; ++gr) zs[gr] = (__uint_as_float(zr[gr]) + __uint_as_float(zr[4 + gr])) * izf;
        }
      }
      const bool live_row = row < p.rows;
      const float iv = tc_pow2(-Gv);
      const int qi = row / p.gqa, hq = j * p.gqa + row % p.gqa;
      float* rec = p.n_parts > 1 ? p.parts + (((int64_t)part * p.hkv + j) * p.rows + row) * kPrefillRecFloats : nullptr;
      const float inv = 1.0f / l;
#pragma unroll 1
      for (int o0 = 0; o0 < kHeadDim; o0 += 32) {
        uint32_t orr[32];
        tld32(lane_base + kTO + o0, orr);
        tld_wait();
        const float z = zs[o0 >> 5];
        if (live_row && rec) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(rec + o0 + i) =
                make_float4(fmaf(__uint_as_float(orr[i]), iv, z), fmaf(__uint_as_float(orr[i + 1]), iv, z),
                            fmaf(__uint_as_float(orr[i + 2]), iv, z), fmaf(__uint_as_float(orr[i + 3]), iv, z));
        } else if (live_row) {
          uint32_t* orow = reinterpret_cast<uint32_t*>(p.out + ((int64_t)qi * p.hq + hq) * kHeadDim + o0);
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint32_t u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float o_0 = fmaf(__uint_as_float(orr[i + 2 * e]), iv, z) * inv;
              const float o_1 = fmaf(__uint_as_float(orr[i + 2 * e + 1]), iv, z) * inv;
              u[e] = f32_to_bf16_bits(o_0) | (f32_to_bf16_bits(o_1) << 16);
            }
            *reinterpret_cast<uint4*>(orow + i / 2) = make_uint4(u[0], u[1], u[2], u[3]);
          }
        }
      }
      if (!live_row) {
      } else if (rec) {
        *reinterpret_cast<float2*>(rec + kHeadDim) = make_float2(m_used, l);
      } else if (p.lse != nullptr) {
        p.lse[(int64_t)qi * p.hq + hq] = (m_used + log2f(l)) * 0.69314718055994530942f;
      }
    }
  }

  // ---- teardown: copies still in flight after an abort, then TMEM
  tfence_before();
  __syncthreads();
  if (S.abort_flag && tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      const uint32_t n = *reinterpret_cast<volatile uint32_t*>(&S.nissued[s]);
      if (n == 0) continue;
      for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(&S.full[s], (n - 1) & 1)) break;
    }
  }
  __syncthreads();
  if (warp == 8) {
    tfence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTCols) : "memory");
  }
}

}  // namespace

template <bool M16>
cudaError_t launch_prefill_tc_t(const PrefillParams& p, const uint8_t* arena, cudaStream_t stream) {
  static bool attr_done[64] = {};
  const int smem = (int)sizeof(TcSmem) + 1024;
  cudaError_t e = ensure_smem_attr(prefill_tc_kernel<M16>, smem, attr_done);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.rows + kTcRows - 1) / kTcRows, p.hkv, p.n_parts);
  prefill_tc_kernel<M16><<<grid, kTcThreads, smem, stream>>>(p, arena);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const PrefillParams& p, const uint8_t* arena, bool meta16, cudaStream_t stream) {
  return meta16 ? launch_prefill_tc_t<true>(p, arena, stream) : launch_prefill_tc_t<false>(p, arena, stream);
}

}  // namespace oscar
