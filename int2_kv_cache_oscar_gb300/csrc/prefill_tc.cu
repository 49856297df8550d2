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
// row) and a range of the history's groups; 8 warps:
//   * builders (warps 4-7): per group, expand the packed codes into exact
//     fp16 B operands in shared memory (no-swizzle K-major core matrices):
//     scores B[token][channel] = code * S_i(c) and values B[channel][token] =
//     code * S_i^V(t, group), where S_1 + S_2 is the scale split into two
//     9-significant-bit pieces (so code * S_i, code <= 3, is exact in fp16);
//     extra B rows carry the key and value zeros (hi + lo).  Key and value
//     operands have buffers of their own, so the keys of group k + 1 are
//     built while the rows work on group k.  Their first thread also streams
//     the group blocks through a ring of bulk copies and issues every
//     tcgen05.mma: the P.V of group k - 1 and then the scores of group k;
//   * rows (warps 0-3, thread = row): online softmax over the scores read
//     from TMEM; P (hi + lo fp16) goes back to TMEM over the scores just read
//     and is the A operand of P.V; the output accumulator O stays in TMEM and
//     is rescaled only when a row's maximum grows by more than 8 (log2 units;
//     P stays below 2^8).
// Products (hi + lo of the rows' rotated queries, constant in TMEM):
//   scores  S = Qhi B1 + Qlo B1 + Qhi B2          (N = 144: 128 tokens + zero rows)
//   values  O += Phi V1 + Plo V1 + Phi V2         (N = 128 channels)
//           Z  = Phi Vz + Plo Vz                  (N = 16: the value-zero term)
// dropping only the products of two low parts (relative 2^-20).  The window
// comes last, on bf16 operands (q and k exact; P as bf16 hi + lo).  With a
// workspace the history is split into parts (grid.z), each writing per-row
// records (o unnormalised, m, l) that the merge kernel combines.
#include <cstddef>

#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int kTcRows = 128;
constexpr int kTcThreads = 12 * 32;
constexpr int kTcStages = 3;
constexpr int kNS = 144;                 // score B rows (and value B rows with the zero rows): 128 + 16
constexpr int kBBytes = kNS * kHeadDim * 2;
constexpr int kBVBytes2 = kHeadDim * kGroup * 2;     // value piece 2: 128 channel rows only
constexpr uint32_t kLboB = (kNS / 8) * 128;          // B: core matrices adjacent along K
constexpr uint32_t kLboV2 = (kHeadDim / 8) * 128;
constexpr uint32_t kSbo = 128;                       // core matrices adjacent along M / N
// TMEM columns (512 allocated)
constexpr uint32_t kTQ = 0;        // rotated q * 2^F: hi fp16 pairs [0, 64), lo [64, 128)
constexpr uint32_t kTQraw = 128;   // raw q, bf16 pairs [128, 192)
constexpr uint32_t kTS = 192;      // scores [192, 336); P over [192, 320) (see p_col)
constexpr uint32_t kTO = 336;      // output accumulator [336, 464)
constexpr uint32_t kTZ = 464;      // value-zero term [464, 480)
constexpr uint32_t kTCols = 512;
constexpr float kRescaleLog2 = 8.0f;

// TMEM column of the P pairs of k-step ks (tokens 16 ks .. 16 ks + 15), hi or
// lo: each 32-token chunk c of the scores becomes [hi of its two k-steps | lo
// of its two k-steps] in the chunk's own 32 columns.
__host__ __device__ constexpr uint32_t p_col(int ks, bool lo) {
  return kTS + 32 * (ks >> 1) + (lo ? 16 : 0) + 8 * (ks & 1);
}

struct TcSmem {
  alignas(1024) uint8_t k1[kBBytes];                  // key B piece 1 (+ zero rows)
  alignas(1024) uint8_t k2[kBBytes];                  // key B piece 2 (zero rows cleared)
  alignas(1024) uint8_t v1[kBBytes];                  // value B piece 1 (+ zero rows)
  alignas(1024) uint8_t v2[kBVBytes2];                // value B piece 2
  alignas(128) uint8_t stage[kTcStages][kBlockBytes];
  float nrm[2][kGroup];                               // key norms of groups k, k + 1
  alignas(16) uint16_t s1[kHeadDim], s2[kHeadDim];    // key-scale pieces (fp16) per channel
  alignas(16) uint16_t w1[kVGroups][kGroup], w2[kVGroups][kGroup];   // value-scale pieces [group][token]
  float zmax[2][4];                                   // per builder warp: max |z^V| (double-buffered)
  int gz[2];                                          // the value-zero rows carry 2^gz (double-buffered)
  float fexp[kTcRows];                                // 2^-(F_row + 2) * scale_log2
  float pmax[2][kTcRows];                             // row maxima of the two token halves
  float lpart[kTcRows];                               // the second half's sum of p
  alignas(8) uint64_t full[kTcStages];
  uint64_t zred, sdone, pready, odone;
  // steps whose key / value operands (and norms / zero exponent) are complete:
  // monotonic counts, since the builders may run a step ahead of a waiter
  uint32_t kready, vready;
  uint32_t nissued[kTcStages];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(TcSmem) + 1024 <= 232448, "one CTA per SM");
static_assert(offsetof(TcSmem, stage) % 128 == 0 && offsetof(TcSmem, full) % 8 == 0, "alignment");
static_assert(kBBytes + kBVBytes2 >= kTcRows * kHeadDim * 4, "q staging fits in the value buffers");

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

// Key operands of one group into k1 / k2 (builder thread b = token and
// channel b): scale pieces (x 4), zero rows 128, 129 (z hi, lo x 4), cleared
// rows, the norms, then the codes of token b.
template <bool M16>
__device__ __forceinline__ void build_keys(TcSmem& S, const uint8_t* blk, int b, float* nrm) {
  using B = Blk<M16>;
  using MR = Meta<M16>;
  pieces(MR::one(blk + B::kKScale, b) * 4.0f, S.s1[b], S.s2[b]);
  uint32_t zh, zl;
  split2(MR::one(blk + B::kKZero, b) * 4.0f, 0.0f, false, zh, zl);
  *reinterpret_cast<uint16_t*>(S.k1 + canon(128, b, kNS)) = (uint16_t)(zh & 0xffffu);
  *reinterpret_cast<uint16_t*>(S.k1 + canon(129, b, kNS)) = (uint16_t)(zl & 0xffffu);
  nrm[b] = MR::one(blk + B::kKNorm, b);
  for (int i = b; i < 16 * 16 * 2; i += 128) {   // rows 130..143 of k1, 128..143 of k2
    const int h2 = i >> 8, rr = 128 + ((i >> 4) & 15), kb = i & 15;
    if (h2 == 0 && rr < 130) continue;
    *reinterpret_cast<uint4*>((h2 ? S.k2 : S.k1) + canon(rr, 8 * kb, kNS)) = make_uint4(0u, 0u, 0u, 0u);
  }
  bar_sync_threads(2, 128);    // the scale pieces are complete
  const int t = b, mt = t >> 4, g = t & 7, r = (t >> 3) & 1;
  uint32_t w0[4], w1[4];       // fragment words of token t: channel halves j = 0, 1
#pragma unroll
  for (int tig = 0; tig < 4; ++tig) {
    const uint4 q4 = *reinterpret_cast<const uint4*>(blk + kOffKCodes + (mt * 32 + 4 * g + tig) * 16);
    w0[tig] = r ? q4.y : q4.x;
    w1[tig] = r ? q4.w : q4.z;
  }
#pragma unroll 2
  for (int kb = 0; kb < 16; ++kb) {
    const int ks = kb >> 1, hf = kb & 1, kk = ks & 3;
    const uint4 p1 = *reinterpret_cast<const uint4*>(&S.s1[8 * kb]);
    const uint4 p2 = *reinterpret_cast<const uint4*>(&S.s2[8 * kb]);
    const uint32_t pa[4] = {p1.x, p1.y, p1.z, p1.w}, pb[4] = {p2.x, p2.y, p2.z, p2.w};
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int tig = 0; tig < 4; ++tig) {
      const __half2 cd = code_pair(ks >= 4 ? w1[tig] : w0[tig], 4 * kk + 2 * hf);
      o1[tig] = h2u(__hmul2(cd, u2h(pa[tig])));
      o2[tig] = h2u(__hmul2(cd, u2h(pb[tig])));
    }
    *reinterpret_cast<uint4*>(S.k1 + canon(t, 8 * kb, kNS)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    *reinterpret_cast<uint4*>(S.k2 + canon(t, 8 * kb, kNS)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  }
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
    mbar_init(&S.zred, 4);
    mbar_init(&S.sdone, 1);
    mbar_init(&S.pready, 1);
    mbar_init(&S.odone, 1);
    S.kready = 0;
    S.vready = 0;
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
  uint32_t* qraw = reinterpret_cast<uint32_t*>(S.k1);             // [128][64] raw bf16 pairs
  for (int r = warp; r < kTcRows; r += 12) {
    const int row = blockIdx.x * kTcRows + r;
    uint2 raw = make_uint2(0u, 0u);
    if (row < p.rows) {
      const int qi = row / p.gqa, h = j * p.gqa + row % p.gqa;
      raw = *reinterpret_cast<const uint2*>(p.q + ((int64_t)qi * p.hq + h) * kHeadDim + 4 * lane);
    }
    qraw[r * 64 + 2 * lane] = raw.x;
    qraw[r * 64 + 2 * lane + 1] = raw.y;
    float qv[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
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
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qv[i] *= 0.088388347648318440550f;   // 1/sqrt(128)
      mx = fmaxf(mx, fabsf(qv[i]));
    }
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
    // row thread r stores hi / lo fp16 pairs and the raw bf16 pairs into its lane
    const int r = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t hi[32], lo[32], rw[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x0 = qst[r * kHeadDim + 2 * (c0 + i)], x1 = qst[r * kHeadDim + 2 * (c0 + i) + 1];
        split2(x0, x1, false, hi[i], lo[i]);
        rw[i] = qraw[r * 64 + c0 + i];
      }
      tst32(lane_base + kTQ + c0, hi);
      tst32(lane_base + kTQ + 64 + c0, lo);
      tst32(lane_base + kTQraw + c0, rw);
    }
    tst_wait();
  }
  tfence_before();
  __syncthreads();   // the staging areas are free again
  tfence_after();

  if (warp >= 8) {
    // =============================================================== builders
    // Every builder runs the same barriers in every step; after a wait gives
    // up (abort) the work is skipped but the control flow stays the same.
    const int b = tid - 256;     // token (key codes, value zero rows) or channel (value codes)
    const int bw = warp - 8;
    const float gv = tc_pow2(Gv);
    const bool lead = b == 0;    // also streams the group blocks
    const uint8_t* wsrc = arena + p.windows_off + ((int64_t)p.slot * p.hkv + j) * kWindowBytes;
    if (lead) {
      for (int k = 0; k < ng && k < kTcStages; ++k) {
        mbar_arrive_expect_tx(&S.full[k], B::kBytes);
        bulk_g2s(S.stage[k], blocks + (int64_t)k * B::kBytes, B::kBytes, &S.full[k]);
        S.nissued[k] = 1;
      }
    }
    for (int k = 0; k < nsteps; ++k) {
      const bool win = k == ng;
      const int s = k % kTcStages;
      const uint32_t par = (uint32_t)(k & 1);
      // ---- key operands of step k, once the scores of step k - 1 are done
      bool ok = win || tc_wait(&S.full[s], (uint32_t)((k / kTcStages) & 1), &S.abort_flag, p.err_word);
      ok = ok && (k == 0 || tc_wait(&S.sdone, (uint32_t)((k - 1) & 1), &S.abort_flag, p.err_word));
      const uint8_t* blk = S.stage[s];
      if (win) {
        // the window keys as B[token][channel], bf16 (rows past wlen zero)
        if (ok) {
          const uint4* krow = reinterpret_cast<const uint4*>(wsrc + b * kHeadDim * 2);
#pragma unroll 4
          for (int kb = 0; kb < 16; ++kb)
            *reinterpret_cast<uint4*>(S.k1 + canon(b, 8 * kb, kNS)) = b < wlen ? krow[kb] : make_uint4(0u, 0u, 0u, 0u);
        }
        bar_sync_threads(2, 128);   // (matches the barrier inside build_keys)
      } else if (ok) {
        build_keys<M16>(S, blk, b, S.nrm[k & 1]);
      } else {
        bar_sync_threads(2, 128);
      }
      async_fence();
      bar_sync_threads(2, 128);
      if (lead) publish(&S.kready, (uint32_t)(k + 1));
      // ---- value operands of step k, once the P.V of step k - 1 is done
      ok = ok && (k == 0 || tc_wait(&S.odone, (uint32_t)((k - 1) & 1), &S.abort_flag, p.err_word));
      if (win) {
        if (ok) {
          // the window values transposed into B[channel][token], bf16
          const uint16_t* vrow = reinterpret_cast<const uint16_t*>(wsrc + kGroup * kHeadDim * 2 + b * kHeadDim * 2);
#pragma unroll 1
          for (int c = 0; c < kHeadDim; c += 8) {
            const uint4 v8 = b < wlen ? *reinterpret_cast<const uint4*>(vrow + c) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t e4[4] = {v8.x, v8.y, v8.z, v8.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint16_t*>(S.v1 + canon(c + i, b, kNS)) = (uint16_t)(e4[i >> 1] >> (16 * (i & 1)));
          }
        }
        async_fence();
        bar_sync_threads(2, 128);
        if (lead) publish(&S.vready, (uint32_t)(k + 1));
        continue;
      }
      float zm = 0.0f;
      if (ok) {
        // token b: its four value scales as pieces (x 2^Gv), and max |z^V|
        const float4 sv = MR::v4(blk + B::kVScale, b);
        const float4 zv = MR::v4(blk + B::kVZero, b);
        pieces(sv.x * gv, S.w1[0][b], S.w2[0][b]);
        pieces(sv.y * gv, S.w1[1][b], S.w2[1][b]);
        pieces(sv.z * gv, S.w1[2][b], S.w2[2][b]);
        pieces(sv.w * gv, S.w1[3][b], S.w2[3][b]);
        zm = fmaxf(fmaxf(fabsf(zv.x), fabsf(zv.y)), fmaxf(fabsf(zv.z), fabsf(zv.w)));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, o));
      if (lane == 0) {
        S.zmax[k & 1][bw] = zm;
        mbar_arrive(&S.zred);
      }
      ok = ok && tc_wait(&S.zred, par, &S.abort_flag, p.err_word);
      if (ok) {
        const float zmx = fmaxf(fmaxf(S.zmax[k & 1][0], S.zmax[k & 1][1]), fmaxf(S.zmax[k & 1][2], S.zmax[k & 1][3]));
        int Gz = 0;
        if (zmx > 0.0f) {
          int e;
          frexpf(zmx, &e);   // zmx < 2^e
          Gz = 14 - e;
        }
        const float gzf = tc_pow2(Gz);
        const float4 zv = MR::v4(blk + B::kVZero, b);
        const float zz[4] = {zv.x * gzf, zv.y * gzf, zv.z * gzf, zv.w * gzf};
        // rows 128 + gr: z hi, 132 + gr: z lo (B[row][token b]); rows 136..143 zero
#pragma unroll
        for (int gr = 0; gr < 4; ++gr) {
          uint32_t zh, zl;
          split2(zz[gr], 0.0f, false, zh, zl);
          *reinterpret_cast<uint16_t*>(S.v1 + canon(128 + gr, b, kNS)) = (uint16_t)(zh & 0xffffu);
          *reinterpret_cast<uint16_t*>(S.v1 + canon(132 + gr, b, kNS)) = (uint16_t)(zl & 0xffffu);
        }
#pragma unroll
        for (int rr = 136; rr < 144; ++rr) *reinterpret_cast<uint16_t*>(S.v1 + canon(rr, b, kNS)) = 0;
        if (b == 0) S.gz[k & 1] = Gz;   // read by the row threads once this step's P.V is done
      }
      bar_sync_threads(2, 128);    // the value-scale pieces are complete
      if (ok) {
        const int c = b, mt = c >> 4, g = c & 7, r = (c >> 3) & 1, gr = c >> 5;
        uint32_t w0[4], w1[4];     // V-order words of channel c: token halves j = 0, 1
#pragma unroll
        for (int tig = 0; tig < 4; ++tig) {
          const uint2 a2 = *reinterpret_cast<const uint2*>(blk + B::kVCodes + ((mt * 2 + 0) * 32 + 4 * g + tig) * 8);
          const uint2 b2 = *reinterpret_cast<const uint2*>(blk + B::kVCodes + ((mt * 2 + 1) * 32 + 4 * g + tig) * 8);
          w0[tig] = r ? a2.y : a2.x;
          w1[tig] = r ? b2.y : b2.x;
        }
#pragma unroll 2
        for (int kb = 0; kb < 16; ++kb) {
          const int ks = kb >> 1, hf = kb & 1, kk = ks & 3;
          const uint4 p1 = *reinterpret_cast<const uint4*>(&S.w1[gr][8 * kb]);
          const uint4 p2 = *reinterpret_cast<const uint4*>(&S.w2[gr][8 * kb]);
          const uint32_t pa[4] = {p1.x, p1.y, p1.z, p1.w}, pb[4] = {p2.x, p2.y, p2.z, p2.w};
          uint32_t o1[4], o2[4];
#pragma unroll
          for (int tig = 0; tig < 4; ++tig) {
            const __half2 cd = code_pair(ks >= 4 ? w1[tig] : w0[tig], 4 * kk + 2 * hf);
            o1[tig] = h2u(__hmul2(cd, u2h(pa[tig])));
            o2[tig] = h2u(__hmul2(cd, u2h(pb[tig])));
          }
          *reinterpret_cast<uint4*>(S.v1 + canon(c, 8 * kb, kNS)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          *reinterpret_cast<uint4*>(S.v2 + canon(c, 8 * kb, kHeadDim)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        }
      }
      async_fence();
      bar_sync_threads(2, 128);
      if (lead) publish(&S.vready, (uint32_t)(k + 1));
      if (lead && ok && k + kTcStages < ng) {
        // the block is consumed: refill its stage
        async_fence();
        mbar_arrive_expect_tx(&S.full[s], B::kBytes);
        bulk_g2s(S.stage[s], blocks + (int64_t)(k + kTcStages) * B::kBytes, B::kBytes, &S.full[s]);
        S.nissued[s] += 1;
      }
    }
  } else {
    // =================================================================== rows
    // Warps w and w + 4 share rows 32 (w & 3) .. + 31 (their TMEM lanes) and
    // split the tokens: half 0 takes tokens 0..63 and owns O, the zero sums
    // and the output; half 1 takes tokens 64..127.  As for the builders: the
    // same barriers in every step, work skipped after an abort.  Thread 0 also
    // issues every tcgen05.mma: the scores of step k + 1 right after the P.V
    // of step k (the scores overwrite its P).
    const int half = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int row = blockIdx.x * kTcRows + r;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const bool issuer = tid == 0;
    const float fr = S.fexp[r];
    float m_used = -INFINITY, l = 0.0f;   // l: this half's sum of p
    float zacc[kVGroups] = {0.0f, 0.0f, 0.0f, 0.0f};
    bool ok = true;
    const uint32_t idS = idesc_f16(kNS, false), idO = idesc_f16(kHeadDim, false), idZ = idesc_f16(16, false);
    const uint32_t idW = idesc_f16(kHeadDim, true);
    const uint32_t sk1 = smem_u32(S.k1), sk2 = smem_u32(S.k2), sv1 = smem_u32(S.v1), sv2 = smem_u32(S.v2);
    uint32_t n_sdone = 0, n_odone = 0;   // commits issued (issuer)
    auto issue_scores = [&](int ks_step) {
      if (!tc_wait_count(&S.kready, (uint32_t)ks_step, &S.abort_flag, p.err_word)) return;
      tfence_after();
      const bool w = ks_step == ng;
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t dk1 = sdesc(sk1 + 2 * ks * kLboB, kLboB, kSbo);
        if (w) {
          mma_ts(tmem + kTS, tmem + kTQraw + 8 * ks, dk1, idW, ks > 0);
        } else {
          const uint64_t dk2 = sdesc(sk2 + 2 * ks * kLboB, kLboB, kSbo);
          mma_ts(tmem + kTS, tmem + kTQ + 8 * ks, dk1, idS, ks > 0);
          mma_ts(tmem + kTS, tmem + kTQ + 64 + 8 * ks, dk1, idS, true);
          mma_ts(tmem + kTS, tmem + kTQ + 8 * ks, dk2, idS, true);
        }
      }
      mma_commit(&S.sdone);
      ++n_sdone;
    };
    auto issue_pv = [&](int kp) {
      if (!tc_wait_count(&S.vready, (uint32_t)kp, &S.abort_flag, p.err_word)) return;
      tfence_after();
      const bool w = kp == ng;
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ah = tmem + p_col(ks, false), al = tmem + p_col(ks, true);
        const uint64_t dv1 = sdesc(sv1 + 2 * ks * kLboB, kLboB, kSbo);
        if (w) {
          mma_ts(tmem + kTO, ah, dv1, idW, kp > 0 || ks > 0);
          mma_ts(tmem + kTO, al, dv1, idW, true);
        } else {
          const uint64_t dv2 = sdesc(sv2 + 2 * ks * kLboV2, kLboV2, kSbo);
          const uint64_t dvz = sdesc(sv1 + 2 * ks * kLboB + (kHeadDim / 8) * 128, kLboB, kSbo);
          mma_ts(tmem + kTO, ah, dv1, idO, kp > 0 || ks > 0);
          mma_ts(tmem + kTO, al, dv1, idO, true);
          mma_ts(tmem + kTO, ah, dv2, idO, true);
          mma_ts(tmem + kTZ, ah, dvz, idZ, ks > 0);
          mma_ts(tmem + kTZ, al, dvz, idZ, true);
        }
      }
      mma_commit(&S.odone);
      ++n_odone;
    };
    // the value-zero term of step kz (after its P.V), folded into zacc (half 0)
    auto take_z = [&](int kz) {
      uint32_t zr[16];
      tld16(lane_base + kTZ, zr);
      tld_wait();
      const float iz = tc_pow2(-S.gz[kz & 1]);
#pragma unroll
      for (int gr = 0; gr < 4; ++gr) zacc[gr] = fmaf(__uint_as_float(zr[gr]) + __uint_as_float(zr[4 + gr]), iz, zacc[gr]);
    };
    if (issuer && nsteps > 0) issue_scores(0);
    const int t0 = 64 * half;   // this half's first token
    for (int k = 0; k < nsteps; ++k) {
      const bool win = k == ng;
      const uint32_t par = (uint32_t)(k & 1);
      // the scores of step k are done, and with them the P.V of step k - 1
      ok = ok && tc_wait(&S.sdone, par, &S.abort_flag, p.err_word);
      ok = ok && (win || tc_wait_count(&S.kready, (uint32_t)k, &S.abort_flag, p.err_word));
      ok = ok && (k == 0 || tc_wait_count(&S.vready, (uint32_t)(k - 1), &S.abort_flag, p.err_word));
      ok = __all_sync(0xffffffffu, ok);   // TMEM loads and stores are warp-collective
      float mx = -INFINITY;
      float dz = 0.0f;
      const float4* nrm4 = reinterpret_cast<const float4*>(S.nrm[k & 1]);
      const float fs = win ? p.scale_log2 : 0.0f;
      const float psc = win ? tc_pow2(Gv) : 1.0f;    // window P.V in the value pieces' units
      // s - base for tokens c0 + i .. + 3 (log2 units): groups n_t (S_t + dz) fr,
      // the window S_t scale (-inf past wlen)
      auto shifted = [&](const uint32_t (&sr)[32], int c0, int i, float base, float2& w01, float2& w23) {
        const float2 s01 = make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
        const float2 s23 = make_float2(__uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3]));
        const float2 nb = make_float2(-base, -base);
        if (win) {
          const float2 f2 = make_float2(fs, fs);
          w01 = __ffma2_rn(s01, f2, nb);
          w23 = __ffma2_rn(s23, f2, nb);
          if (c0 + i >= wlen) w01.x = -INFINITY;
          if (c0 + i + 1 >= wlen) w01.y = -INFINITY;
          if (c0 + i + 2 >= wlen) w23.x = -INFINITY;
          if (c0 + i + 3 >= wlen) w23.y = -INFINITY;
        } else {
          const float4 n4 = nrm4[(c0 + i) >> 2];
          const float2 d2 = make_float2(dz, dz), f2 = make_float2(fr, fr);
          w01 = __ffma2_rn(__fadd2_rn(s01, d2), __fmul2_rn(make_float2(n4.x, n4.y), f2), nb);
          w23 = __ffma2_rn(__fadd2_rn(s23, d2), __fmul2_rn(make_float2(n4.z, n4.w), f2), nb);
        }
      };
      if (ok) {
        tfence_after();
        if (half == 0 && k > 0) take_z(k - 1);   // before this step's rescale and P.V
        if (!win) {
          uint32_t zr[16];
          tld16(lane_base + kTS + 128, zr);
          tld_wait();
          dz = __uint_as_float(zr[0]) + __uint_as_float(zr[1]);
        }
        // pass 1: this half's maximum (the scores stay in TMEM; pass 2 writes P over them)
#pragma unroll 1
        for (int c0 = t0; c0 < t0 + 64; c0 += 32) {
          uint32_t sr[32];
          tld32(lane_base + kTS + c0, sr);
          tld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float2 w01, w23;
            shifted(sr, c0, i, 0.0f, w01, w23);
            mx = fmaxf(mx, fmaxf(fmaxf(w01.x, w01.y), fmaxf(w23.x, w23.y)));
          }
        }
        S.pmax[half][r] = mx;
      }
      named_bar_sync(3, 256);
      if (ok) {
        mx = fmaxf(mx, S.pmax[half ^ 1][r]);
        // running maximum: rescale O (TMEM, half 0), the zero sums and l only when
        // it grows by > 8 (per row, the same decision in both halves; the TMEM
        // pass runs for the whole warp when any of its rows needs it)
        const float m_new = fmaxf(m_used, mx);
        const bool need = m_new > m_used + kRescaleLog2 || m_used == -INFINITY;
        const float alpha = !need ? 1.0f : m_used == -INFINITY ? 0.0f : tc_exp2(m_used - m_new);
        if (half == 0 && k > 0 && __any_sync(0xffffffffu, need)) {   // O is not being written (see above)
#pragma unroll 1
          for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
            uint32_t orr[32];
            tld32(lane_base + kTO + c0, orr);
            tld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tst32(lane_base + kTO + c0, orr);
          }
        }
        if (need) {
#pragma unroll
          for (int gr = 0; gr < kVGroups; ++gr) zacc[gr] *= alpha;
          l *= alpha;
          m_used = m_new;
        }
        // pass 2: P = 2^(s - m_used) <= 2^8 into TMEM over the 32 score
        // columns just read (see p_col)
        const float base = m_used == -INFINITY ? 0.0f : m_used;
        float2 lsum = make_float2(0.0f, 0.0f);
#pragma unroll 1
        for (int c0 = t0; c0 < t0 + 64; c0 += 32) {
          uint32_t sr[32];
          tld32(lane_base + kTS + c0, sr);
          tld_wait();
          uint32_t pk[32];   // [hi pairs of the chunk (16) | lo pairs (16)]
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float2 w01, w23;
            shifted(sr, c0, i, base, w01, w23);
            const float2 p01 = make_float2(tc_exp2(w01.x), tc_exp2(w01.y));
            const float2 p23 = make_float2(tc_exp2(w23.x), tc_exp2(w23.y));
            lsum = __fadd2_rn(lsum, __fadd2_rn(p01, p23));
            split_p(p01.x * psc, p01.y * psc, win, pk[i >> 1], pk[16 + (i >> 1)]);
            split_p(p23.x * psc, p23.y * psc, win, pk[(i >> 1) + 1], pk[16 + (i >> 1) + 1]);
          }
          tst32(lane_base + kTS + c0, pk);
        }
        l += lsum.x + lsum.y;
      }
      tst_wait();
      tfence_before();
      named_bar_sync(3, 256);
      if (issuer && ok) {
        issue_pv(k);
        if (k + 1 < nsteps) issue_scores(k + 1);
      }
    }
    // ---- the last P.V, its value-zero term, then the rows out (half 0):
    // o = (O 2^-Gv + z) / l, lse = (m + log2 l) ln 2 (the TMEM loads for the
    // whole warp, the stores for rows that exist)
    if (half == 1) S.lpart[r] = l;
    ok = ok && (nsteps == 0 || tc_wait(&S.odone, (uint32_t)((nsteps - 1) & 1), &S.abort_flag, p.err_word));
    ok = __all_sync(0xffffffffu, ok);
    named_bar_sync(3, 256);
    if (half == 0 && ok) {
      tfence_after();
      if (nsteps > 0 && nsteps - 1 != ng) take_z(nsteps - 1);
      l += S.lpart[r];
      const bool live_row = row < p.rows;
      const float iv = tc_pow2(-Gv);
      const int qi = row / p.gqa, h = j * p.gqa + row % p.gqa;
      float* rec = p.n_parts > 1 ? p.parts + (((int64_t)part * p.hkv + j) * p.rows + row) * kPrefillRecFloats : nullptr;
      const float inv = 1.0f / l;
#pragma unroll 1
      for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
        uint32_t orr[32];
        tld32(lane_base + kTO + c0, orr);
        tld_wait();
        const float z = zacc[c0 >> 5];
        if (live_row && rec) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(rec + c0 + i) =
                make_float4(fmaf(__uint_as_float(orr[i]), iv, z), fmaf(__uint_as_float(orr[i + 1]), iv, z),
                            fmaf(__uint_as_float(orr[i + 2]), iv, z), fmaf(__uint_as_float(orr[i + 3]), iv, z));
        } else if (live_row) {
          uint32_t* orow = reinterpret_cast<uint32_t*>(p.out + ((int64_t)qi * p.hq + h) * kHeadDim + c0);
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint32_t u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float o0 = fmaf(__uint_as_float(orr[i + 2 * e]), iv, z) * inv;
              const float o1 = fmaf(__uint_as_float(orr[i + 2 * e + 1]), iv, z) * inv;
              u[e] = f32_to_bf16_bits(o0) | (f32_to_bf16_bits(o1) << 16);
            }
            *reinterpret_cast<uint4*>(orow + i / 2) = make_uint4(u[0], u[1], u[2], u[3]);
          }
        }
      }
      if (!live_row) {
      } else if (rec) {
        *reinterpret_cast<float2*>(rec + kHeadDim) = make_float2(m_used, l);
      } else if (p.lse != nullptr) {
        p.lse[(int64_t)qi * p.hq + h] = (m_used + log2f(l)) * 0.69314718055994530942f;
      }
    }
    if (issuer) {
      // before TMEM is freed: the last committed MMAs have completed (bounded,
      // whatever the abort state: MMAs always complete)
      for (int q = 0; q < 2; ++q) {
        const uint32_t n = q ? n_odone : n_sdone;
        if (n == 0) continue;
        for (uint32_t i = 0; i < kSpinLimit; ++i)
          if (mbar_try_wait(q ? &S.odone : &S.sdone, (n - 1) & 1)) break;
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
