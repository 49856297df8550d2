// Shared constants, arena layout and PTX helpers of the sm_103a OScaR kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace oscar {

constexpr int kHeadDim = 128;        // d
constexpr int kGroup = 128;          // G: tokens per key group
constexpr int kVGroup = 32;          // channels per value group
constexpr int kVGroups = kHeadDim / kVGroup;

// One quantised group of one KV head (see include/oscar.h).
constexpr int kOffKCodes = 0;
constexpr int kOffKScale = 4096;
constexpr int kOffKZero = 4608;
constexpr int kOffKNorm = 5120;
constexpr int kOffVCodes = 5632;
constexpr int kOffVScale = 9728;
constexpr int kOffVZero = 11776;
constexpr int kBlockBytes = 13824;

// The same block with float16 metadata (scales, zeros, norms).
constexpr int kOff16KScale = 4096;
constexpr int kOff16KZero = 4352;
constexpr int kOff16KNorm = 4608;
constexpr int kOff16VCodes = 4864;
constexpr int kOff16VScale = 8960;
constexpr int kOff16VZero = 9984;
constexpr int kBlockBytes16 = 11008;

// Row of token t in the float32 value scale and zero arrays ([128][4]):
// tokens t and t ^ 1 trade places where bit 3 of t is set.  Decode lanes read
// the scales of tokens t and t + 8 (the two threads of a B-column pair) in
// the same 128-bit load; unswizzled those rows are 128 bytes apart, in the
// same banks.  An involution: the stored row p holds token vmeta_row(p).
__host__ __device__ constexpr int vmeta_row(int t) { return t ^ ((t >> 3) & 1); }

// Byte offset, within the value-code section, of fragment word pair (r = 0, 1)
// of m-tile mt, token half j and lane ("V order": a warp's pairs for one
// (mt, j) are 256 contiguous bytes).  Key codes keep the "K order"
// ((mt * 32 + lane) * 4 + 2 j + r) * 4 (a lane's four words are contiguous).
__host__ __device__ constexpr int vword_off(int mt, int j, int lane) { return ((mt * 2 + j) * 32 + lane) * 8; }

// Block layout by metadata width: section offsets, block size, bytes per
// metadata element.
template <bool M16>
struct Blk {
  static constexpr int kKScale = M16 ? kOff16KScale : kOffKScale;
  static constexpr int kKZero = M16 ? kOff16KZero : kOffKZero;
  static constexpr int kKNorm = M16 ? kOff16KNorm : kOffKNorm;
  static constexpr int kVCodes = M16 ? kOff16VCodes : kOffVCodes;
  static constexpr int kVScale = M16 ? kOff16VScale : kOffVScale;
  static constexpr int kVZero = M16 ? kOff16VZero : kOffVZero;
  static constexpr int kBytes = M16 ? kBlockBytes16 : kBlockBytes;
  static constexpr int kMeta = M16 ? 2 : 4;
};

constexpr int kWindowBytes = 2 * kGroup * kHeadDim * 2;  // K rows then V rows, bf16
constexpr int kMetaHeader = 256;                          // status words

// Largest GQA group one pass of the INT2 / bf16 decode kernels serves.
constexpr int kMaxGqa = 4;       // query heads per KV head in one launch of the BF16 reference decode
constexpr int kMaxGqaInt2 = 8;   // ... of the INT2 decode (two head sets of 4, see decode.cu)

// Bounded spin of every mbarrier wait (each try_wait may itself suspend).
constexpr uint32_t kSpinLimit = 1u << 24;
constexpr uint32_t kErrTimeout = 1u;

struct ArenaLayout {
  int64_t meta_bytes;     // header + per (slot, head) s_v maxima + per (slot, head) |z_v| maxima, 256-aligned
  int64_t zmax_off;       // the |z_v| maxima
  int64_t blocks_off;
  int64_t windows_off;
  int64_t total;
  int32_t max_groups;
};

__host__ __device__ inline ArenaLayout arena_layout(int32_t max_batch, int32_t hkv, int32_t max_len,
                                                    int32_t block_bytes = kBlockBytes) {
  ArenaLayout L;
  L.max_groups = (max_len + kGroup - 1) / kGroup;
  L.zmax_off = kMetaHeader + (int64_t)max_batch * hkv * 4;
  const int64_t meta = L.zmax_off + (int64_t)max_batch * hkv * 4;
  L.meta_bytes = (meta + 255) / 256 * 256;
  L.blocks_off = L.meta_bytes;
  int64_t blocks = (int64_t)max_batch * hkv * L.max_groups * block_bytes;
  L.windows_off = (L.blocks_off + blocks + 255) / 256 * 256;
  L.total = L.windows_off + (int64_t)max_batch * hkv * kWindowBytes;
  return L;
}

// Raise a kernel's dynamic shared-memory limit once per device (the attribute
// is per device); later launches skip the driver call.
template <typename Kernel>
inline cudaError_t ensure_smem_attr(Kernel kernel, int smem_bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` with a bounded spin.  On timeout, sets the
// CTA abort flag and the device error word; once the abort flag is set every
// later wait returns immediately so that the CTA still reaches its barriers
// and exits.  err_word may be NULL (no device status word).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  uint32_t* err_word, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  if (err_word != nullptr) atomicOr(err_word, kErrTimeout);
  return false;
}

// Wait until the producer has issued use `n` of a ring stage (issued[s] > n).
// A consumer that waits on the stage's "full" barrier for use n only after
// this point sees that barrier in phase n or n + 1, never an older phase with
// the same parity, so the parity test cannot be fooled when several consumer
// warps share a ring.
__device__ __forceinline__ bool wait_issued(const volatile uint32_t* issued, uint32_t n, volatile int* abort_flag,
                                            uint32_t* err_word, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (*issued > n) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  if (err_word != nullptr) atomicOr(err_word, kErrTimeout);
  return false;
}

// 1-D bulk copy global -> shared, completing on `bar` (bytes multiple of 16,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// D += A * B, m16n8k16, A row-major fp16, B column-major fp16, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Pack two floats into half2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float half_lo_to_float(uint32_t h2) {
  float f;
  asm("{\n\t.reg .f16 h;\n\tmov.b32 {h, _}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

__device__ __forceinline__ float half_hi_to_float(uint32_t h2) {
  float f;
  asm("{\n\t.reg .f16 h;\n\tmov.b32 {_, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// Split the pair (x0, x1) into an fp16 "hi" pair and the fp16 "lo" pair of
// the remainders; return hi when want_lo == 0, lo otherwise.  x - hi is exact
// in fp32, so hi + lo carries ~22 significant bits.
__device__ __forceinline__ uint32_t split_half2(float x0, float x1, bool want_lo) {
  uint32_t hi = pack_half2(x0, x1);
  float r0 = x0 - half_lo_to_float(hi);
  float r1 = x1 - half_hi_to_float(hi);
  uint32_t lo = pack_half2(r0, r1);
  return want_lo ? lo : hi;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7f800000u) == 0x7f800000u) return (u >> 16) | ((u & 0xffffu) ? 0x40u : 0u);  // inf / nan
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// Bit position exponent p of fragment slot i = 2*kk + hf: codes at bits
// 2i (i <= 4) are read in place; codes at i = 5..7 are read after a 10-bit
// right shift, i.e. at bits 2(i - 5).  An extracted fp16 is then the
// subnormal code * 2^(p - 24).
__host__ __device__ constexpr int frag_p(int i) { return i <= 4 ? 2 * i : 2 * (i - 5); }

// Extract the half2 (two subnormal fp16 codes) of fragment slot i from word w.
template <int I>
__device__ __forceinline__ uint32_t frag_extract(uint32_t w) {
  if constexpr (I <= 4) {
    return w & (0x00030003u << (2 * I));
  } else {
    return (w >> 10) & (0x00030003u << (2 * (I - 5)));
  }
}

// Metadata of a staged block as float: float32 sections, or float16 ones
// (converted exactly).
template <bool M16>
struct Meta {
  // elements i, i + 1 of a per-channel or per-token array
  __device__ static float2 two(const uint8_t* a, int i) {
    if constexpr (M16) {
      const uint32_t h = *reinterpret_cast<const uint32_t*>(a + 2 * i);
      return make_float2(half_lo_to_float(h), half_hi_to_float(h));
    } else {
      return *reinterpret_cast<const float2*>(a + 4 * i);
    }
  }
  __device__ static float one(const uint8_t* a, int i) {
    if constexpr (M16) {
      return half_lo_to_float(*reinterpret_cast<const uint16_t*>(a + 2 * i));
    } else {
      return reinterpret_cast<const float*>(a)[i];
    }
  }
  // the four value scales (or zeros) of token t, one per 32-channel group
  __device__ static float4 v4(const uint8_t* a, int t) {
    if constexpr (M16) {
      const uint2 h = *reinterpret_cast<const uint2*>(a + 8 * t);
      return make_float4(half_lo_to_float(h.x), half_hi_to_float(h.x), half_lo_to_float(h.y), half_hi_to_float(h.y));
    } else {
      return *reinterpret_cast<const float4*>(a + 16 * vmeta_row(t));
    }
  }
  // those of tokens t and t + 1, t even (one 16-byte load with float16 metadata)
  __device__ static void v4x2(const uint8_t* a, int t, float4& s0, float4& s1) {
    if constexpr (M16) {
      const uint4 h = *reinterpret_cast<const uint4*>(a + 8 * t);
      s0 = make_float4(half_lo_to_float(h.x), half_hi_to_float(h.x), half_lo_to_float(h.y), half_hi_to_float(h.y));
      s1 = make_float4(half_lo_to_float(h.z), half_hi_to_float(h.z), half_lo_to_float(h.w), half_hi_to_float(h.w));
    } else {
      s0 = *reinterpret_cast<const float4*>(a + 16 * vmeta_row(t));       // the pair's other row
      s1 = *reinterpret_cast<const float4*>(a + 16 * vmeta_row(t + 1));   // when bit 3 of t is set
    }
  }
};

}  // namespace oscar
