// Host-side launch interface between the C ABI (oscar_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace oscar {

// One 128-token group of one sequence that fills during an append (all KV
// heads run it, grid.y = head).  Tokens 0..n_win-1 of the group come from
// the window, the rest from input rows in_row, in_row + 1, ...  When
// tail_count > 0 the same CTA afterwards writes input rows tail_in_row ...
// into window positions tail_pos ... (the window it has just read).
struct QuantTask {
  int32_t slot;
  int32_t group;
  int32_t n_win;
  int32_t in_row;
  int32_t tail_pos;
  int32_t tail_count;
  int32_t tail_in_row;
  int32_t kind;  // 0 = quantise a group (+ optional tail), 1 = window append only
};

// A QuantTask as the kernel reads it, 16 bytes, so that a whole 128K-token
// append (1,024 tasks) fits in one launch's parameters:
//   a = slot | n_win << 24 | kind << 31   (kind 1: the n_win bits hold
//                                          tail_pos mod 128)
//   b = group | tail_count << 24
//   c = in_row, d = tail_in_row
// A kind-0 task's tail always starts on a group boundary (tail_pos mod 128
// = 0).  slot and group are below 2^24 (max_batch * Hkv <= 2^24; groups of
// an int32 length), n_win and tail_count below 128.
struct PackedTask {
  uint32_t a, b;
  int32_t c, d;
  __host__ __device__ int slot() const { return (int)(a & 0xFFFFFFu); }
  __host__ __device__ int kind() const { return (int)(a >> 31); }
  __host__ __device__ int n_win() const { return kind() ? 0 : (int)((a >> 24) & 0x7Fu); }
  __host__ __device__ int tail_pos_mod() const { return kind() ? (int)((a >> 24) & 0x7Fu) : 0; }
  __host__ __device__ int group() const { return (int)(b & 0xFFFFFFu); }
  __host__ __device__ int tail_count() const { return (int)((b >> 24) & 0x7Fu); }
  __host__ __device__ int in_row() const { return c; }
  __host__ __device__ int tail_in_row() const { return d; }
};
static_assert(sizeof(PackedTask) == 16, "16-byte tasks");

inline PackedTask pack_task(const QuantTask& t) {
  PackedTask p;
  const uint32_t low7 = (uint32_t)(t.kind ? (t.tail_pos & 127) : t.n_win) & 0x7Fu;
  p.a = ((uint32_t)t.slot & 0xFFFFFFu) | (low7 << 24) | ((uint32_t)(t.kind & 1) << 31);
  p.b = ((uint32_t)(t.kind ? 0 : t.group) & 0xFFFFFFu) | (((uint32_t)t.tail_count & 0x7Fu) << 24);
  p.c = t.in_row;
  p.d = t.tail_in_row;
  return p;
}

constexpr int kQuantPlanSmall = 64;
constexpr int kQuantPlanLarge = 2000;   // 32 + 2000 * 16 bytes of plan: within the 32,764-byte parameter limit

template <int CAP>
struct QuantPlan {
  int32_t n_tasks;
  int32_t hkv;
  int32_t max_groups;
  int32_t wide;          // 1: k and v are 32-byte aligned (32-byte row loads)
  int64_t blocks_off;
  int64_t windows_off;
  int64_t zmax_off;      // per (slot, head) largest |value zero| (float bits, atomicMax)
  PackedTask t[CAP];
};
static_assert(sizeof(QuantPlan<kQuantPlanLarge>) + 3 * sizeof(void*) <= 32764, "kernel parameter limit");

// meta16: the float16-metadata block layout (see include/oscar.h)
cudaError_t launch_quantize_small(const QuantPlan<kQuantPlanSmall>& plan, uint8_t* arena, const uint16_t* k,
                                  const uint16_t* v, bool meta16, cudaStream_t stream);
cudaError_t launch_quantize_large(const QuantPlan<kQuantPlanLarge>& plan, uint8_t* arena, const uint16_t* k,
                                  const uint16_t* v, bool meta16, cudaStream_t stream);

// ------------------------------------------------------------------ decode

// Per-sequence data of one decode launch.  Work units are (sequence, KV head,
// unit) triples in that order (a unit is one 128-token group of the INT2
// cache, or one 64-token tile of the bf16 reference cache); sequence b owns
// units [ubase, ubase + hkv * units_b).
struct DecodeSeq {
  int32_t slot;
  int32_t len;
  int64_t ubase;  // first unit of this sequence
  int32_t rank;   // number of earlier sequences with >= 1 unit
  // INT2: groups 0..settled-1 of each of this sequence's rows were written by
  // kernels that have completed before this launch can start (the host tracks
  // appends), so their blocks may be copied before the grid dependency wait
  int32_t settled;
};

struct DecodeHeader {
  int32_t n_seqs;
  int32_t hkv;
  int32_t gqa;           // query heads of each KV head served by this launch (<= kMaxGqa BF16, kMaxGqaInt2 INT2)
  int32_t hq;
  int32_t max_groups;    // INT2: groups per (slot, head); bf16: max_seq_len
  int32_t n_ctas;        // main-kernel CTAs (N)
  int32_t bf16_mode;     // 1: bf16 reference cache (64-token units, no window)
  int32_t q_group;       // query heads per KV head in the q / out layout (hq / hkv >= gqa)
  int64_t n_units;       // T
  int64_t blocks_off;
  int64_t windows_off;
  float scale_log2;      // softmax_scale * log2(e)
  int32_t q_head0;       // this launch's first query head within each KV head's group
  const uint16_t* q;
  uint16_t* out;
  float* partials;
  uint32_t* err_word;
  // fused append: when set, each (sequence, KV head) row's newest window
  // token (window row len mod 128 - 1) is taken from these [n_seqs, hkv, d]
  // bf16 rows instead of the arena, and stored into the arena window
  const uint16_t* k_new;
  const uint16_t* v_new;
  // combine staging, sized by the host for this launch: window rows (the
  // longest window of the batch) and bytes of partial records per chunk
  int32_t comb_wrows;
  int32_t comb_part_bytes;
  int32_t out_f32;       // the combine writes float32 outputs (else bf16)
  // bounded waits of the INT2 main kernel give up after this many polls; a
  // test of that path sets fault_unit >= 0: CTA 0's producer then leaves that
  // unit's copy unissued (its consumer's wait runs out), and a small limit
  uint32_t spin_limit;
  int32_t fault_unit;
};

template <int MAXS>
struct DecodeParams {
  DecodeHeader h;
  DecodeSeq seq[MAXS];
};

constexpr int kDecodeSeqsSmall = 16;
constexpr int kDecodeSeqsLarge = 1024;

// Floats of one partial record (o[128], m, l, 2 pad) per query head.
constexpr int kPartialFloats = 132;

// ----------------------------------------------------------------- prefill

// One chunked-prefill attention launch: n_q queries of one sequence against
// every token in its cache.  Rows are (query, head) pairs, query-major.
struct PrefillParams {
  int32_t slot;
  int32_t hkv;
  int32_t gqa;
  int32_t hq;
  int32_t rows;          // n_q * gqa (per KV head)
  int32_t ng;            // full groups in the cache
  int32_t wlen;          // window tokens
  int32_t max_groups;
  int64_t blocks_off;
  int64_t windows_off;
  int64_t zmax_off;      // per (slot, head) largest |value zero| quantised so far (float bits)
  float scale_log2;      // softmax_scale * log2(e)
  int32_t n_parts;       // the groups are split into this many parts (grid.z); 1: no split
  const uint16_t* q;     // [n_q, hq, d] bf16
  uint16_t* out;         // [n_q, hq, d] bf16
  float* lse;            // [n_q, hq] fp32 natural-log log-sum-exp, or NULL
  uint32_t* err_word;
  // n_parts > 1: partial records [part][KV head][row][kPrefillRecFloats]
  // (o unnormalised = sum p v, then m in log2 units and l), merged by a
  // second kernel
  float* parts;
};

// Floats of one partial prefill record (o[128], m, l, 2 pad).
constexpr int kPrefillRecFloats = 132;

cudaError_t launch_prefill(const PrefillParams& p, const uint8_t* arena, bool meta16, cudaStream_t stream);
// the tcgen05 history kernel (prefill_tc.cu); launch_prefill adds the merge of split parts
cudaError_t launch_prefill_tc(const PrefillParams& p, const uint8_t* arena, bool meta16, cudaStream_t stream);

int num_sms(int device);
int decode_int2_ctas_per_sm();
int decode_bf16_ctas_per_sm();

template <int MAXS>
cudaError_t launch_decode_int2(const DecodeParams<MAXS>& p, const uint8_t* arena, bool meta16, cudaStream_t stream,
                               cudaEvent_t ev_start, cudaEvent_t ev_stop);
template <int MAXS>
cudaError_t launch_decode_bf16(const DecodeParams<MAXS>& p, const uint16_t* kc, const uint16_t* vc,
                               cudaStream_t stream, cudaEvent_t ev_start, cudaEvent_t ev_stop);
template <int MAXS>
cudaError_t launch_combine(const DecodeParams<MAXS>& p, const uint8_t* arena, cudaStream_t stream);

}  // namespace oscar
