// C ABI of the OScaR INT2 KV-cache library: host-side validation, planning
// and launches.  Every argument is checked before anything is enqueued; on
// error nothing is enqueued and no host state changes.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <exception>
#include <string>
#include <mutex>
#include <vector>

#include "../../include/oscar.h"
#include "common.cuh"
#include "launch.h"

using namespace oscar;

struct oscar_cache {
  oscar_cache_config cfg;
  bool meta16;               // float16 metadata layout
  int block_bytes;
  uint8_t* arena;
  size_t arena_bytes;
  ArenaLayout layout;
  std::vector<int32_t> len;  // host mirror of every slot's length
  int sms;
  // Pre-wait copies of the decode kernel (see DecodeSeq::settled): per slot,
  // the lowest group an append may have written since the last decode call
  // (INT32_MAX: none).  Every kernel enqueued before a decode call has
  // completed by the time a later decode's main kernel starts on the same
  // stream (each kernel of the chain triggers its dependents only after its
  // own grid dependency wait), so a decode on the stream of the previous one
  // may copy the blocks of groups below that bound early.
  std::vector<int32_t> fresh_from;
  bool decoded = false;          // a decode was enqueued on last_stream
  cudaStream_t last_stream = nullptr;
};

namespace {

thread_local std::string g_err;
thread_local cudaEvent_t g_ev_start = nullptr;
thread_local cudaEvent_t g_ev_stop = nullptr;
// armed by oscar_test_arm_wait_timeout: the next INT2 decode launch on this
// thread leaves one copy unissued and gives up its waits early
thread_local bool g_arm_timeout = false;

oscar_status fail(oscar_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

oscar_status ok() {
  g_err.clear();
  return OSCAR_OK;
}

oscar_status cuda_fail(cudaError_t e, const char* what) {
  return fail(OSCAR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Makes cfg.device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != dev) {
      err = cudaSetDevice(dev);
      changed = err == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

oscar_status check_config(const oscar_cache_config* c) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "config is NULL");
  if (c->head_dim != kHeadDim) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", c->head_dim);
  if (c->group_size != kGroup) return fail(OSCAR_ERR_UNSUPPORTED, "group_size must be 128 (got %d)", c->group_size);
  if (c->value_group != kVGroup)
    return fail(OSCAR_ERR_UNSUPPORTED, "value_group must be 32 (got %d)", c->value_group);
  if (c->max_batch < 1 || c->num_kv_heads < 1 || c->max_seq_len < 1)
    return fail(OSCAR_ERR_INVALID_ARG, "max_batch, num_kv_heads and max_seq_len must be >= 1");
  if (c->device < 0) return fail(OSCAR_ERR_INVALID_ARG, "device must be >= 0");
  if (c->meta_bits != 0 && c->meta_bits != 32 && c->meta_bits != 16)
    return fail(OSCAR_ERR_UNSUPPORTED, "meta_bits must be 32 or 16 (got %d)", c->meta_bits);
  if ((int64_t)c->max_batch * c->num_kv_heads > (1 << 24))
    return fail(OSCAR_ERR_CAPACITY, "max_batch * num_kv_heads too large");
  return OSCAR_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The address the kernels use for a caller buffer, with the cache's device
// current: device or managed memory of that device as it is; page-locked host
// memory (cudaHostAlloc, cudaHostRegister) through its device mapping, which
// the kernels then read or write in place (over NVLink-C2C on Grace systems)
// instead of the caller staging copies.  Pageable host memory is refused.
oscar_status device_view(const void* ptr, const char* name, int device, const void** out, bool allow_host = true) {
  cudaPointerAttributes a;
  const cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(OSCAR_ERR_INVALID_ARG, "%s: not an address known to CUDA (%s)", name, cudaGetErrorString(e));
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
      if (a.device != device)
        return fail(OSCAR_ERR_INVALID_ARG, "%s is on device %d, the cache on device %d", name, a.device, device);
      *out = ptr;
      return OSCAR_OK;
    case cudaMemoryTypeManaged:
      if (!allow_host) return fail(OSCAR_ERR_INVALID_ARG, "%s must be device memory", name);
      *out = ptr;
      return OSCAR_OK;
    case cudaMemoryTypeHost:
      if (!allow_host) return fail(OSCAR_ERR_INVALID_ARG, "%s must be device memory", name);
      if (a.devicePointer == nullptr)
        return fail(OSCAR_ERR_INVALID_ARG, "%s: page-locked host memory not mapped for the device", name);
      *out = a.devicePointer;
      return OSCAR_OK;
    default:
      return fail(OSCAR_ERR_INVALID_ARG, "%s is pageable host memory: pass device or page-locked host memory", name);
  }
}

template <typename T>
oscar_status device_view_as(T* ptr, const char* name, int device, T** out, bool allow_host = true) {
  const void* r = nullptr;
  const oscar_status s = device_view(ptr, name, device, &r, allow_host);
  if (s == OSCAR_OK) *out = const_cast<T*>(static_cast<const T*>(r));
  return s;
}

oscar_status check_slots(const oscar_cache* c, int32_t n, const int32_t* ids, std::vector<char>& seen) {
  seen.assign(c->cfg.max_batch, 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = ids[i];
    if (s < 0 || s >= c->cfg.max_batch) return fail(OSCAR_ERR_INVALID_ARG, "seq_ids[%d] = %d out of range", i, s);
    if (seen[s]) return fail(OSCAR_ERR_INVALID_ARG, "seq_ids[%d] = %d repeated", i, s);
    seen[s] = 1;
  }
  return OSCAR_OK;
}

template <int CAP>
oscar_status run_quant_plan(oscar_cache* c, const std::vector<QuantTask>& tasks, size_t begin, size_t end,
                            const uint16_t* k, const uint16_t* v, cudaStream_t stream) {
  QuantPlan<CAP> plan;
  std::memset(&plan, 0, sizeof(plan));
  plan.n_tasks = (int32_t)(end - begin);
  plan.hkv = c->cfg.num_kv_heads;
  plan.max_groups = c->layout.max_groups;
  plan.wide = (aligned(k, 32) && aligned(v, 32)) ? 1 : 0;   // the arena's window rows are 256-byte aligned
  plan.blocks_off = c->layout.blocks_off;
  plan.windows_off = c->layout.windows_off;
  plan.zmax_off = c->layout.zmax_off;
  for (size_t i = begin; i < end; ++i) plan.t[i - begin] = pack_task(tasks[i]);
  cudaError_t e;
  if constexpr (CAP == kQuantPlanSmall)
    e = launch_quantize_small(plan, c->arena, k, v, c->meta16, stream);
  else
    e = launch_quantize_large(plan, c->arena, k, v, c->meta16, stream);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return OSCAR_OK;
}

size_t partial_bytes(int64_t slots, int gqa) { return (size_t)slots * gqa * kPartialFloats * sizeof(float); }

// Fill the per-sequence table and unit counts of one decode launch.
template <int MAXS>
void fill_decode(DecodeParams<MAXS>& P, int32_t n, const int32_t* slots, const int32_t* lens, int hkv,
                 int bf16_mode, int64_t& rows_nonempty) {
  int64_t ubase = 0;
  int32_t rank = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int len = lens[i];
    const int units = bf16_mode ? (len + 63) / 64 : len / kGroup;
    P.seq[i].slot = slots[i];
    P.seq[i].len = len;
    P.seq[i].ubase = ubase;
    P.seq[i].rank = rank;
    P.seq[i].settled = 0;
    ubase += (int64_t)hkv * units;
    if (units > 0) ++rank;
  }
  P.h.n_units = ubase;
  rows_nonempty = (int64_t)rank * hkv;
}

template <int MAXS>
oscar_status run_decode(int device, int sms, int ctas_per_sm, int32_t n, const int32_t* slots, const int32_t* lens,
                        int hkv, int hq, float scale, int bf16_mode, int max_groups, int64_t blocks_off,
                        int64_t windows_off, const uint8_t* arena, uint32_t* err_word, const uint16_t* kc,
                        const uint16_t* vc, const void* q, void* out, void* ws, size_t ws_bytes,
                        cudaStream_t stream, const void* k_new = nullptr, const void* v_new = nullptr,
                        bool meta16 = false, bool out_f32 = false, const int32_t* settled = nullptr) {
  DecodeParams<MAXS> P;
  std::memset(&P, 0, sizeof(P));
  int64_t rows = 0;
  fill_decode(P, n, slots, lens, hkv, bf16_mode, rows);
  if (settled)
    for (int32_t i = 0; i < n; ++i) P.seq[i].settled = settled[i];
  const int q_group = hq / hkv;
  const int64_t T = P.h.n_units;
  const int64_t maxN = (int64_t)sms * ctas_per_sm;
  // persistent CTAs: as many as fit (ctas_per_sm per SM), but for short caches
  // no more than one unit per consumer warp (4 per CTA): fewer partial records
  // and CTA launches (8K-token batch-1 step 15.3 -> 14.0 us)
  const int64_t N = std::min(std::min(T, maxN), (T + 3) / 4);
  const int max_gqa = bf16_mode ? kMaxGqa : kMaxGqaInt2;   // query heads per KV head in one launch
  const size_t need = partial_bytes(N + rows, q_group < max_gqa ? q_group : max_gqa);
  if (ws_bytes < need)
    return fail(OSCAR_ERR_CAPACITY, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  P.h.n_seqs = n;
  P.h.hkv = hkv;
  P.h.hq = hq;
  P.h.q_group = q_group;
  P.h.max_groups = max_groups;
  P.h.n_ctas = (int32_t)N;
  P.h.bf16_mode = bf16_mode;
  P.h.blocks_off = blocks_off;
  P.h.windows_off = windows_off;
  P.h.scale_log2 = scale * 1.4426950408889634f;
  P.h.q = static_cast<const uint16_t*>(q);
  P.h.out = static_cast<uint16_t*>(out);
  P.h.partials = static_cast<float*>(ws);
  P.h.err_word = err_word;
  P.h.k_new = static_cast<const uint16_t*>(k_new);
  P.h.v_new = static_cast<const uint16_t*>(v_new);
  P.h.out_f32 = out_f32 ? 1 : 0;
  P.h.spin_limit = kSpinLimit;
  P.h.fault_unit = -1;
  if (g_arm_timeout && !bf16_mode) {
    g_arm_timeout = false;
    P.h.spin_limit = 1u << 14;
    P.h.fault_unit = 0;
  }
  // The kernels serve at most max_gqa query heads of a KV head per launch (mma
  // columns = 4 heads x {hi, lo}; the INT2 kernel takes two such head sets on
  // the same blocks); larger groups run as consecutive passes, each streaming
  // the cache again.  A pass's main kernel writes the shared
  // workspace only after its grid dependency wait (the previous pass's
  // combine has completed), and a fused step's passes all store the same new
  // token.
  // combine staging: the longest window of the batch, and the most split-K
  // records any row has (same split as the kernels: unit u in CTA
  // ((u + 1) N - 1) / T), so that small stages let several combine CTAs share an SM
  int wrows = 0;
  int64_t max_count = 1;
  for (int32_t i = 0; i < n; ++i) {
    if (!bf16_mode) wrows = std::max(wrows, lens[i] % kGroup);
    const int64_t units = bf16_mode ? (lens[i] + 63) / 64 : lens[i] / kGroup;
    if (units == 0 || T == 0) continue;
    for (int j = 0; j < hkv; ++j) {
      const int64_t U = P.seq[i].ubase + (int64_t)j * units;
      const int64_t first = ((U + 1) * N - 1) / T, last = ((U + units) * N - 1) / T;
      max_count = std::max(max_count, last - first + 1);
    }
  }
  // Sized staging pays when the combine has more CTAs (one per row) than the
  // GPU has SMs: several then share an SM once the main grid is gone.  With
  // fewer, the full size keeps combine CTAs off SMs where a main CTA still runs
  // (measured: sharing one slows short contexts, 8K 15.3 -> 16.4 us).
  const bool pack = (int64_t)n * hkv > sms;
  P.h.comb_wrows = pack ? (wrows + 7) & ~7 : kGroup;   // multiples of 8 rows keep 16-byte alignment
  for (int head0 = 0; head0 < q_group; head0 += max_gqa) {
    P.h.gqa = q_group - head0 < max_gqa ? q_group - head0 : max_gqa;
    P.h.q_head0 = head0;
    const int64_t rec_bytes = (int64_t)P.h.gqa * kPartialFloats * 4;
    const int64_t cap = (96 * 1024) / rec_bytes;          // records of one chunk at most
    P.h.comb_part_bytes = (int32_t)((pack ? std::min(max_count, cap) : cap) * rec_bytes);
    cudaError_t e;
    if (bf16_mode)
      e = launch_decode_bf16(P, kc, vc, stream, g_ev_start, g_ev_stop);
    else
      e = launch_decode_int2(P, arena, meta16, stream, g_ev_start, g_ev_stop);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    e = launch_combine(P, arena, stream);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    // a later pass's main kernel starts after this pass's main kernel has
    // completed, and with it every kernel before it: all groups are settled
    for (int32_t i = 0; i < n; ++i) P.seq[i].settled = INT32_MAX;
  }
  (void)device;
  return OSCAR_OK;
}

}  // namespace

extern "C" {

const char* oscar_last_error(void) { return g_err.c_str(); }

oscar_status oscar_cache_required_bytes(const oscar_cache_config* cfg, size_t* out_bytes) {
  oscar_status s = check_config(cfg);
  if (s != OSCAR_OK) return s;
  if (!out_bytes) return fail(OSCAR_ERR_INVALID_ARG, "out_bytes is NULL");
  *out_bytes = (size_t)arena_layout(cfg->max_batch, cfg->num_kv_heads, cfg->max_seq_len,
                                    cfg->meta_bits == 16 ? kBlockBytes16 : kBlockBytes).total;
  return ok();
}

oscar_status oscar_cache_create(const oscar_cache_config* cfg, void* device_arena, size_t arena_bytes,
                                oscar_cache** out) {
  try {
    oscar_status s = check_config(cfg);
    if (s != OSCAR_OK) return s;
    if (!out) return fail(OSCAR_ERR_INVALID_ARG, "out is NULL");
    if (!device_arena) return fail(OSCAR_ERR_INVALID_ARG, "device_arena is NULL");
    if (!aligned(device_arena, 256)) return fail(OSCAR_ERR_INVALID_ARG, "device_arena must be 256-byte aligned");
    const bool meta16 = cfg->meta_bits == 16;
    const ArenaLayout L = arena_layout(cfg->max_batch, cfg->num_kv_heads, cfg->max_seq_len,
                                       meta16 ? kBlockBytes16 : kBlockBytes);
    if (arena_bytes < (size_t)L.total)
      return fail(OSCAR_ERR_CAPACITY, "arena too small: %zu < %lld bytes", arena_bytes, (long long)L.total);
    DeviceGuard dg(cfg->device);
    if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
    int sms = num_sms(cfg->device);
    if (sms <= 0) return fail(OSCAR_ERR_CUDA, "cannot query the SM count of device %d", cfg->device);
    cudaError_t e = cudaMemset(device_arena, 0, (size_t)L.meta_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(arena metadata)");
    oscar_cache* c = new oscar_cache;
    c->cfg = *cfg;
    c->meta16 = meta16;
    c->block_bytes = meta16 ? kBlockBytes16 : kBlockBytes;
    c->arena = static_cast<uint8_t*>(device_arena);
    c->arena_bytes = arena_bytes;
    c->layout = L;
    c->len.assign(cfg->max_batch, 0);
    c->fresh_from.assign(cfg->max_batch, 0);
    c->sms = sms;
    *out = c;
    return ok();
  } catch (const std::exception& ex) {
    return fail(OSCAR_ERR_INVALID_ARG, "host allocation failed: %s", ex.what());
  }
}

oscar_status oscar_cache_destroy(oscar_cache* cache) {
  delete cache;
  return ok();
}

oscar_status oscar_cache_reset(oscar_cache* c, int32_t seq, void* stream) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (seq < -1 || seq >= c->cfg.max_batch) return fail(OSCAR_ERR_INVALID_ARG, "seq %d out of range", seq);
  DeviceGuard dg(c->cfg.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  const int hkv = c->cfg.num_kv_heads;
  // the slot's value-scale and |value zero| maxima
  uint8_t* meta = c->arena + kMetaHeader;
  uint8_t* zmax = c->arena + c->layout.zmax_off;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (seq < 0) {
    e = cudaMemsetAsync(meta, 0, (size_t)c->cfg.max_batch * hkv * 4 * 2, st);   // both arrays, contiguous
  } else {
    e = cudaMemsetAsync(meta + (size_t)seq * hkv * 4, 0, (size_t)hkv * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(zmax + (size_t)seq * hkv * 4, 0, (size_t)hkv * 4, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(reset)");
  if (seq < 0) {
    std::fill(c->len.begin(), c->len.end(), 0);
    std::fill(c->fresh_from.begin(), c->fresh_from.end(), 0);
  } else {
    c->len[seq] = 0;
    c->fresh_from[seq] = 0;
  }
  return ok();
}

oscar_status oscar_cache_length(const oscar_cache* c, int32_t seq, int32_t* out_len) {
  if (!c || !out_len) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  if (seq < 0 || seq >= c->cfg.max_batch) return fail(OSCAR_ERR_INVALID_ARG, "seq %d out of range", seq);
  *out_len = c->len[seq];
  return ok();
}

oscar_status oscar_quantize_append(oscar_cache* c, int32_t n_seqs, const int32_t* seq_ids, const int32_t* cu_new,
                                   const void* k, const void* v, void* stream) {
  try {
    if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
    if (n_seqs < 0) return fail(OSCAR_ERR_INVALID_ARG, "n_seqs < 0");
    if (n_seqs == 0) return ok();
    if (!seq_ids || !cu_new) return fail(OSCAR_ERR_INVALID_ARG, "seq_ids / cu_new is NULL");
    std::vector<char> seen;
    oscar_status s = check_slots(c, n_seqs, seq_ids, seen);
    if (s != OSCAR_OK) return s;
    if (cu_new[0] != 0) return fail(OSCAR_ERR_INVALID_ARG, "cu_new[0] must be 0");
    for (int32_t i = 0; i < n_seqs; ++i) {
      if (cu_new[i + 1] < cu_new[i]) return fail(OSCAR_ERR_INVALID_ARG, "cu_new must be non-decreasing");
      const int64_t nl = (int64_t)c->len[seq_ids[i]] + (cu_new[i + 1] - cu_new[i]);
      if (nl > c->cfg.max_seq_len)
        return fail(OSCAR_ERR_CAPACITY, "sequence %d would reach %lld tokens > max_seq_len %d", seq_ids[i],
                    (long long)nl, c->cfg.max_seq_len);
    }
    const int32_t total = cu_new[n_seqs];
    if (total == 0) return ok();
    if (!k || !v) return fail(OSCAR_ERR_INVALID_ARG, "k / v is NULL");
    if (!aligned(k, 16) || !aligned(v, 16)) return fail(OSCAR_ERR_INVALID_ARG, "k and v must be 16-byte aligned");

    std::vector<QuantTask> tasks;
    for (int32_t i = 0; i < n_seqs; ++i) {
      const int32_t n = cu_new[i + 1] - cu_new[i];
      if (n == 0) continue;
      const int32_t slot = seq_ids[i];
      const int32_t L0 = c->len[slot];
      const int32_t L1 = L0 + n;
      const int32_t g_first = L0 / kGroup, g_end = L1 / kGroup;
      const int32_t tail_start = std::max(L0, g_end * kGroup);
      const int32_t tail_count = L1 - tail_start;
      const int32_t tail_row = cu_new[i] + (tail_start - L0);
      bool tail_done = tail_count == 0;
      for (int32_t g = g_first; g < g_end; ++g) {
        QuantTask t{};
        t.kind = 0;
        t.slot = slot;
        t.group = g;
        t.n_win = (g == g_first) ? L0 - g * kGroup : 0;
        t.in_row = cu_new[i] + (g * kGroup + t.n_win - L0);
        t.tail_count = 0;
        if (g == g_first && t.n_win > 0 && !tail_done) {
          t.tail_pos = tail_start;
          t.tail_count = tail_count;
          t.tail_in_row = tail_row;
          tail_done = true;
        }
        tasks.push_back(t);
      }
      if (!tail_done) {
        QuantTask t{};
        t.kind = 1;
        t.slot = slot;
        t.tail_pos = tail_start;
        t.tail_count = tail_count;
        t.tail_in_row = tail_row;
        tasks.push_back(t);
      }
    }
    DeviceGuard dg(c->cfg.device);
    if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
    // appended rows: device memory only
    if ((s = device_view_as(k, "k", c->cfg.device, &k, false)) != OSCAR_OK) return s;
    if ((s = device_view_as(v, "v", c->cfg.device, &v, false)) != OSCAR_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t* kp = static_cast<const uint16_t*>(k);
    const uint16_t* vp = static_cast<const uint16_t*>(v);
    for (size_t b = 0; b < tasks.size();) {
      const size_t rem = tasks.size() - b;
      if (rem <= (size_t)kQuantPlanSmall) {
        s = run_quant_plan<kQuantPlanSmall>(c, tasks, b, tasks.size(), kp, vp, st);
        b = tasks.size();
      } else {
        const size_t e = b + std::min(rem, (size_t)kQuantPlanLarge);
        s = run_quant_plan<kQuantPlanLarge>(c, tasks, b, e, kp, vp, st);
        b = e;
      }
      if (s != OSCAR_OK) return s;  // earlier chunks may already be enqueued
    }
    for (int32_t i = 0; i < n_seqs; ++i) {
      const int32_t slot = seq_ids[i];
      const int32_t L0 = c->len[slot], L1 = L0 + (cu_new[i + 1] - cu_new[i]);
      if (L1 / kGroup > L0 / kGroup) c->fresh_from[slot] = std::min(c->fresh_from[slot], L0 / kGroup);
      c->len[slot] = L1;
    }
    return ok();
  } catch (const std::exception& ex) {
    return fail(OSCAR_ERR_INVALID_ARG, "host allocation failed: %s", ex.what());
  }
}

oscar_status oscar_decode_workspace_bytes(const oscar_cache* c, int32_t n_seqs, int32_t num_q_heads,
                                          size_t* out_bytes) {
  if (!c || !out_bytes) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  if (n_seqs < 0 || num_q_heads < 1) return fail(OSCAR_ERR_INVALID_ARG, "bad n_seqs / num_q_heads");
  const int hkv = c->cfg.num_kv_heads;
  if (num_q_heads % hkv != 0) return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads must be a multiple of Hkv");
  const int64_t slots = (int64_t)c->sms * decode_int2_ctas_per_sm() + (int64_t)n_seqs * hkv;
  const int per_pass = num_q_heads / hkv < kMaxGqaInt2 ? num_q_heads / hkv : kMaxGqaInt2;   // heads per decode pass
  *out_bytes = partial_bytes(slots, per_pass);
  return ok();
}

}  // extern "C"

namespace {

// Per decoded sequence, the groups whose blocks the main kernel may copy
// before its grid dependency wait (none unless the previous decode on this
// cache ran on the same stream).
std::vector<int32_t> settled_groups(const oscar_cache* c, int32_t n, const int32_t* ids, cudaStream_t st) {
  std::vector<int32_t> r(n, 0);
  if (c->decoded && c->last_stream == st)
    for (int32_t i = 0; i < n; ++i) r[i] = c->fresh_from[ids[i]];
  return r;
}

// After a decode is enqueued: appends before it have completed when the next
// decode on this stream starts.
void note_decode(oscar_cache* c, int32_t n, const int32_t* ids, cudaStream_t st) {
  if (!(c->decoded && c->last_stream == st)) std::fill(c->fresh_from.begin(), c->fresh_from.end(), 0);
  for (int32_t i = 0; i < n; ++i) c->fresh_from[ids[i]] = INT32_MAX;
  c->decoded = true;
  c->last_stream = st;
}

// oscar_decode_attention and oscar_decode_attention_f32 (out_f32: float32 outputs).
oscar_status decode_call(oscar_cache* c, int32_t n_seqs, const int32_t* seq_ids, const void* q, int32_t num_q_heads,
                         float softmax_scale, void* out, bool out_f32, void* workspace, size_t workspace_bytes,
                         void* stream) {
  try {
    if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
    if (n_seqs < 1) return fail(OSCAR_ERR_INVALID_ARG, "n_seqs must be >= 1");
    if (n_seqs > kDecodeSeqsLarge) return fail(OSCAR_ERR_CAPACITY, "at most %d sequences per call", kDecodeSeqsLarge);
    if (!seq_ids || !q || !out || !workspace) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    const int hkv = c->cfg.num_kv_heads;
    if (num_q_heads < hkv || num_q_heads % hkv != 0)
      return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of Hkv");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16))
      return fail(OSCAR_ERR_INVALID_ARG, "q, out and workspace must be 16-byte aligned");
    if (!(softmax_scale >= 0.0f) || std::isinf(softmax_scale))
      return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
    std::vector<char> seen;
    oscar_status s = check_slots(c, n_seqs, seq_ids, seen);
    if (s != OSCAR_OK) return s;
    std::vector<int32_t> lens(n_seqs);
    for (int32_t i = 0; i < n_seqs; ++i) {
      lens[i] = c->len[seq_ids[i]];
      if (lens[i] < 1) return fail(OSCAR_ERR_INVALID_ARG, "sequence %d is empty", seq_ids[i]);
    }
    const float scale = softmax_scale == 0.0f ? 1.0f / std::sqrt((float)kHeadDim) : softmax_scale;
    DeviceGuard dg(c->cfg.device);
    if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
    if ((s = device_view_as(q, "q", c->cfg.device, &q)) != OSCAR_OK) return s;
    if ((s = device_view_as(out, "out", c->cfg.device, &out)) != OSCAR_OK) return s;
    if ((s = device_view_as(workspace, "workspace", c->cfg.device, &workspace, false)) != OSCAR_OK) return s;
    uint32_t* err_word = reinterpret_cast<uint32_t*>(c->arena);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const std::vector<int32_t> settled = settled_groups(c, n_seqs, seq_ids, st);
    if (n_seqs <= kDecodeSeqsSmall)
      s = run_decode<kDecodeSeqsSmall>(c->cfg.device, c->sms, decode_int2_ctas_per_sm(), n_seqs, seq_ids,
                                       lens.data(), hkv, num_q_heads, scale, 0, c->layout.max_groups,
                                       c->layout.blocks_off, c->layout.windows_off, c->arena, err_word, nullptr,
                                       nullptr, q, out, workspace, workspace_bytes, st, nullptr, nullptr,
                                       c->meta16, out_f32, settled.data());
    else
      s = run_decode<kDecodeSeqsLarge>(c->cfg.device, c->sms, decode_int2_ctas_per_sm(), n_seqs, seq_ids,
                                       lens.data(), hkv, num_q_heads, scale, 0, c->layout.max_groups,
                                       c->layout.blocks_off, c->layout.windows_off, c->arena, err_word, nullptr,
                                       nullptr, q, out, workspace, workspace_bytes, st, nullptr, nullptr,
                                       c->meta16, out_f32, settled.data());
    if (s != OSCAR_OK) return s;
    note_decode(c, n_seqs, seq_ids, st);
    return ok();
  } catch (const std::exception& ex) {
    return fail(OSCAR_ERR_INVALID_ARG, "host allocation failed: %s", ex.what());
  }
}

}  // namespace

extern "C" {

oscar_status oscar_decode_attention(oscar_cache* c, int32_t n_seqs, const int32_t* seq_ids, const void* q,
                                    int32_t num_q_heads, float softmax_scale, void* out, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return decode_call(c, n_seqs, seq_ids, q, num_q_heads, softmax_scale, out, false, workspace, workspace_bytes,
                     stream);
}

oscar_status oscar_decode_attention_f32(oscar_cache* c, int32_t n_seqs, const int32_t* seq_ids, const void* q,
                                        int32_t num_q_heads, float softmax_scale, void* out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  return decode_call(c, n_seqs, seq_ids, q, num_q_heads, softmax_scale, out, true, workspace, workspace_bytes,
                     stream);
}

oscar_status oscar_test_settled_groups(const oscar_cache* c, int32_t n_seqs, const int32_t* seq_ids, void* stream,
                                       int32_t* out) {
  try {
    if (!c || !seq_ids || !out) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (n_seqs < 0) return fail(OSCAR_ERR_INVALID_ARG, "n_seqs < 0");
    std::vector<char> seen;
    oscar_status s = check_slots(c, n_seqs, seq_ids, seen);
    if (s != OSCAR_OK) return s;
    const std::vector<int32_t> r = settled_groups(c, n_seqs, seq_ids, static_cast<cudaStream_t>(stream));
    for (int32_t i = 0; i < n_seqs; ++i) out[i] = r[i];
    return ok();
  } catch (const std::exception& ex) {
    return fail(OSCAR_ERR_INVALID_ARG, "host allocation failed: %s", ex.what());
  }
}

oscar_status oscar_append_decode(oscar_cache* c, int32_t n_seqs, const int32_t* seq_ids, const void* k_new,
                                 const void* v_new, const void* q, int32_t num_q_heads, float softmax_scale, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  try {
    // every argument is checked before anything is enqueued
    if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
    if (n_seqs < 1) return fail(OSCAR_ERR_INVALID_ARG, "n_seqs must be >= 1");
    if (n_seqs > kDecodeSeqsLarge) return fail(OSCAR_ERR_CAPACITY, "at most %d sequences per call", kDecodeSeqsLarge);
    if (!seq_ids || !k_new || !v_new || !q || !out || !workspace) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    const int hkv = c->cfg.num_kv_heads;
    if (num_q_heads < hkv || num_q_heads % hkv != 0)
      return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of Hkv");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16))
      return fail(OSCAR_ERR_INVALID_ARG, "k_new, v_new, q, out and workspace must be 16-byte aligned");
    if (!(softmax_scale >= 0.0f) || std::isinf(softmax_scale))
      return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
    std::vector<char> seen;
    oscar_status s = check_slots(c, n_seqs, seq_ids, seen);
    if (s != OSCAR_OK) return s;
    size_t need = 0;
    s = oscar_decode_workspace_bytes(c, n_seqs, num_q_heads, &need);
    if (s != OSCAR_OK) return s;
    if (workspace_bytes < need)
      return fail(OSCAR_ERR_CAPACITY, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    bool closes = false;
    std::vector<int32_t> lens(n_seqs);
    for (int32_t i = 0; i < n_seqs; ++i) {
      lens[i] = c->len[seq_ids[i]] + 1;
      if (lens[i] > c->cfg.max_seq_len)
        return fail(OSCAR_ERR_CAPACITY, "sequence %d would reach %d tokens > max_seq_len %d", seq_ids[i], lens[i],
                    c->cfg.max_seq_len);
      if (lens[i] % kGroup == 0) closes = true;
    }
    {
      DeviceGuard dg(c->cfg.device);
      if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
      if ((s = device_view_as(k_new, "k_new", c->cfg.device, &k_new, false)) != OSCAR_OK) return s;
      if ((s = device_view_as(v_new, "v_new", c->cfg.device, &v_new, false)) != OSCAR_OK) return s;
      if ((s = device_view_as(q, "q", c->cfg.device, &q)) != OSCAR_OK) return s;
      if ((s = device_view_as(out, "out", c->cfg.device, &out)) != OSCAR_OK) return s;
      const void* wv = nullptr;
      if ((s = device_view(workspace, "workspace", c->cfg.device, &wv, false)) != OSCAR_OK) return s;
    }
    if (closes) {
      // a group closes: it is attended quantised, so the quantiser runs first
      std::vector<int32_t> cu(n_seqs + 1);
      for (int32_t i = 0; i <= n_seqs; ++i) cu[i] = i;
      s = oscar_quantize_append(c, n_seqs, seq_ids, cu.data(), k_new, v_new, stream);
      if (s != OSCAR_OK) return s;
      return oscar_decode_attention(c, n_seqs, seq_ids, q, num_q_heads, softmax_scale, out, workspace,
                                    workspace_bytes, stream);
    }
    const float scale = softmax_scale == 0.0f ? 1.0f / std::sqrt((float)kHeadDim) : softmax_scale;
    DeviceGuard dg(c->cfg.device);
    if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
    uint32_t* err_word = reinterpret_cast<uint32_t*>(c->arena);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const std::vector<int32_t> settled = settled_groups(c, n_seqs, seq_ids, st);
    if (n_seqs <= kDecodeSeqsSmall)
      s = run_decode<kDecodeSeqsSmall>(c->cfg.device, c->sms, decode_int2_ctas_per_sm(), n_seqs, seq_ids,
                                       lens.data(), hkv, num_q_heads, scale, 0, c->layout.max_groups,
                                       c->layout.blocks_off, c->layout.windows_off, c->arena, err_word, nullptr,
                                       nullptr, q, out, workspace, workspace_bytes, st, k_new, v_new,
                                       c->meta16, false, settled.data());
    else
      s = run_decode<kDecodeSeqsLarge>(c->cfg.device, c->sms, decode_int2_ctas_per_sm(), n_seqs, seq_ids,
                                       lens.data(), hkv, num_q_heads, scale, 0, c->layout.max_groups,
                                       c->layout.blocks_off, c->layout.windows_off, c->arena, err_word, nullptr,
                                       nullptr, q, out, workspace, workspace_bytes, st, k_new, v_new,
                                       c->meta16, false, settled.data());
    if (s != OSCAR_OK) return s;
    note_decode(c, n_seqs, seq_ids, st);
    for (int32_t i = 0; i < n_seqs; ++i) c->len[seq_ids[i]] = lens[i];
    return ok();
  } catch (const std::exception& ex) {
    return fail(OSCAR_ERR_INVALID_ARG, "host allocation failed: %s", ex.what());
  }
}

// Parts the prefill splits a history of ng groups into, for CTAs of 128 rows
// over hkv KV heads on `sms` SMs (one CTA per SM): the fewest parts whose
// CTAs fill at least 95 % of their waves, with at least 8 groups a part, else
// the best fill among those; capped by the workspace (max_parts).
static int prefill_parts(int64_t rows, int hkv, int ng, int sms, int64_t max_parts) {
  if (ng < 16 || sms < 1 || max_parts < 2) return 1;
  const int64_t ctas = ((rows + 127) / 128) * hkv;
  int best = 1;
  double best_fill = 0.0;
  for (int parts = 1; parts <= 32 && parts <= ng / 8 && parts <= max_parts; ++parts) {
    const int64_t n = ctas * parts;
    const double fill = (double)n / (double)(((n + sms - 1) / sms) * sms);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = parts;
    }
    if (fill >= 0.95) break;
  }
  return best;
}

oscar_status oscar_prefill_workspace_bytes(const oscar_cache* c, int32_t seq, int32_t n_q, int32_t num_q_heads,
                                           size_t* out_bytes) {
  if (!c || !out_bytes) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  if (seq < 0 || seq >= c->cfg.max_batch) return fail(OSCAR_ERR_INVALID_ARG, "seq %d out of range", seq);
  const int hkv = c->cfg.num_kv_heads;
  if (n_q < 1 || num_q_heads < hkv || num_q_heads % hkv != 0)
    return fail(OSCAR_ERR_INVALID_ARG, "bad n_q / num_q_heads");
  const int64_t rows = (int64_t)n_q * (num_q_heads / hkv);
  const int parts = prefill_parts(rows, hkv, c->len[seq] / kGroup, num_sms(c->cfg.device), 32);
  *out_bytes = parts > 1 ? (size_t)parts * hkv * rows * kPrefillRecFloats * sizeof(float) : 0;
  return ok();
}

oscar_status oscar_prefill_attention(oscar_cache* c, int32_t seq, int32_t n_q, const void* q, int32_t num_q_heads,
                                     float softmax_scale, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (seq < 0 || seq >= c->cfg.max_batch) return fail(OSCAR_ERR_INVALID_ARG, "seq %d out of range", seq);
  if (n_q < 1) return fail(OSCAR_ERR_INVALID_ARG, "n_q must be >= 1");
  if (!q || !out) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  const int hkv = c->cfg.num_kv_heads;
  if (num_q_heads < hkv || num_q_heads % hkv != 0)
    return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of Hkv");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(workspace, 16))
    return fail(OSCAR_ERR_INVALID_ARG, "q, out and workspace must be 16-byte aligned, lse 4-byte aligned");
  if (!(softmax_scale >= 0.0f) || std::isinf(softmax_scale))
    return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  const int L = c->len[seq];
  if (L < 1) return fail(OSCAR_ERR_INVALID_ARG, "sequence %d is empty", seq);
  const int64_t rows = (int64_t)n_q * (num_q_heads / hkv);
  if (rows > (int64_t)INT32_MAX / 2) return fail(OSCAR_ERR_CAPACITY, "too many query rows");
  PrefillParams P;
  std::memset(&P, 0, sizeof(P));
  P.slot = seq;
  P.hkv = hkv;
  P.gqa = num_q_heads / hkv;
  P.hq = num_q_heads;
  P.rows = (int32_t)rows;
  P.ng = L / kGroup;
  P.wlen = L % kGroup;
  P.max_groups = c->layout.max_groups;
  P.blocks_off = c->layout.blocks_off;
  P.windows_off = c->layout.windows_off;
  P.zmax_off = c->layout.zmax_off;
  const float scale = softmax_scale == 0.0f ? 1.0f / std::sqrt((float)kHeadDim) : softmax_scale;
  P.scale_log2 = scale * 1.4426950408889634f;
  P.q = static_cast<const uint16_t*>(q);
  P.out = static_cast<uint16_t*>(out);
  P.lse = lse;
  P.err_word = reinterpret_cast<uint32_t*>(c->arena);
  DeviceGuard dg(c->cfg.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  // split the history when the workspace holds the partial records
  const size_t rec_set = (size_t)hkv * rows * kPrefillRecFloats * sizeof(float);   // one part's records
  P.n_parts = workspace != nullptr ? prefill_parts(rows, hkv, P.ng, num_sms(c->cfg.device),
                                                   (int64_t)(workspace_bytes / rec_set))
                                   : 1;
  if (P.n_parts > 1) {
    float* wd = nullptr;
    const oscar_status sw = device_view_as(static_cast<float*>(workspace), "workspace", c->cfg.device, &wd,
                                           /*allow_host=*/false);
    if (sw != OSCAR_OK) return sw;
    P.parts = wd;
  }
  {
    // q, out and lse: device or page-locked host memory (plain loads and stores)
    oscar_status sv;
    if ((sv = device_view_as(P.q, "q", c->cfg.device, &P.q)) != OSCAR_OK) return sv;
    if ((sv = device_view_as(P.out, "out", c->cfg.device, &P.out)) != OSCAR_OK) return sv;
    if (P.lse != nullptr && (sv = device_view_as(P.lse, "lse", c->cfg.device, &P.lse)) != OSCAR_OK) return sv;
  }
  cudaError_t e = launch_prefill(P, c->arena, c->meta16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return ok();
}

oscar_status oscar_cache_bytes(const oscar_cache* c, int32_t seq, int32_t kind, size_t* out_bytes) {
  if (!c || !out_bytes) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  if (kind == OSCAR_BYTES_ARENA) {
    *out_bytes = (size_t)c->layout.total;
    return ok();
  }
  if (kind != OSCAR_BYTES_USED && kind != OSCAR_BYTES_BF16_EQUIVALENT)
    return fail(OSCAR_ERR_INVALID_ARG, "unknown kind %d", kind);
  if (seq < -1 || seq >= c->cfg.max_batch) return fail(OSCAR_ERR_INVALID_ARG, "seq %d out of range", seq);
  const int hkv = c->cfg.num_kv_heads;
  size_t total = 0;
  for (int32_t s = (seq < 0 ? 0 : seq); s < (seq < 0 ? c->cfg.max_batch : seq + 1); ++s) {
    const int64_t L = c->len[s];
    if (kind == OSCAR_BYTES_USED)
      total += (size_t)hkv * ((L / kGroup) * (int64_t)c->block_bytes + (L % kGroup) * 2 * kHeadDim * 2);
    else
      total += (size_t)hkv * L * 2 * kHeadDim * 2;
  }
  *out_bytes = total;
  return ok();
}

oscar_status oscar_cache_block_offset(const oscar_cache* c, int32_t seq, int32_t kv_head, int32_t group,
                                      size_t* out_offset) {
  if (!c || !out_offset) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  if (seq < 0 || seq >= c->cfg.max_batch || kv_head < 0 || kv_head >= c->cfg.num_kv_heads || group < 0 ||
      group >= c->layout.max_groups)
    return fail(OSCAR_ERR_INVALID_ARG, "index out of range");
  *out_offset = (size_t)(c->layout.blocks_off +
                         (((int64_t)seq * c->cfg.num_kv_heads + kv_head) * c->layout.max_groups + group) *
                             (int64_t)c->block_bytes);
  return ok();
}

oscar_status oscar_cache_window_offset(const oscar_cache* c, int32_t seq, int32_t kv_head, size_t* out_offset) {
  if (!c || !out_offset) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  if (seq < 0 || seq >= c->cfg.max_batch || kv_head < 0 || kv_head >= c->cfg.num_kv_heads)
    return fail(OSCAR_ERR_INVALID_ARG, "index out of range");
  *out_offset = (size_t)(c->layout.windows_off + ((int64_t)seq * c->cfg.num_kv_heads + kv_head) * kWindowBytes);
  return ok();
}

oscar_status oscar_cache_check(oscar_cache* c, void* stream) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  DeviceGuard dg(c->cfg.device);
  if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, c->arena, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  if (word != 0) {
    cudaMemset(c->arena, 0, 4);
    return fail(OSCAR_ERR_DEVICE_TIMEOUT, "a kernel wait timed out (flags 0x%x)", word);
  }
  return ok();
}

oscar_status oscar_bf16_decode_workspace_bytes(int32_t n_seqs, int32_t num_kv_heads, int32_t num_q_heads,
                                               size_t* out_bytes) {
  if (!out_bytes || n_seqs < 0 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0)
    return fail(OSCAR_ERR_INVALID_ARG, "bad arguments");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const int sms = num_sms(dev);
  if (sms <= 0) return fail(OSCAR_ERR_CUDA, "cannot query the SM count");
  const int64_t slots = (int64_t)sms * decode_bf16_ctas_per_sm() + (int64_t)n_seqs * num_kv_heads;
  const int per_pass = num_q_heads / num_kv_heads < kMaxGqa ? num_q_heads / num_kv_heads : kMaxGqa;
  *out_bytes = partial_bytes(slots, per_pass);
  return ok();
}

oscar_status oscar_bf16_decode_attention(int32_t n_seqs, const int32_t* seq_ids, const int32_t* seq_lens,
                                         const void* k_cache, const void* v_cache, int32_t num_kv_heads,
                                         int32_t max_seq_len, const void* q, int32_t num_q_heads,
                                         float softmax_scale, void* out, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  try {
    if (n_seqs < 1) return fail(OSCAR_ERR_INVALID_ARG, "n_seqs must be >= 1");
    if (n_seqs > kDecodeSeqsLarge) return fail(OSCAR_ERR_CAPACITY, "at most %d sequences per call", kDecodeSeqsLarge);
    if (!seq_ids || !seq_lens || !k_cache || !v_cache || !q || !out || !workspace)
      return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
    if (num_kv_heads < 1 || max_seq_len < 1) return fail(OSCAR_ERR_INVALID_ARG, "bad num_kv_heads / max_seq_len");
    if (num_q_heads < num_kv_heads || num_q_heads % num_kv_heads != 0)
      return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of Hkv");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(workspace, 16))
      return fail(OSCAR_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    if (!(softmax_scale >= 0.0f) || std::isinf(softmax_scale))
      return fail(OSCAR_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
    for (int32_t i = 0; i < n_seqs; ++i) {
      if (seq_ids[i] < 0) return fail(OSCAR_ERR_INVALID_ARG, "seq_ids[%d] < 0", i);
      if (seq_lens[i] < 1 || seq_lens[i] > max_seq_len)
        return fail(OSCAR_ERR_INVALID_ARG, "seq_lens[%d] = %d outside [1, max_seq_len]", i, seq_lens[i]);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const int sms = num_sms(dev);
    if (sms <= 0) return fail(OSCAR_ERR_CUDA, "cannot query the SM count");
    const float scale = softmax_scale == 0.0f ? 1.0f / std::sqrt((float)kHeadDim) : softmax_scale;
    // the caches are read with tensor copies (device memory only); q and out
    // may be page-locked host memory as for oscar_decode_attention
    oscar_status sv;
    if ((sv = device_view_as(k_cache, "k_cache", dev, &k_cache, false)) != OSCAR_OK) return sv;
    if ((sv = device_view_as(v_cache, "v_cache", dev, &v_cache, false)) != OSCAR_OK) return sv;
    if ((sv = device_view_as(q, "q", dev, &q)) != OSCAR_OK) return sv;
    if ((sv = device_view_as(out, "out", dev, &out)) != OSCAR_OK) return sv;
    if ((sv = device_view_as(workspace, "workspace", dev, &workspace, false)) != OSCAR_OK) return sv;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t* kc = static_cast<const uint16_t*>(k_cache);
    const uint16_t* vc = static_cast<const uint16_t*>(v_cache);
    oscar_status s;
    if (n_seqs <= kDecodeSeqsSmall)
      s = run_decode<kDecodeSeqsSmall>(dev, sms, decode_bf16_ctas_per_sm(), n_seqs, seq_ids, seq_lens,
                                       num_kv_heads, num_q_heads, scale, 1, max_seq_len, 0, 0, nullptr, nullptr, kc,
                                       vc, q, out, workspace, workspace_bytes, st);
    else
      s = run_decode<kDecodeSeqsLarge>(dev, sms, decode_bf16_ctas_per_sm(), n_seqs, seq_ids, seq_lens,
                                       num_kv_heads, num_q_heads, scale, 1, max_seq_len, 0, 0, nullptr, nullptr, kc,
                                       vc, q, out, workspace, workspace_bytes, st);
    if (s != OSCAR_OK) return s;
    return ok();
  } catch (const std::exception& ex) {
    return fail(OSCAR_ERR_INVALID_ARG, "host allocation failed: %s", ex.what());
  }
}

// ------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they decode:
// code running inside a memory pool or arena it does not own, plugins whose
// host framework forbids allocation on the serving path, and callers that
// must keep a fixed device footprint.  For them the split-K partials live in
// a fixed file-scope device array instead of a workspace argument.  Every GPU
// that loads this library holds the array until the process exits.
constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
// In host code the array's name is only a host-side stand-in; the address
// that kernels may use is looked up once per device and remembered.
oscar_status noalloc_scratch(int device, void** out) {
  if (device < 0 || device >= kNoAllocMaxDevices)
    return fail(OSCAR_ERR_UNSUPPORTED, "device %d beyond the %d supported", device, kNoAllocMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[device] == nullptr) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
    g_noalloc_ptr[device] = ptr;
  }
  *out = g_noalloc_ptr[device];
  return OSCAR_OK;
}
}  // namespace

oscar_status oscar_decode_attention_noalloc(oscar_cache* c, int32_t n_seqs, const int32_t* seq_ids, const void* q,
                                            int32_t num_q_heads, float softmax_scale, void* out, void* stream) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (n_seqs < 1) return fail(OSCAR_ERR_INVALID_ARG, "n_seqs must be >= 1");
  const int hkv = c->cfg.num_kv_heads;
  if (num_q_heads < hkv || num_q_heads % hkv != 0)
    return fail(OSCAR_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of Hkv");
  size_t need = 0;
  oscar_status s = oscar_decode_workspace_bytes(c, n_seqs, num_q_heads, &need);
  if (s != OSCAR_OK) return s;
  if (need > kNoAllocScratchBytes)
    return fail(OSCAR_ERR_CAPACITY,
                "decode of %d sequences x %d query heads needs %zu bytes of partials, more than the %zu-byte "
                "built-in scratch; use oscar_decode_attention with a workspace",
                n_seqs, num_q_heads, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  {
    DeviceGuard dg(c->cfg.device);
    if (dg.err != cudaSuccess) return cuda_fail(dg.err, "cudaSetDevice");
    s = noalloc_scratch(c->cfg.device, &scratch);
    if (s != OSCAR_OK) return s;
  }
  return oscar_decode_attention(c, n_seqs, seq_ids, q, num_q_heads, softmax_scale, out, scratch,
                                kNoAllocScratchBytes, stream);
}

oscar_status oscar_test_arm_wait_timeout(void) {
  g_arm_timeout = true;
  return ok();
}

oscar_status oscar_set_timing_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(OSCAR_ERR_INVALID_ARG, "pass both events or neither");
  g_ev_start = static_cast<cudaEvent_t>(start_event);
  g_ev_stop = static_cast<cudaEvent_t>(stop_event);
  return ok();
}

}  // extern "C"
