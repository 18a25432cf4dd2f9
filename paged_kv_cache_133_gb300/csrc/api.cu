// C ABI entry points: host-side validation, workspace sizing and dispatch.
// Nothing here allocates device memory or synchronises with the device.
#include <math.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "pa.h"

namespace pa {

static std::atomic<uint64_t> g_launches{0};
static thread_local int g_last_cuda_error = 0;
// Limit of the tensor-core kernels' pipeline waits (pa_set_wait_limit_ns; 0: default)
static std::atomic<uint64_t> g_wait_ns{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int device_num_sms() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

// Per-device side stream and fork/join events for running the decode rows
// concurrently with the persistent prefill kernel.  Created once per device;
// no device memory.
// Streams for a mixed step: the prefill on `hi` (highest priority, so that
// when both kernels become ready at once the block scheduler places the
// persistent prefill CTAs first) and the decode on `lo`, both forked from and
// joined back into the caller's stream.  Without the priority, back-to-back
// steps sometimes let the decode grid fill every SM first and starve the
// prefill (measured 1.22 against 0.92 ms on the mixed workload).
struct SideStream {
  int least = 0, greatest = 0;  // stream priority range of the device
  cudaStream_t hi = nullptr, lo = nullptr;
  cudaEvent_t fork = nullptr, join_hi = nullptr, join_lo = nullptr;
  bool ready = false;
};
static SideStream g_side[64];
static std::mutex g_side_mu;

static SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& s = g_side[dev];
  if (!s.ready) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithPriority(&s.hi, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&s.lo, cudaStreamNonBlocking, least) != cudaSuccess)
      return nullptr;
    if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.join_hi, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.join_lo, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    s.least = least;
    s.greatest = greatest;
    s.ready = true;
  }
  return &s;
}

// SMs given to the decode rows while the prefill kernel runs beside them:
// PA_MIXED_DECODE_SMS overrides, else 84 of every 152 SMs (the best of a
// sweep on the mixed workload, 240 decode rows beside two 3976-token chunks:
// 40 .. 96 decode SMs gave 0.894, 0.868, 0.841, 0.799, 0.800 (80), 0.780
// (84), 0.829 (88), 0.886 (92) and 0.954 ms (96)).
static int mixed_decode_sms(int num_sms) {
  const char* env = getenv("PA_MIXED_DECODE_SMS");
  if (env) {
    const int v = atoi(env);
    if (v <= 0) return 0;
    return v < num_sms - 1 ? v : num_sms - 1;
  }
  return (num_sms * 84 + 76) / 152;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PA_OK;
  g_last_cuda_error = static_cast<int>(e);
  return PA_ERR_CUDA;
}

int record_cuda_error(cudaError_t e) { return e == cudaSuccess ? PA_OK : cuda_status(e); }

static int ilog2_exact(int x) {
  if (x <= 0 || (x & (x - 1))) return -1;
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// Workspace = kWorkspaceHeader bytes (prefill work-queue counter) followed by
// the split-KV decode partials, when the decode rows are split.
static size_t decode_workspace(int num_decode, int hq, int hkv, int head_dim, int max_seq_len,
                               int* part, int* nsplit) {
  *part = 64;
  *nsplit = 1;
  if (num_decode <= 0 || hkv <= 0 || hq <= 0 || hq % hkv || max_seq_len <= 0) return 0;
  const int group = hq / hkv;
  const int units = hkv * ((group + 15) / 16);
  decode_partition(num_decode, units, max_seq_len, device_num_sms(), part, nsplit);
  if (*nsplit <= 1) return 0;
  return static_cast<size_t>(*nsplit) * num_decode * hq * (head_dim + 2) * sizeof(float);
}

// Cascade: suffix splits over the longest own-key range and prefix chunks;
// partials of both for every (decode sequence, query head).
static size_t cascade_workspace(int num_decode, int hq, int hkv, int head_dim, int max_seq_len,
                                int prefix_len, bool tc, int* part, int* nsplit, int* part_p,
                                int* nsplit_p) {
  *part = 64;
  *nsplit = 1;
  *part_p = 64;
  *nsplit_p = 0;
  if (num_decode <= 0 || hkv <= 0 || hq <= 0 || hq % hkv || prefix_len <= 0 ||
      max_seq_len <= prefix_len)
    return 0;
  const int group = hq / hkv;
  const int units = hkv * ((group + 15) / 16);
  // the own keys run after the prefix pass has filled the GPU: about one wave
  // of CTAs (a quarter of the SMs' worth of the usual split target)
  decode_partition(num_decode, units, max_seq_len - prefix_len, (device_num_sms() + 3) / 4, part,
                   nsplit);
  cascade_partition(num_decode, hq, hkv, prefix_len, device_num_sms(), tc, part_p, nsplit_p);
  return static_cast<size_t>(*nsplit + *nsplit_p) * num_decode * hq * (head_dim + 2) *
         sizeof(float);
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    default: return "PA_ERR_UNKNOWN";
  }
}

int pa_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t pa_set_wait_limit_ns(uint64_t ns) { return g_wait_ns.exchange(ns); }

uint64_t pa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int pa_write_kv(const void* k, const void* v, int64_t k_stride_t, int64_t v_stride_t,
                void* k_cache, void* v_cache, const int32_t* slot_mapping, int num_tokens,
                int num_blocks, int block_size, int num_kv_heads, int head_dim,
                uint32_t* err_flag, void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (!k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!k || !v || !slot_mapping)) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row % 8 || k_stride_t % 8 || v_stride_t % 8 || k_stride_t < row || v_stride_t < row)
    return PA_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache) || (num_tokens > 0 && (!aligned16(k) || !aligned16(v))))
    return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  return cuda_status(launch_write_kv(k, v, k_stride_t, v_stride_t, k_cache, v_cache, slot_mapping,
                                     num_tokens, num_blocks, block_size, static_cast<int>(row),
                                     err_flag, static_cast<cudaStream_t>(stream)));
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                   int num_blocks, int block_size, int num_kv_heads, int head_dim,
                   uint32_t* err_flag, void* stream) {
  if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || (num_pairs > 0 && !pairs)) return PA_ERR_INVALID_ARG;
  if (num_pairs > 65535) return PA_ERR_UNSUPPORTED;
  const int64_t elems = static_cast<int64_t>(block_size) * num_kv_heads * head_dim;
  if (elems % 8 || elems > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  return cuda_status(launch_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_blocks,
                                        static_cast<int>(elems), err_flag,
                                        static_cast<cudaStream_t>(stream)));
}

// The address a kernel on the current device uses for `p`, or nullptr when the
// device cannot reach it: device and managed memory as is, page-locked host
// memory through its mapped device address, other host memory only where the
// device reads pageable memory coherently.
static const void* device_view(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return at.devicePointer;
    default: {
      int dev = 0, pageable = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess)
        return nullptr;
      return pageable ? p : nullptr;
    }
  }
}

int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                   const int32_t* pairs, int num_pairs, int src_num_blocks, int dst_num_blocks,
                   int block_size, int num_kv_heads, int head_dim, uint32_t* err_flag,
                   void* stream) {
  if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_size <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (!src_k || !src_v || !dst_k || !dst_v || (num_pairs > 0 && !pairs)) return PA_ERR_INVALID_ARG;
  if (num_pairs > 65535) return PA_ERR_UNSUPPORTED;
  const int64_t elems = static_cast<int64_t>(block_size) * num_kv_heads * head_dim;
  if (elems % 8 || elems > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
    return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  const void* sk = device_view(src_k);
  const void* sv = device_view(src_v);
  const void* dk = device_view(dst_k);
  const void* dv = device_view(dst_v);
  if (!sk || !sv || !dk || !dv) return PA_ERR_INVALID_ARG;
  return cuda_status(launch_swap_blocks(sk, sv, const_cast<void*>(dk), const_cast<void*>(dv), pairs,
                                        num_pairs, src_num_blocks, dst_num_blocks,
                                        static_cast<int>(elems), err_flag,
                                        static_cast<cudaStream_t>(stream)));
}

size_t pa_attention_workspace_size(int num_decode_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int max_seq_len) {
  int part, nsplit;
  return kWorkspaceHeader + decode_workspace(num_decode_seqs, num_q_heads, num_kv_heads, head_dim,
                                             max_seq_len, &part, &nsplit);
}

// The new tokens' K/V and their slots, for the fused scatter + attention.
struct FusedIn {
  const void* k;
  const void* v;
  int64_t k_stride, v_stride;
  const int32_t* slots;
};

static int attention_impl(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                          const void* k_cache, const void* v_cache,
                          const int32_t* query_start_loc, const int32_t* seq_lens,
                          const int32_t* block_tables, int num_seqs, int num_tokens,
                          int max_blocks_per_seq, int num_decode_seqs, int max_query_len,
                          int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int num_blocks, float scale, void* workspace,
                          size_t workspace_bytes, uint32_t* err_flag, void* stream,
                          const FusedIn* fused, const float* kv_scales = nullptr,
                          int prefix_blocks = 0) {
  if (num_seqs < 0 || num_tokens < 0 || num_decode_seqs < 0 || num_decode_seqs > num_seqs ||
      max_query_len < 0 || max_seq_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  const int bs_log2 = ilog2_exact(block_size);
  if (bs_log2 < 0 || block_size > 256) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_tokens == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !query_start_loc || !seq_lens || !block_tables)
    return PA_ERR_INVALID_ARG;
  if (q_stride_t % 8 || out_stride_t % 8 ||
      q_stride_t < static_cast<int64_t>(num_q_heads) * head_dim ||
      out_stride_t < static_cast<int64_t>(num_q_heads) * head_dim)
    return PA_ERR_UNSUPPORTED;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  const int64_t hunits = static_cast<int64_t>(num_kv_heads) * ((group + 15) / 16);
  if (num_decode_seqs > 65535 || num_seqs - num_decode_seqs > 65535 || hunits > 65535)
    return PA_ERR_UNSUPPORTED;

  AttnArgs a{};
  a.inv_v_scale = 1.f;
  a.out = out;
  a.out_stride = out_stride_t;
  a.q = q;
  a.q_stride = q_stride_t;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.qsl = query_start_loc;
  a.seq_lens = seq_lens;
  a.block_tables = block_tables;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_blocks = max_blocks_per_seq;
  a.num_decode = num_decode_seqs;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.group = group;
  a.head_dim = head_dim;
  a.bs_log2 = bs_log2;
  a.num_blocks = num_blocks;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = err_flag;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  size_t decode_need = 0;
  if (prefix_blocks < 0) return PA_ERR_INVALID_ARG;
  if (prefix_blocks > 0) {
    // Shared-prefix decode: decode rows only, bf16 cache, no fused scatter.
    if (num_decode_seqs != num_seqs || fused || kv_scales) return PA_ERR_UNSUPPORTED;
    const int64_t plen = static_cast<int64_t>(prefix_blocks) * block_size;
    if (prefix_blocks > max_blocks_per_seq || plen >= max_seq_len) return PA_ERR_INVALID_ARG;
    a.cascade = true;
    a.prefix_len = static_cast<int>(plen);
    a.key_begin = a.prefix_len;
    a.casc_tc = cascade_tc_supported(a);
    decode_need = cascade_workspace(num_decode_seqs, num_q_heads, num_kv_heads, head_dim,
                                    max_seq_len, a.prefix_len, a.casc_tc, &a.part, &a.nsplit,
                                    &a.part_prefix, &a.nsplit_prefix);
    a.split0 = a.nsplit_prefix;
  } else if (num_decode_seqs > 0 && max_seq_len > 0) {
    decode_need = decode_workspace(num_decode_seqs, num_q_heads, num_kv_heads, head_dim,
                                   max_seq_len, &a.part, &a.nsplit);
  }
  if (!workspace || workspace_bytes < kWorkspaceHeader + decode_need ||
      (reinterpret_cast<uintptr_t>(workspace) & 15u))
    return PA_ERR_WORKSPACE;
  a.sched = static_cast<unsigned long long*>(workspace);
  if (decode_need > 0) {
    a.ws_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + kWorkspaceHeader);
    a.ws_ml = a.ws_o + static_cast<size_t>(a.nsplit + a.nsplit_prefix) * num_decode_seqs *
                           num_q_heads * head_dim;
  }
  const bool has_decode = num_decode_seqs > 0 && max_seq_len > 0;
  const bool has_prefill = num_seqs > num_decode_seqs && max_query_len > 0;
  if (kv_scales) {  // 8-bit cache: decode rows only
    if (has_prefill) return PA_ERR_UNSUPPORTED;
    a.kv_fp8 = true;
    a.scale_log2 *= kv_scales[0];
    a.inv_v_scale = 1.f / kv_scales[1];
  }
  if (fused) {
    if (has_decode || (has_prefill && !prefill_tc_supported(a))) {
      // Steps with decode rows (which run beside the prefill and read every
      // key from the cache) and steps the general prefill kernel takes:
      // scatter first, then attend.  Folding the scatter into a prefill that
      // shares the GPU with an HBM-bound decode measured slower.
      const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
      const int rc = cuda_status(launch_write_kv(fused->k, fused->v, fused->k_stride,
                                                 fused->v_stride, const_cast<void*>(k_cache),
                                                 const_cast<void*>(v_cache), fused->slots,
                                                 num_tokens, num_blocks, block_size,
                                                 static_cast<int>(row), err_flag, st));
      if (rc != PA_OK) return rc;
    } else if (has_prefill) {
      // Prefill-only step on the tensor-core path: it reads the new tokens'
      // K/V from k, v and stores them into their slots itself.
      a.k_new = fused->k;
      a.v_new = fused->v;
      a.kn_stride = fused->k_stride;
      a.vn_stride = fused->v_stride;
      a.slots = fused->slots;
    }
  }
  // Mixed step: the decode rows are HBM-bound and the tensor-core prefill is
  // bound by its softmax and issue chain, so they run side by side: the
  // persistent prefill kernel takes all but mixed_decode_sms() SMs on a
  // high-priority side stream and the decode launches on a low-priority one
  // (fork/join with events, which CUDA graph capture also records).
  const int reserve = has_decode && has_prefill && prefill_tc_supported(a)
                          ? mixed_decode_sms(device_num_sms())
                          : 0;
  if (reserve > 0) {
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream* side = side_stream();
    if (side) {
      // One small operation on the caller's stream before the fork, so that
      // in a captured graph both kernels hang off one node and become ready
      // together and the priorities decide.  Without it (the fork right
      // after the previous step's join) the decode grid filled the SMs first
      // and the step took 1.18 instead of 0.81 ms; a memset on the prefill
      // side alone had the same effect.  The memset clears the work-queue
      // word, which the prefill kernel would otherwise reset itself.
      if (cudaMemsetAsync(a.sched, 0, sizeof(unsigned long long), st) != cudaSuccess)
        return cuda_status(cudaGetLastError());
      if (cudaEventRecord(side->fork, st) != cudaSuccess ||
          cudaStreamWaitEvent(side->hi, side->fork, 0) != cudaSuccess ||
          cudaStreamWaitEvent(side->lo, side->fork, 0) != cudaSuccess)
        return cuda_status(cudaGetLastError());
      a.max_ctas = device_num_sms() - reserve;
      a.has_priority = true;
      a.priority = side->greatest;
      int rc = cuda_status(launch_prefill(a, side->hi));
      if (rc != PA_OK) return rc;
      a.priority = side->least;
      rc = cuda_status(launch_decode(a, side->lo));
      if (rc != PA_OK) return rc;
      if (cudaEventRecord(side->join_hi, side->hi) != cudaSuccess ||
          cudaEventRecord(side->join_lo, side->lo) != cudaSuccess ||
          cudaStreamWaitEvent(st, side->join_hi, 0) != cudaSuccess ||
          cudaStreamWaitEvent(st, side->join_lo, 0) != cudaSuccess)
        return cuda_status(cudaGetLastError());
      return PA_OK;
    }
  }
  if (a.cascade) {
    // The prefix pass and each sequence's own keys write disjoint partial
    // slots: run them side by side (the persistent prefix kernel on the
    // high-priority side stream, the own keys on the low-priority one) and
    // join before the combine, which launch_decode queues after them.
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream* side = a.casc_tc ? side_stream() : nullptr;
    if (side) {
      if (cudaEventRecord(side->fork, st) != cudaSuccess ||
          cudaStreamWaitEvent(side->hi, side->fork, 0) != cudaSuccess ||
          cudaStreamWaitEvent(side->lo, side->fork, 0) != cudaSuccess)
        return cuda_status(cudaGetLastError());
      AttnArgs ap = a;
      ap.has_priority = true;
      ap.priority = side->greatest;
      int rc = cuda_status(launch_cascade_prefix(ap, side->hi));
      if (rc != PA_OK) return rc;
      AttnArgs ad = a;
      ad.has_priority = true;
      ad.priority = side->least;
      ad.defer_combine = true;
      rc = cuda_status(launch_decode(ad, side->lo));
      if (rc != PA_OK) return rc;
      if (cudaEventRecord(side->join_hi, side->hi) != cudaSuccess ||
          cudaEventRecord(side->join_lo, side->lo) != cudaSuccess ||
          cudaStreamWaitEvent(st, side->join_hi, 0) != cudaSuccess ||
          cudaStreamWaitEvent(st, side->join_lo, 0) != cudaSuccess)
        return cuda_status(cudaGetLastError());
      return cuda_status(launch_combine(a, st));
    }
    int rc = cuda_status(launch_cascade_prefix(a, st));
    if (rc != PA_OK) return rc;
  }
  if (has_decode) {
    int rc = cuda_status(launch_decode(a, st));
    if (rc != PA_OK) return rc;
  }
  if (has_prefill) {
    int rc = cuda_status(launch_prefill(a, st));
    if (rc != PA_OK) return rc;
  }
  return PA_OK;
}

int pa_attention(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                 const void* k_cache, const void* v_cache, const int32_t* query_start_loc,
                 const int32_t* seq_lens, const int32_t* block_tables, int num_seqs,
                 int num_tokens, int max_blocks_per_seq, int num_decode_seqs, int max_query_len,
                 int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                 int block_size, int num_blocks, float scale, void* workspace,
                 size_t workspace_bytes, uint32_t* err_flag, void* stream) {
  return attention_impl(out, out_stride_t, q, q_stride_t, k_cache, v_cache, query_start_loc,
                        seq_lens, block_tables, num_seqs, num_tokens, max_blocks_per_seq,
                        num_decode_seqs, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks, scale, workspace, workspace_bytes,
                        err_flag, stream, nullptr);
}

int pa_write_kv_attention(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                          const void* k, int64_t k_stride_t, const void* v, int64_t v_stride_t,
                          void* k_cache, void* v_cache, const int32_t* slot_mapping,
                          const int32_t* query_start_loc, const int32_t* seq_lens,
                          const int32_t* block_tables, int num_seqs, int num_tokens,
                          int max_blocks_per_seq, int num_decode_seqs, int max_query_len,
                          int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int num_blocks, float scale, void* workspace,
                          size_t workspace_bytes, uint32_t* err_flag, void* stream) {
  if (num_tokens > 0) {
    if (!k || !v || !slot_mapping) return PA_ERR_INVALID_ARG;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (k_stride_t < row || v_stride_t < row) return PA_ERR_INVALID_ARG;
    if (k_stride_t % 8 || v_stride_t % 8 || !aligned16(k) || !aligned16(v)) return PA_ERR_UNSUPPORTED;
  }
  const FusedIn f{k, v, k_stride_t, v_stride_t, slot_mapping};
  return attention_impl(out, out_stride_t, q, q_stride_t, k_cache, v_cache, query_start_loc,
                        seq_lens, block_tables, num_seqs, num_tokens, max_blocks_per_seq,
                        num_decode_seqs, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks, scale, workspace, workspace_bytes,
                        err_flag, stream, &f);
}

int pa_write_kv_fp8(const void* k, const void* v, int64_t k_stride_t, int64_t v_stride_t,
                    void* k_cache, void* v_cache, const int32_t* slot_mapping, int num_tokens,
                    int num_blocks, int block_size, int num_kv_heads, int head_dim, float k_scale,
                    float v_scale, uint32_t* err_flag, void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale))
    return PA_ERR_INVALID_ARG;
  if (!k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping) return PA_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row % 16 || k_stride_t % 8 || v_stride_t % 8 || k_stride_t < row || v_stride_t < row)
    return PA_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_UNSUPPORTED;
  return cuda_status(launch_write_kv_fp8(k, v, k_stride_t, v_stride_t, k_cache, v_cache,
                                         slot_mapping, num_tokens, num_blocks, block_size,
                                         static_cast<int>(row), 1.f / k_scale, 1.f / v_scale,
                                         err_flag, static_cast<cudaStream_t>(stream)));
}

int pa_attention_fp8(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                     const void* k_cache, const void* v_cache, const int32_t* query_start_loc,
                     const int32_t* seq_lens, const int32_t* block_tables, int num_seqs,
                     int num_tokens, int max_blocks_per_seq, int num_decode_seqs,
                     int max_query_len, int max_seq_len, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int num_blocks, float scale, float k_scale,
                     float v_scale, void* workspace, size_t workspace_bytes, uint32_t* err_flag,
                     void* stream) {
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale))
    return PA_ERR_INVALID_ARG;
  const float scales[2] = {k_scale, v_scale};
  return attention_impl(out, out_stride_t, q, q_stride_t, k_cache, v_cache, query_start_loc,
                        seq_lens, block_tables, num_seqs, num_tokens, max_blocks_per_seq,
                        num_decode_seqs, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks, scale, workspace, workspace_bytes,
                        err_flag, stream, nullptr, scales);
}


size_t pa_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_seq_len, int prefix_blocks, int block_size) {
  int part, nsplit, part_p, nsplit_p;
  const int64_t plen = static_cast<int64_t>(prefix_blocks) * block_size;
  if (prefix_blocks <= 0 || block_size <= 0 || plen >= max_seq_len)
    return pa_attention_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len);
  // either prefix pass may run (it depends on the pointers' alignment too)
  const size_t tc = cascade_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                      static_cast<int>(plen), true, &part, &nsplit, &part_p,
                                      &nsplit_p);
  const size_t mma = cascade_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                       max_seq_len, static_cast<int>(plen), false, &part, &nsplit,
                                       &part_p, &nsplit_p);
  return kWorkspaceHeader + (tc > mma ? tc : mma);
}

int pa_attention_cascade(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                         const void* k_cache, const void* v_cache, const int32_t* query_start_loc,
                         const int32_t* seq_lens, const int32_t* block_tables, int num_seqs,
                         int num_tokens, int max_blocks_per_seq, int max_seq_len,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int prefix_blocks, float scale, void* workspace,
                         size_t workspace_bytes, uint32_t* err_flag, void* stream) {
  return attention_impl(out, out_stride_t, q, q_stride_t, k_cache, v_cache, query_start_loc,
                        seq_lens, block_tables, num_seqs, num_tokens, max_blocks_per_seq,
                        num_seqs, 1, max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, scale, workspace, workspace_bytes, err_flag, stream, nullptr,
                        nullptr, prefix_blocks);
}

}  // extern "C"
