// Host-side launch interface between the C ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

void count_launch();

// Records a CUDA error for pa_last_cuda_error on this thread; returns
// PA_ERR_CUDA (PA_OK for cudaSuccess).
int record_cuda_error(cudaError_t e);

// SM count of the current device (cached per device).
int device_num_sms();

struct AttnArgs {
  void* out;
  int64_t out_stride;  // elements between tokens
  const void* q;
  int64_t q_stride;
  const void* k_cache;
  const void* v_cache;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int num_seqs;
  int num_tokens;
  int max_blocks;
  int num_decode;
  int max_query_len;
  int max_seq_len;
  int hq, hkv, group;  // group = hq / hkv
  int head_dim;
  int bs_log2;
  int num_blocks;
  float scale_log2;  // scale * log2(e)
  uint32_t* err;
  // split-KV decode
  int part;      // tokens per split
  int nsplit;    // grid splits = ceil(max_seq_len / part)
  float* ws_o;   // [nsplit, num_decode, hq, head_dim]
  float* ws_ml;  // [nsplit, num_decode, hq, 2]
  // Prefill work queue: a 64-bit word at the start of the workspace header,
  // (launch tag << 32 | number of draws after the first wave).  The launch
  // sets sched_tag (never 0, new for every launch); a word holding another
  // tag is reset by the kernel itself and the kernel leaves it at (tag, 0),
  // so the header needs no zeroing between calls.
  unsigned long long* sched;
  uint32_t sched_tag;
  // cap on the persistent prefill grid (0: one CTA per SM)
  int max_ctas;
  // Fused scatter for the prefill rows (null k_new: none).  The tensor-core
  // prefill reads the new tokens' K/V from k_new / v_new ([T, Hkv, D], token
  // strides in elements) for positions c_s .. L_s - 1 instead of from the
  // cache, and stores each of those tokens' rows into its slot_mapping slot.
  const void* k_new;
  const void* v_new;
  int64_t kn_stride, vn_stride;
  const int32_t* slots;
  // 8-bit cache: k_cache / v_cache hold E4M3 codes; scale_log2 then includes
  // the K scale and the outputs are multiplied by the V scale (1 / inv_v_scale)
  bool kv_fp8;
  float inv_v_scale;
  // Shared-prefix (cascade) decode: the first prefix_len key positions of every
  // decode sequence are the same physical blocks.  The prefix pass writes
  // nsplit_prefix partials per (sequence, head) into workspace slots
  // [0, nsplit_prefix); the decode kernel then covers keys [key_begin, L) and
  // writes its partials from slot split0 on; the combine merges them all.
  bool cascade;
  bool casc_tc;        // the prefix pass runs on the tensor-core prefill kernel
  bool defer_combine;  // launch_decode leaves the combine to launch_combine
  int key_begin, split0, nsplit_prefix, prefix_len, part_prefix;
  // Launch priority of this call's attention kernels (has_priority false: the
  // stream's own).  A mixed step sets it on both sides: the launch attribute
  // is recorded in the kernel node when the step is captured into a CUDA graph.
  bool has_priority;
  int priority;
  // Limit of each pipeline wait inside the tensor-core kernels, in ns (the
  // value pa_set_wait_limit_ns set; 0: the default of 2 s).  Their drain
  // waits on the way out keep the default.
  uint64_t wait_ns;
};

// Launches `kernel` on `st` with the given priority as a launch attribute when
// `has_priority`, else with the stream's.
template <typename... P, typename... A>
cudaError_t launch_prio(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                        cudaStream_t st, bool has_priority, int priority, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributePriority;
  attr[0].val.priority = priority;
  cfg.attrs = attr;
  cfg.numAttrs = has_priority ? 1u : 0u;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

// Bytes at the start of the workspace reserved for the prefill work queue.
constexpr size_t kWorkspaceHeader = 256;

// Split-KV partition for the decode rows; shared by the workspace query and the
// launch so that both agree.
void decode_partition(int num_decode, int hkv_units, int max_seq_len, int num_sms, int* part,
                      int* nsplit);

cudaError_t launch_write_kv(const void* k, const void* v, int64_t ks, int64_t vs, void* kc,
                            void* vc, const int32_t* slots, int T, int num_blocks, int bs,
                            int row_elems, uint32_t* err, cudaStream_t st);
cudaError_t launch_write_kv_fp8(const void* k, const void* v, int64_t ks, int64_t vs, void* kc,
                                void* vc, const int32_t* slots, int T, int num_blocks, int bs,
                                int row_elems, float inv_k_scale, float inv_v_scale,
                                uint32_t* err, cudaStream_t st);
cudaError_t launch_copy_blocks(void* kc, void* vc, const int32_t* pairs, int n, int num_blocks,
                               int block_elems, uint32_t* err, cudaStream_t st);
cudaError_t launch_swap_blocks(const void* sk, const void* sv, void* dk, void* dv,
                               const int32_t* pairs, int n, int src_blocks, int dst_blocks,
                               int block_elems, uint32_t* err, cudaStream_t st);
cudaError_t launch_decode(const AttnArgs& a, cudaStream_t st);
// The split combine alone (after a launch_decode with defer_combine).
cudaError_t launch_combine(const AttnArgs& a, cudaStream_t st);
// Cascade prefix pass (see AttnArgs::cascade); CTAs and slots from
// cascade_partition.
cudaError_t launch_cascade_prefix(const AttnArgs& a, cudaStream_t st);
void cascade_partition(int num_decode, int hq, int hkv, int prefix_len, int num_sms, bool tc,
                       int* part_prefix, int* nsplit_prefix);
// The prefix pass on the tensor-core prefill kernel (query heads per kv head a
// multiple of 8 dividing 128, and the prefill kernel's own conditions).
bool cascade_tc_supported(const AttnArgs& a);
cudaError_t launch_cascade_tc(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_prefill(const AttnArgs& a, cudaStream_t st);

// Tensor-core (tcgen05) prefill: whether the shapes and the environment allow
// it, and its launch (cudaErrorNotSupported, with nothing launched, when a
// TMA descriptor cannot be encoded).
bool prefill_tc_supported(const AttnArgs& a);
cudaError_t launch_prefill_tc(const AttnArgs& a, cudaStream_t st);

}  // namespace pa
