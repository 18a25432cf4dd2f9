// pa_attention_noalloc: pa_attention for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain scratch memory for the split-KV decode
// partials: code embedded in a host application that owns every device
// allocation and hands out no allocator, a runtime whose device memory is
// fully reserved up front, or a latency-critical loop that must not call
// cudaMalloc (which can block until the device is idle).  This entry point
// takes no workspace.  Its scratch is the file-scope device array below,
// kNoallocScratchBytes in size, which every GPU that loads this library
// keeps allocated until the process exits.
//
// The array's name is only meaningful in device code.  Host code needs the
// device address, which cudaGetSymbolAddress returns; that lookup happens on
// the first call made on each device (with that device current), so make that
// first call before any stream capture begins.
//
// All calls share the one array and it keeps whatever the previous call left
// in it.  Nothing in it needs to start at zero: every partial result the
// combine pass reads is written earlier in the same call.  Two calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on the array and produce garbage; serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "pa.h"

namespace {

constexpr size_t kNoallocScratchBytes = PA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      // Clear the runtime's last error: a later launch check in another call
      // must not pick up this failure and report its own launch as failed.
      cudaGetLastError();
      return static_cast<int>(e);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return 0;
}

}  // namespace

extern "C" int pa_attention_noalloc(void* out, int64_t out_stride_t, const void* q,
                                    int64_t q_stride_t, const void* k_cache, const void* v_cache,
                                    const int32_t* query_start_loc, const int32_t* seq_lens,
                                    const int32_t* block_tables, int num_seqs, int num_tokens,
                                    int max_blocks_per_seq, int num_decode_seqs,
                                    int max_query_len, int max_seq_len, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, float scale, uint32_t* err_flag,
                                    void* stream) {
  const size_t need = pa_attention_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads,
                                                  head_dim, max_seq_len);
  if (need > kNoallocScratchBytes) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const int e = scratch_address(&scratch);
    if (e != 0) return pa::record_cuda_error(static_cast<cudaError_t>(e));
  }
  return pa_attention(out, out_stride_t, q, q_stride_t, k_cache, v_cache, query_start_loc,
                      seq_lens, block_tables, num_seqs, num_tokens, max_blocks_per_seq,
                      num_decode_seqs, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, scratch,
                      need > 0 ? kNoallocScratchBytes : 0, err_flag, stream);
}
