/*
 * pa.h — C ABI of the paged-KV attention library (one continuous-batching step).
 *
 * Terms (all from "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数",
 * §2.1 and §2.3补充):
 *   S   number of sequences scheduled this step, T number of new tokens.
 *   The new tokens of all sequences form one flat [T] batch; sequence s owns
 *   rows query_start_loc[s] .. query_start_loc[s+1]-1.
 *   seq_lens[s] = cached history + new tokens of sequence s (its KV length
 *   after this step).  New token i of sequence s sits at position
 *   seq_lens[s] - q_s + i, q_s = query_start_loc[s+1] - query_start_loc[s].
 *   block_tables[s][j] is the physical block holding logical block j of
 *   sequence s (rows padded with -1), "vLLM 原理" §3.7 item 4.
 *   slot_mapping[t] = physical_block * block_size + offset is the cache slot
 *   that flat token t's K/V are written to (§2.3补充 第一步).
 *
 * Memory layout (one layer of the "vLLM 原理" §3.6 cache tensor):
 *   k_cache, v_cache : bf16 [num_blocks, block_size, num_kv_heads, head_dim],
 *                      contiguous, 16-byte aligned.
 *   q, out           : bf16 [T, num_q_heads, head_dim]; head_dim contiguous,
 *                      heads contiguous within a token, token stride given.
 *   k, v (new)       : bf16 [T, num_kv_heads, head_dim], same convention.
 *   Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: every pointer is a device pointer owned by the caller unless it
 * says otherwise; the library allocates no device memory and keeps no
 * pointer after a call returns.  Every call is asynchronous and ordered on
 * the given stream (a cudaStream_t passed as void*, NULL = default stream);
 * none synchronises with the host.
 *
 * Errors: a problem visible on the host (null pointer, unsupported shape,
 * workspace too small) returns a non-zero pa_status and launches nothing.  A
 * problem that only the device can see (bad slot, bad block id, inconsistent
 * lengths) sets PA_DEV_* bits in *err_flag with atomicOr (err_flag may be
 * NULL to skip reporting); the offending rows are skipped and their outputs
 * are unspecified.  No kernel traps and no kernel waits on another block.
 *
 * Environment (read at each call; results are unchanged within rounding):
 *   PA_PREFILL_IMPL=mma    prefill rows on the mma.sync kernel instead of the
 *                          tcgen05 one.
 *   PA_CASCADE_IMPL=mma    pa_attention_cascade's prefix pass on the mma.sync
 *                          kernel instead of the tcgen05 one.
 *   PA_MIXED_DECODE_SMS=n  SMs left to the decode rows while a mixed step's
 *                          prefill runs beside them (default 84 of every 152 SMs).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent counts     */
  PA_ERR_UNSUPPORTED = 2, /* head_dim, block_size or head ratio not supported     */
  PA_ERR_WORKSPACE = 3,   /* workspace smaller than pa_attention_workspace_size()  */
  PA_ERR_CUDA = 4         /* a launch failed; see pa_last_cuda_error()             */
} pa_status;

/* Device-side error bits OR-ed into *err_flag. */
#define PA_DEV_BAD_SLOT 1u   /* slot_mapping entry >= num_blocks * block_size      */
#define PA_DEV_BAD_BLOCK 2u  /* a live position maps to a block id outside the pool */
#define PA_DEV_BAD_LEN 4u    /* seq_len < q_len, seq_len > max_blocks*block_size,
                                q_len > max_query_len or seq_len > max_seq_len     */
#define PA_DEV_BAD_DECODE 8u /* a row below num_decode_seqs has q_len != 1          */
#define PA_DEV_BAD_PAIR 16u  /* a copy pair names a block outside the pool          */
#define PA_DEV_TIMEOUT 32u   /* a pipeline wait inside a kernel ran out of time (2 s,
                                or pa_set_wait_limit_ns); the kernel drained its
                                copies and products and exited, outputs unspecified */

/*
 * pa_write_kv — scatter the new tokens' K and V into the paged cache.
 * "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数" §2.3补充 第一步;
 * store_kvcache in "vLLM 原理" §3.7.
 *
 *   k, v           bf16 [T, num_kv_heads, head_dim]; row t starts at element
 *                  t * k_stride_t (resp. v_stride_t).
 *   k_cache,v_cache bf16 [num_blocks, block_size, num_kv_heads, head_dim].
 *   slot_mapping   int32 [T]; slot < 0 means "do not write this token".
 * For every t with slot_mapping[t] = b * block_size + o >= 0:
 *   k_cache[b, o] = k[t], v_cache[b, o] = v[t]   (bit-exact copy).
 * Needs num_kv_heads * head_dim % 8 == 0, strides % 8 == 0, 16-byte aligned
 * pointers.  Slots must be distinct; duplicate slots race.
 */
int pa_write_kv(const void* k, const void* v, int64_t k_stride_t, int64_t v_stride_t,
                void* k_cache, void* v_cache, const int32_t* slot_mapping, int num_tokens,
                int num_blocks, int block_size, int num_kv_heads, int head_dim,
                uint32_t* err_flag, void* stream);

/*
 * pa_attention_workspace_size — bytes of scratch pa_attention needs: a
 * 256-byte header (the prefill kernel's work-queue counter, which that
 * kernel tags per launch and resets itself, so no call zeroes it) followed by the
 * split-KV decode partials (fp32 running max, sum and
 * weighted value per split, sequence and query head) when the decode rows are
 * split.  Never 0.  Depends on the current device's SM count; query it on the
 * device that will run the call.
 */
size_t pa_attention_workspace_size(int num_decode_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int max_seq_len);

/*
 * pa_attention — causal attention of one step's flat query batch over the
 * paged cache.  Each query attends only to its own sequence's keys at
 * positions 0 .. its own position ("A 不会看 B", §0 and §2.3 of the first
 * page); keys are read through block_tables (§2.3补充 第二步); the new
 * tokens' K/V must already be in the cache (call pa_write_kv first on the same
 * stream, as "vLLM 原理" §3.7 Attention.forward does).
 *
 *   out      bf16 [T, num_q_heads, head_dim], token stride out_stride_t.
 *   q        bf16 [T, num_q_heads, head_dim], token stride q_stride_t.
 *   query_start_loc int32 [S+1], seq_lens int32 [S],
 *   block_tables    int32 [S, max_blocks_per_seq], -1 padded.
 *   num_decode_seqs sequences [0, num_decode_seqs) must have exactly one new
 *                   token; they run on the split-KV decode kernel, the rest
 *                   on the prefill kernel.  0 is always correct.
 *   max_query_len, max_seq_len  host-known upper bounds of q_s and seq_lens[s]
 *                   (like max_seqlen_q / max_seqlen_k of "vLLM 原理" §3.7).
 *   scale    softmax scale (1/sqrt(head_dim) in the usual case).
 *   workspace, workspace_bytes  device scratch of at least
 *                   pa_attention_workspace_size(num_decode_seqs, ...) bytes,
 *                   16-byte aligned; its contents need no initialisation.
 *                   Calls that overlap on the GPU must not share it.
 * out[t, h] = sum_p softmax_p(scale * q[t,h] . k_p) v_p over the visible keys
 * of t's sequence, accumulated in fp32, rounded once to bf16.
 * Supports head_dim 64 or 128, block_size a power of two in [1, 256],
 * num_q_heads % num_kv_heads == 0.  Rows of sequences with q_s = 0 are untouched.
 */
int pa_attention(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                 const void* k_cache, const void* v_cache, const int32_t* query_start_loc,
                 const int32_t* seq_lens, const int32_t* block_tables, int num_seqs,
                 int num_tokens, int max_blocks_per_seq, int num_decode_seqs, int max_query_len,
                 int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                 int block_size, int num_blocks, float scale, void* workspace,
                 size_t workspace_bytes, uint32_t* err_flag, void* stream);

/*
 * pa_write_kv_attention — pa_write_kv followed by pa_attention in one call,
 * with the scatter folded into the attention kernels.  "vLLM 原理" §3.7 runs
 * the two back to back in every forward (store_kvcache, then the attention
 * call); "vLLM Continuous Batching：从 Forward Shape 理解两个核心参数"
 * §2.3补充 defines slot_mapping as the slot that the block table gives to
 * each new token's position.
 *
 * Arguments are those of pa_attention plus k, v ([num_tokens, num_kv_heads,
 * head_dim] bf16, token strides k_stride_t / v_stride_t in elements, multiples
 * of 8, 16-byte aligned) and slot_mapping ([num_tokens] int32, as in
 * pa_write_kv).  k_cache / v_cache are written.
 *
 * Result: the caches are written exactly as pa_write_kv writes them, and out
 * is the attention of pa_write_kv then pa_attention, provided that each new
 * token's slot is the one its sequence's block table gives to its position.
 *
 * A step with no decode rows whose prefill runs on the tensor-core path is
 * one launch: the kernel takes the K/V of positions c_s .. L_s - 1 from k, v
 * rather than from the cache and stores each token's row into its slot.  It
 * groups those new keys into 128-key tiles starting at c_s (the cached
 * history keeps its tiles from position 0), so the result is bit-identical
 * to the two calls for sequences without history and otherwise equal up to
 * the order of the fp32 sums.  Any other step (decode rows present, or
 * scale <= 0) scatters first and then attends, bit-identical to the two
 * calls.
 * Errors: as pa_write_kv and pa_attention.
 */
int pa_write_kv_attention(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                          const void* k, int64_t k_stride_t, const void* v, int64_t v_stride_t,
                          void* k_cache, void* v_cache, const int32_t* slot_mapping,
                          const int32_t* query_start_loc, const int32_t* seq_lens,
                          const int32_t* block_tables, int num_seqs, int num_tokens,
                          int max_blocks_per_seq, int num_decode_seqs, int max_query_len,
                          int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int num_blocks, float scale, void* workspace,
                          size_t workspace_bytes, uint32_t* err_flag, void* stream);

/*
 * pa_copy_blocks — copy-on-write block copies, "vLLM 原理" §2.1: for each
 * pair (src, dst) in pairs (int32 [num_pairs, 2], device memory),
 * k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src], all
 * block_size slots, bit-exact.  Destinations must be distinct and must not be
 * the source of any pair (copy-on-write always copies into a fresh block);
 * otherwise the result is unspecified.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                   int num_blocks, int block_size, int num_kv_heads, int head_dim,
                   uint32_t* err_flag, void* stream);

/*
 * pa_swap_blocks — move whole blocks between two K/V pools, e.g. a GPU pool
 * and a pool in host memory, for CPU offload of the cache: "LLM 推理引擎
 * Continuous Batching 与 PagedAttention：从 vLLM 原理到生产级部署实战" §4.4
 * (swap_out copies a request's blocks device -> host, swap_in host -> device)
 * and the block-table role ③ of "vLLM Continuous Batching：从 Forward Shape
 * 理解两个核心参数" §2.3补充.  For each pair (s, d) of pairs (int32
 * [num_pairs, 2], device memory):
 *   dst_k[d] = src_k[s] and dst_v[d] = src_v[s], all block_size slots, bit-exact.
 * Both pools have the [blocks, block_size, num_kv_heads, head_dim] bf16
 * layout, 16-byte aligned; the caller owns all five buffers.  Each pool
 * pointer may be device memory, managed memory, or page-locked host memory
 * (cudaHostAlloc / cudaHostRegister; the kernel uses its mapped device
 * address); other host memory only where the device reports coherent
 * pageable-memory access.  A pool pointer the device cannot reach returns
 * PA_ERR_INVALID_ARG before any launch.  The copy is one kernel reading and
 * writing through those pointers, so no staging buffer is made.  Destination
 * blocks must be distinct and must not be source blocks of the same call.
 * A pair naming a block outside its pool sets PA_DEV_BAD_PAIR and copies
 * nothing for that pair.  num_pairs == 0 launches nothing; more than 65535
 * pairs returns PA_ERR_UNSUPPORTED (split the call).
 */
int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                   const int32_t* pairs, int num_pairs, int src_num_blocks, int dst_num_blocks,
                   int block_size, int num_kv_heads, int head_dim, uint32_t* err_flag,
                   void* stream);

/*
 * 8-bit KV cache (an extension: the pages' cache is bf16).  The cache holds
 * OCP E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, largest finite magnitude 448) with one scale per tensor:
 * value = code * scale.  Same [num_blocks, block_size, num_kv_heads,
 * head_dim] layout, one byte per element, 16-byte aligned.
 *
 * pa_write_kv_fp8 — pa_write_kv into an 8-bit cache: each element x of the
 * new rows is stored as the E4M3 code nearest to fp32(x) * fp32(1 / scale)
 * (ties to the even code, magnitudes past 448 clamped to 448).  Scales must
 * be positive and finite (PA_ERR_INVALID_ARG); num_kv_heads * head_dim must
 * be a multiple of 16 and the token strides multiples of 8 elements
 * (PA_ERR_UNSUPPORTED).  Device errors as pa_write_kv.
 */
int pa_write_kv_fp8(const void* k, const void* v, int64_t k_stride_t, int64_t v_stride_t,
                    void* k_cache, void* v_cache, const int32_t* slot_mapping, int num_tokens,
                    int num_blocks, int block_size, int num_kv_heads, int head_dim, float k_scale,
                    float v_scale, uint32_t* err_flag, void* stream);

/*
 * pa_attention_fp8 — pa_attention over an 8-bit cache, for decode steps:
 * every sequence must be a decode row (num_decode_seqs == num_seqs, else
 * PA_ERR_UNSUPPORTED; the tensor-core prefill reads bf16 only).  Keys and
 * values are the codes times k_scale / v_scale.  The kernel stages the codes
 * in shared memory as they are, converts each mma fragment to fp16 in
 * registers (exact for every code) and runs the products in fp16 with fp32
 * accumulation; q is converted to fp16 once, so |q| must stay below 65504.
 * Workspace and errors as pa_attention.
 */
int pa_attention_fp8(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                     const void* k_cache, const void* v_cache, const int32_t* query_start_loc,
                     const int32_t* seq_lens, const int32_t* block_tables, int num_seqs,
                     int num_tokens, int max_blocks_per_seq, int num_decode_seqs,
                     int max_query_len, int max_seq_len, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int num_blocks, float scale, float k_scale,
                     float v_scale, void* workspace, size_t workspace_bytes, uint32_t* err_flag,
                     void* stream);

/*
 * pa_attention_noalloc — pa_attention without a workspace argument, for
 * callers that cannot allocate device memory (a library embedded in a host
 * application that owns every device allocation, a runtime whose memory is
 * reserved up front, or a loop that must not call cudaMalloc, which can wait
 * for the whole device).  The pages have no counterpart: this is a calling
 * convention of this library, not part of the method.
 *
 * Same arguments, result and errors as pa_attention minus workspace and
 * workspace_bytes.  The split-KV scratch is a static device array of
 * PA_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  A call whose decode
 * rows would need more scratch than that returns PA_ERR_WORKSPACE and
 * launches nothing (use pa_attention with a workspace instead).
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.  A
 * failed lookup returns PA_ERR_CUDA and records the CUDA error for
 * pa_last_cuda_error (the runtime's own last-error state is cleared).
 * Every call shares the array and it keeps the previous call's contents;
 * nothing in it has to start at zero.  Calls that overlap on the GPU (other
 * streams or host threads) race on the array: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
int pa_attention_noalloc(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                         const void* k_cache, const void* v_cache,
                         const int32_t* query_start_loc, const int32_t* seq_lens,
                         const int32_t* block_tables, int num_seqs, int num_tokens,
                         int max_blocks_per_seq, int num_decode_seqs, int max_query_len,
                         int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int num_blocks, float scale, uint32_t* err_flag,
                         void* stream);

/*
 * pa_attention_cascade — decode attention for a batch whose sequences all
 * start with the same cached blocks: a common prompt served from the prefix
 * cache ("vLLM 原理" §2.3 Automatic Prefix Cache), whose shared blocks
 * copy-on-write keeps read-only (§2.1).
 *
 * Same result, within rounding, as pa_attention with num_decode_seqs =
 * num_seqs (every row a decode row) and max_query_len = 1.  The caller
 * promises that the first prefix_blocks entries of every block_tables row
 * hold the same physical block ids, so that key positions
 * [0, prefix_blocks * block_size) are the same K/V for every sequence.  The
 * host scheduler knows this from the tables it built.  The call then reads
 * those keys once for each group of 128 (sequence, query head) rows of a kv
 * head instead of once per sequence, reads each sequence's own keys
 * [prefix_blocks * block_size, L) as pa_attention does, and merges the two
 * exactly (online-softmax partials).
 *
 * Arguments: those of pa_attention without num_decode_seqs and
 * max_query_len, plus prefix_blocks (>= 0; 0 is plain decode attention).
 * bf16 cache only.  Workspace: pa_cascade_workspace_size(...) bytes.
 * Errors: PA_ERR_INVALID_ARG when prefix_blocks < 0, prefix_blocks >
 * max_blocks_per_seq or prefix_blocks * block_size >= max_seq_len.  Device
 * errors are those of pa_attention.  A sequence with seq_len <=
 * prefix_blocks * block_size has no key of its own and sets PA_DEV_BAD_LEN;
 * its output row is not written.  Tables that break the promise give the
 * attention of the first sequence's prefix blocks, which is undefined for
 * the others (not detected).
 */
size_t pa_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_seq_len, int prefix_blocks, int block_size);
int pa_attention_cascade(void* out, int64_t out_stride_t, const void* q, int64_t q_stride_t,
                         const void* k_cache, const void* v_cache,
                         const int32_t* query_start_loc, const int32_t* seq_lens,
                         const int32_t* block_tables, int num_seqs, int num_tokens,
                         int max_blocks_per_seq, int max_seq_len, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         int prefix_blocks, float scale, void* workspace, size_t workspace_bytes,
                         uint32_t* err_flag, void* stream);

/* Human-readable name of a pa_status value (static string). */
const char* pa_status_string(int status);

/* The cudaError_t of the last call that returned PA_ERR_CUDA on this thread. */
int pa_last_cuda_error(void);

/* Number of kernels this library has launched since it was loaded (all threads). */
uint64_t pa_kernel_launches(void);

/*
 * pa_set_wait_limit_ns — failure-detection control (not part of the method).
 *
 * The tensor-core prefill kernel (also the shared-prefix pass) waits on
 * shared-memory barriers for its copies and products.  Each such wait gives
 * up after a limit: the kernel then sets PA_DEV_TIMEOUT in err_flag, waits
 * for its own copies and products still in flight (each of those drain waits
 * bounded at 2 s), frees its tensor memory and exits, so that the context
 * stays usable.  This sets that limit for launches made after the call, for
 * every thread and device of the process; 0 restores the default of 2 s.  A
 * short limit makes an ordinary call time out on purpose, which is how a
 * test checks that the give-up path returns cleanly.  Returns the previous
 * setting.
 */
uint64_t pa_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
