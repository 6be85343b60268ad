/*
 * pa.h -- C ABI of the paged-KV attention step (libpagedattn.so, CUDA, sm_103a).
 *
 * One continuous-batching attention step over a paged KV cache has two calls:
 *
 *   pa_cache_append  writes each new token's key and value into its slot of the block pool.
 *                    "Serving LLMs with vLLM: Continuous Batching and PagedAttention
 *                    Explained", section "Growing During Decode": each step appends the token
 *                    into the last block of its sequence; section "Blocks and Block Tables":
 *                    blocks are fixed-size (e.g. 16 tokens) and found through a per-sequence
 *                    block table.  The caller has already folded the table into a slot.
 *
 *   pa_attention     attends a ragged batch of query tokens (decode tokens and chunked-prefill
 *                    pieces) to their own sequence's keys and values, fetched block by block
 *                    through the block tables.  Same page, section "Attention Over Scattered
 *                    Blocks": the mathematics is ordinary attention, softmax of the query times
 *                    the keys over the whole history; only the addressing changes.  Sections
 *                    "Prefill Versus Decode" and "Chunked Prefill": one step mixes prompt chunks
 *                    with decode tokens.  Section "Shared Prefixes": several tables may point at
 *                    the same physical blocks.
 *
 * Conventions shared by every call
 *   - Memory: every pointer argument named *_cache, q, k, v, out, slot_mapping, block_tables,
 *     context_lens, query_start_loc and workspace is a DEVICE pointer on the current device.
 *     `cache` descriptors are HOST pointers.  The caller allocates and owns all of it; the
 *     library never allocates or frees device memory.
 *   - Execution: calls are asynchronous on `stream` (0 = legacy default stream) and ordered by
 *     it; nothing synchronises the host except pa_check_error.  pa_cache_append must precede
 *     pa_attention on the same stream when the step's new tokens are to be attended.
 *   - Errors: argument errors are detected on the host and returned before anything is
 *     launched (PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED).  Errors that only the device can see
 *     (a block id or slot outside the pool, inconsistent lengths, an internal wait that timed
 *     out) make the kernel skip the offending access and set a bit in the error word held in
 *     the first bytes of `workspace`; pa_check_error reports and clears it.  No call traps,
 *     aborts or hangs on bad input.  pa_last_error_string describes the last host-side error
 *     of the calling thread.
 *
 * Layouts (all row-major, contiguous)
 *   block pool:  k_cache, v_cache = [num_blocks][num_kv_heads][block_size][head_dim], elements
 *                bf16, or OCP E4M3 bytes holding x / k_scale (resp. v_scale) with fp32 per-tensor
 *                scales.  One (block, kv head) tile of block_size x head_dim is contiguous.
 *   slot:        physical_block * block_size + offset; a negative slot means "skip".
 *   new k, v:    [num_tokens][num_kv_heads][head_dim] bf16.
 *   q, out:      [num_q_tokens][num_q_heads][head_dim]; q bf16, out fp32 or bf16.
 *   block_tables [num_seqs][max_blocks_per_seq] int32; entries past ceil(context_len/block_size)
 *                are never read.
 *   context_lens [num_seqs] int32: keys of the sequence after this step's append.
 *   query_start_loc [num_seqs + 1] int32: exclusive prefix sum of per-sequence query counts
 *                n_s, starting at 0.  The n_s queries of sequence s are its last n_s positions
 *                p_i = context_len - n_s + i, and query i attends keys 0..p_i.
 *   GQA:         q head h reads kv head h / (num_q_heads / num_kv_heads); groups of up to 16
 *                q heads per kv head are built.
 */
#ifndef PAGED_KV_PA_H_
#define PAGED_KV_PA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent shapes, small workspace */
  PA_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, block_size, dtype or GQA group */
  PA_ERR_OUT_OF_RANGE = 3, /* device saw a block id or slot outside the pool, or bad lengths */
  PA_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up (results are not valid) */
  PA_ERR_CUDA = 5          /* a CUDA runtime call failed; see pa_last_error_string */
} pa_status;

typedef enum { PA_BF16 = 0, PA_FP8_E4M3 = 1, PA_FP32 = 2 } pa_dtype;

/* Geometry of one pool (both k_cache and v_cache).  Supported: block_size 16; head_dim 64 or
 * 128 for bf16, 128 for PA_FP8_E4M3; num_blocks * num_kv_heads * block_size (the pool's rows)
 * at most 2^31 - 1.  k_scale / v_scale are used only for PA_FP8_E4M3. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t cache_dtype; /* pa_dtype: PA_BF16 or PA_FP8_E4M3 */
  float k_scale;
  float v_scale;
} pa_cache_desc;

/* Bytes at the start of every workspace that hold the device error word; a workspace passed
 * to pa_cache_append needs at least this many bytes (pa_attention's workspace qualifies). */
#define PA_WORKSPACE_HEADER_BYTES 256

/* Device error-word bits (pa_check_error maps them to its status and returns the raw word
 * through its word_out argument). */
#define PA_DEVERR_BLOCK_ID 0x1u    /* block table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT 0x2u        /* slot >= num_blocks * block_size */
#define PA_DEVERR_LENGTHS 0x4u     /* n_s < 0, n_s > context_len, or a host hint exceeded */
#define PA_DEVERR_TIMEOUT 0x8u     /* bounded wait expired */

/* Scatter new keys/values into the pool.
 *   k, v          [num_tokens][num_kv_heads][head_dim] bf16 (device).
 *   slot_mapping  [num_tokens] int64 (device); slot of token t; < 0 skips the token.
 *   k_cache, v_cache  pool tensors described by `cache` (device, written in place).
 *   workspace     >= PA_WORKSPACE_HEADER_BYTES bytes (device); receives PA_DEVERR_SLOT.
 * bf16 pools receive the bits unchanged.  E4M3 pools receive, per element, the E4M3 encoding
 * (round to nearest even, saturating to +-448) of the fp32 quotient x / scale rounded to
 * nearest.  num_tokens == 0 is a no-op.  A slot written twice in one call ends up holding one
 * of the writes. */
pa_status pa_cache_append(const void* k, const void* v, const int64_t* slot_mapping,
                          int32_t num_tokens, void* k_cache, void* v_cache,
                          const pa_cache_desc* cache, void* workspace, cudaStream_t stream);

/* Copy whole blocks inside the pool: for each pair i, block block_pairs[2i] (source) is copied
 * to block block_pairs[2i+1] (destination), all kv heads, K and V, bit for bit.
 * "Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained", section
 * "Copy-on-Write": before a sequence writes into a shared block, the engine copies it to a
 * fresh block and points only that sequence's table at the copy.
 *   block_pairs  [num_pairs][2] int32 (device); num_pairs <= 65535.
 *   workspace    >= PA_WORKSPACE_HEADER_BYTES bytes (device); a block id outside the pool sets
 *                PA_DEVERR_BLOCK_ID and that pair is skipped.
 * Pairs must not overlap (no block is both a source and a destination, no destination twice);
 * otherwise the result is undefined. */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const pa_cache_desc* cache,
                         const int32_t* block_pairs, int32_t num_pairs, void* workspace,
                         cudaStream_t stream);

/* Workspace bytes pa_attention needs for a step of this shape (host-only, no device call).
 * max_context_len / max_query_len are upper bounds of context_lens[s] and n_s. */
size_t pa_attention_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int32_t max_context_len, int32_t max_query_len);

/* Ragged paged attention of one step.
 *   q             [num_q_tokens][num_q_heads][head_dim] bf16 (device).
 *   k_cache, v_cache, cache   the pool (device / host descriptor).
 *   block_tables  [num_seqs][max_blocks_per_seq] int32 (device).
 *   context_lens  [num_seqs] int32 (device).  query_start_loc [num_seqs + 1] int32 (device),
 *                 query_start_loc[num_seqs] must equal num_q_tokens.
 *   max_context_len, max_query_len   host upper bounds of context_lens and n_s (checked on
 *                 the device; a violation sets PA_DEVERR_LENGTHS and skips that sequence).
 *   scale         multiplies q.k before the softmax (e.g. 1/sqrt(head_dim)).
 *   out           [num_q_tokens][num_q_heads][head_dim], out_dtype PA_FP32 or PA_BF16 (device).
 *   workspace     device buffer of workspace_bytes >= pa_attention_workspace_size(...); its
 *                 first PA_WORKSPACE_HEADER_BYTES hold the error word.
 * A sequence with n_s == 0 produces nothing.  Accumulation is fp32; scores use exp2 of
 * log2(e)-prescaled logits.
 * Kernels: every kernel of the call runs on `stream`, each launched early (programmatic
 * dependent launch) and waiting for what it reads: a plan, then, with a bf16 pool of head_dim
 * 128 or 64 or an E4M3 pool of head_dim 128 and query runs of more than 16 tokens or more than
 * 16 (token x q head) rows, the tensor-core prefill tiles on the part of the SMs the plan gives
 * them, the split-KV kernel on the rest, and the merge of split sequences.
 * Work enqueued on `stream` after the call sees all of it complete.  The call records no event
 * and creates no stream, so it can be captured into a CUDA graph like any kernel launch. */
pa_status pa_attention(const void* q, int32_t num_q_tokens, const void* k_cache,
                       const void* v_cache, const pa_cache_desc* cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, const int32_t* query_start_loc,
                       int32_t num_seqs, int32_t max_context_len, int32_t max_query_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                       void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Scratch bytes built into the library for pa_attention_noalloc (32 MiB per device). */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* pa_attention for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is a library convenience, not part of the method.)
 *
 * Some callers are not allowed to call cudaMalloc: code running under a memory manager that
 * owns all device memory, code that must not grow its footprint after start-up, or code on a
 * path where an allocation could stall the device.  They can still pass inputs and outputs but
 * not a workspace, so this call uses a scratch array built into the library instead:
 * PA_NOALLOC_SCRATCH_BYTES per device, held by every GPU that loads the library until the
 * process exits.  A step whose pa_attention_workspace_size exceeds it is rejected with
 * PA_ERR_INVALID_ARG and a message; use pa_attention with a workspace for larger steps.
 *   Arguments are those of pa_attention without workspace/workspace_bytes, plus
 *   error_word    optional DEVICE pointer (may be NULL) that receives, asynchronously on
 *                 `stream`, this call's PA_DEVERR_* bits (0 for a step with nothing to do).  It
 *                 is written only when the call returns PA_OK; a call rejected on the host
 *                 changes neither *error_word nor the scratch array.
 * Each call looks up the scratch array's device address in the current context
 * (cudaGetSymbolAddress); the first lookup in a context may load the library's device code, so
 * make the first call before any stream capture.  Every call shares the
 * one array and overwrites it, starting from a cleared header: calls whose GPU work overlaps
 * (other streams, other threads) race on it and must be serialised by the caller. */
pa_status pa_attention_noalloc(const void* q, int32_t num_q_tokens, const void* k_cache,
                               const void* v_cache, const pa_cache_desc* cache,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, const int32_t* query_start_loc,
                               int32_t num_seqs, int32_t max_context_len, int32_t max_query_len,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               float scale, void* out, int32_t out_dtype, uint32_t* error_word,
                               cudaStream_t stream);

/* Synchronise `stream`, read and clear the device error word at the start of `workspace`.
 * Returns PA_OK, PA_ERR_OUT_OF_RANGE (block id / slot / length bits), PA_ERR_TIMEOUT, or
 * PA_ERR_CUDA.  *word_out (may be NULL) receives the raw PA_DEVERR_* bits. */
pa_status pa_check_error(void* workspace, cudaStream_t stream, uint32_t* word_out);

/* Zero the error word (asynchronously, on `stream`).  Call once on a fresh workspace. */
pa_status pa_workspace_init(void* workspace, cudaStream_t stream);

/* Text of the calling thread's last host-side error ("" if none). */
const char* pa_last_error_string(void);

/* Library version, e.g. "0.1.0". */
const char* pa_version(void);

/* Benchmark hook.  When both events are non-NULL (cudaEvent_t handles), every later
 * pa_attention call of the calling thread records `before` immediately before, and `after`
 * immediately after, its split-KV attention kernel, on the call's stream.  An event between
 * two of the call's kernels makes the later one wait for the earlier one to finish, so with
 * these events the kernels run one after the other and each is timed alone.  Pass NULLs to
 * stop. */
void pa_set_kernel_timing_events(void* before, void* after);

/* Benchmark hook, like pa_set_kernel_timing_events, for the tensor-core prefill-tile kernel
 * (launched only by steps that hold runs of more than 16 tokens or 16 token x head rows over a
 * bf16 pool with head_dim 128 or 64).  Pass NULLs to stop. */
void pa_set_prefill_timing_events(void* before, void* after);

/* Benchmark hook that times kernels while they overlap: when `device_buffer` is non-NULL
 * (four uint64_t in device memory, set by the caller to {UINT64_MAX, 0, UINT64_MAX, 0}), every
 * later pa_attention call of the calling thread has its split-KV kernel lower [0] to the
 * GPU's global timer (ns) when a CTA starts and raise [1] to it when a CTA finishes its work,
 * and its prefill-tile kernel do the same with [2] and [3].  Pass NULL to stop. */
void pa_set_kernel_span_buffer(uint64_t* device_buffer);

/* Limit of every bounded device-side wait in the calling thread's later pa_attention calls, in
 * nanoseconds of the GPU's global timer; 0 restores the default of 1 s.  A wait that reaches
 * the limit gives up: the kernel sets PA_DEVERR_TIMEOUT, lets the copies it still has in flight
 * land (each with its own bounded wait), and returns; pa_check_error then reports
 * PA_ERR_TIMEOUT and that call's output is not valid.  (Not a step of the method: it bounds
 * how long a lost copy can hold the GPU.) */
void pa_set_wait_limit_ns(uint64_t ns);

/* Test hook, off by default; never enable it outside tests.  While enabled, every pa_attention
 * call of the calling thread leaves out exactly one tile copy of each attention kernel it
 * launches (the first copy of the first work item claimed) while that copy's barrier still
 * expects the bytes, so that the bounded waits on it expire and the call ends with
 * PA_ERR_TIMEOUT without any fault: the expiry and drain paths of the kernels can be exercised
 * on a real GPU. */
void pa_test_skip_one_copy(int32_t enable);

/* Self-test of the bounded wait: one thread waits, for limit_ns (in (0, 10 s]), on an mbarrier
 * phase that nothing completes, then sets PA_DEVERR_TIMEOUT in the error word at the start of
 * `workspace` (>= 4 bytes, device) and returns; read it with pa_check_error.  Asynchronous on
 * `stream`.  (Not a step of the method: it checks the library's failure signal.) */
pa_status pa_selftest_wait_timeout(void* workspace, uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_PA_H_ */
