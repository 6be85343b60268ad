// pa_attention_noalloc: the ragged paged attention of pa_attention for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at all: code that runs under an external memory
// manager which owns every byte of the device (a serving engine that reserves HBM up front and
// hands out fixed tensors), code whose budget forbids new device allocations after start-up,
// and code on a latency-critical path where an allocation could synchronise the device.  Those
// callers can still provide inputs and outputs, but not the scratch workspace that
// pa_attention needs for its work plan, split-KV partials and error word.
//
// This entry point keeps that scratch in one file-scope device array of
// PA_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library holds until the process
// exits.  Host code must not use the array's name as a device address (on the host it is only a
// stand-in symbol); the device address is fetched with cudaGetSymbolAddress on every call, in
// the context current at the call.
#include <cstdio>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.  It is looked up on every call
// rather than kept: after cudaDeviceReset the next context places the array anew.
cudaError_t scratch_address(void** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_attention_noalloc(
    const void* q, int32_t num_q_tokens, const void* k_cache, const void* v_cache,
    const pa_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, const int32_t* query_start_loc, int32_t num_seqs,
    int32_t max_context_len, int32_t max_query_len, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, void* out, int32_t out_dtype, uint32_t* error_word,
    cudaStream_t stream) {
  // Every host-side check runs before the shared scratch is touched, so a rejected call leaves
  // both the scratch and *error_word as they were.
  bool nothing = false;
  pa_status st = pa::check_attention_args(
      q, num_q_tokens, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
      query_start_loc, num_seqs, max_context_len, max_query_len, num_q_heads, num_kv_heads,
      head_dim, scale, out, out_dtype, &nothing);
  if (st != PA_OK) return st;
  if (nothing) {
    if (!error_word) return PA_OK;
    const cudaError_t e = cudaMemsetAsync(error_word, 0, sizeof(uint32_t), stream);
    if (e == cudaSuccess) return PA_OK;
    char msg[256];
    snprintf(msg, sizeof(msg), "pa_attention_noalloc: %s", cudaGetErrorString(e));
    pa::set_last_error(msg);
    return PA_ERR_CUDA;
  }
  const size_t need = pa_attention_workspace_size(num_seqs, num_q_tokens, num_q_heads,
                                                  num_kv_heads, head_dim, pa::kBlockSize,
                                                  max_context_len, max_query_len);
  if (need > PA_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "step needs %zu bytes of scratch; pa_attention_noalloc holds %u bytes "
             "(use pa_attention with a caller-allocated workspace)",
             need, PA_NOALLOC_SCRATCH_BYTES);
    pa::set_last_error(msg);
    return PA_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "pa_attention_noalloc scratch set-up: %s", cudaGetErrorString(e));
    pa::set_last_error(msg);
    return PA_ERR_CUDA;
  }
  // The header (error word, work counters) must start at zero; the rest is rewritten each call.
  e = cudaMemsetAsync(scratch, 0, PA_WORKSPACE_HEADER_BYTES, stream);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "pa_attention_noalloc: %s", cudaGetErrorString(e));
    pa::set_last_error(msg);
    return PA_ERR_CUDA;
  }
  st = pa_attention(q, num_q_tokens, k_cache, v_cache, cache, block_tables,
                                    max_blocks_per_seq, context_lens, query_start_loc, num_seqs,
                                    max_context_len, max_query_len, num_q_heads, num_kv_heads,
                                    head_dim, scale, out, out_dtype, scratch,
                                    PA_NOALLOC_SCRATCH_BYTES, stream);
  if (st != PA_OK || !error_word) return st;
  e = cudaMemcpyAsync(error_word, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "pa_attention_noalloc: %s", cudaGetErrorString(e));
    pa::set_last_error(msg);
    return PA_ERR_CUDA;
  }
  return PA_OK;
}
