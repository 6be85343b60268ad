// Host-side interfaces between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "pa.h"

namespace pa {

// Per-device launch facts of one kernel (SM count, resident CTAs per SM), with its dynamic
// shared-memory limit raised once per device: computed on first use and cached.
struct LaunchInfo {
  int sms = 0;
  int per_sm = 0;
};

// Cached per (kernel address, device): the function's C++ type is shared by every
// instantiation of a kernel template, so the key must be the address.
cudaError_t launch_info_impl(const void* kern, int threads, int smem_bytes, LaunchInfo* out);

template <typename Kernel>
cudaError_t launch_info(Kernel kern, int threads, int smem_bytes, LaunchInfo* out) {
  return launch_info_impl(reinterpret_cast<const void*>(kern), threads, smem_bytes, out);
}

// Everything pa_attention received, after host validation.
struct AttnArgs {
  const void* q;
  int32_t num_q_tokens;
  const void* k_cache;
  const void* v_cache;
  pa_cache_desc cache;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int32_t num_seqs;
  int32_t max_context_len;
  int32_t max_query_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  float scale;
  void* out;
  int32_t out_dtype;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  cudaEvent_t pf_before = nullptr;  // benchmark hook: recorded around the prefill kernel
  cudaEvent_t pf_after = nullptr;
  uint64_t* span = nullptr;         // benchmark hook: kernel start / end times (pa.h)
  uint64_t wait_ns = 0;             // limit of every bounded device-side wait
  int32_t skip_copy = 0;            // test hook (pa_test_skip_one_copy)
};

// Workspace carve-up; a pure function of the step's shape (see workspace_layout).
struct WsLayout {
  size_t item_start;  // int32 [num_seqs + 1], decode work-item prefix sums
  size_t pf_item_start;  // int32 [num_seqs + 1], prefill work-item prefix sums, by claim rank
  size_t pf_order;    // int32 [num_seqs], the sequence of each prefill claim rank
  size_t merge_start;  // int32 [num_seqs + 1], prefix sums of the rows (token x q head) that
                       // the merge combines: those of split-KV sequences with 2+ partitions
  size_t part_lse;    // float [num_q_tokens][num_q_heads][pmax], log2-domain log-sum-exp
  size_t part_o;      // float [num_q_tokens][num_q_heads][pmax][head_dim], normalised partials
  size_t total;
  int32_t pblk;       // blocks per KV partition
  int32_t pmax;       // partitions per sequence at most
};

WsLayout workspace_layout(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t max_context_len,
                          int32_t max_query_len);

cudaError_t launch_cache_append(const void* k, const void* v, const int64_t* slots,
                                int32_t num_tokens, void* k_cache, void* v_cache,
                                const pa_cache_desc& c, uint32_t* err, cudaStream_t stream);

void set_last_error(const char* msg);

// Host checks of pa_attention's arguments other than the workspace (clears, then sets, the
// calling thread's last error).  *nothing is set when the step has no query token or sequence.
pa_status check_attention_args(const void* q, int32_t num_q_tokens, const void* k_cache,
                               const void* v_cache, const pa_cache_desc* cache,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, const int32_t* query_start_loc,
                               int32_t num_seqs, int32_t max_context_len, int32_t max_query_len,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               float scale, const void* out, int32_t out_dtype, bool* nothing);

cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const pa_cache_desc& c,
                               const int32_t* pairs, int32_t num_pairs, uint32_t* err,
                               cudaStream_t stream);

// True when chunks with more than kDecodeMaxQuery queries run on the tcgen05 tile kernel
// (bf16 pool of head_dim 128 or 64, or E4M3 of 128; GQA group dividing 128); otherwise every
// sequence takes the split-KV kernel.
// Kv heads per split-KV work item (1 or 2) for a step of this shape; the pool's tensor maps
// then take boxes of 16 x that many rows.
int decode_heads_per_item(const pa_cache_desc& c, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t max_query_len);
bool prefill_path_enabled(const pa_cache_desc& c, int32_t num_q_heads, int32_t num_kv_heads);

// `qmap` (3-D view of q) is needed only when the prefill path is enabled and
// max_query_len > kDecodeMaxQuery; it may be NULL otherwise.
// Launch with programmatic stream serialization: the kernel may start while the previous kernel
// of the stream finishes, and waits (grid_dependency_wait) before reading its results.
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, int smem,
                                    cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct PoolMaps;
cudaError_t launch_attention(const AttnArgs& a, const WsLayout& ws, const PoolMaps& maps,
                             bool prefill, cudaEvent_t before, cudaEvent_t after);

struct WsHeader;

// Parameters of the tensor-core prefill kernels (prefill.cu, chunk.cu).
struct PrefillParams {
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* qsl;
  const int32_t* item_start;  // [S+1] prefix sums of prefill items over the runs in claim order
  const int32_t* order;       // [S] the sequence of each run in claim order
  void* out;
  WsHeader* hdr;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t num_blocks;
  int32_t out_bf16;
  float score_log2;   // scale * log2(e) (* k_scale for E4M3 pools)
  float v_out_scale;  // v_scale for E4M3 pools, else 1
  uint64_t wait_ns;   // limit of every bounded wait
  int32_t skip_copy;  // test hook: the first item claimed leaves out its first K copy
  uint64_t* span;     // benchmark hook: [first CTA start, last CTA end] in ns, or NULL
  float* part_lse;       // [T][Hq][pmax] log2-domain log-sum-exp of split partials
  float* part_o;         // [T][Hq][pmax][128] normalised split partials
  int32_t pmax;          // partials per row the workspace holds (>= the splits of a pair)
};

// Where split prefill tiles keep their partials (the workspace's split-KV arrays).
struct PrefillScratch {
  float* part_lse;
  float* part_o;
  int32_t pmax;
};


// Tensor maps of one call: the pool as 2-D rows (split-KV kernel, verify tiles), the pool as
// 4-D whole (block, kv head) tiles and q as 3-D tiles (prefill kernels; NULL when unused).
struct PoolMaps {
  CUtensorMap k2, v2, k4, v4, q3;
  bool has_k4 = false, has_q3 = false;
};

cudaError_t launch_prefill(const AttnArgs& a, const int32_t* item_start, const int32_t* order,
                           WsHeader* hdr,
                           const PoolMaps& maps, const PrefillScratch& scratch);


}  // namespace pa
