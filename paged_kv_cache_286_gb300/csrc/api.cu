// C-ABI entry points of libpagedattn: host-side validation, workspace layout, TMA descriptors
// for the block pool, and the device error word.  Every host-detectable problem is reported
// before anything is launched; nothing here allocates device memory.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace {

thread_local std::string g_last_error;
thread_local cudaEvent_t g_before = nullptr;
thread_local cudaEvent_t g_after = nullptr;
thread_local cudaEvent_t g_pf_before = nullptr;
thread_local cudaEvent_t g_pf_after = nullptr;
thread_local uint64_t* g_span = nullptr;
thread_local uint64_t g_wait_ns = pa::kWaitLimitNs;
thread_local int32_t g_skip_copy = 0;

pa_status fail(pa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

pa_status cuda_fail(cudaError_t e, const char* where) {
  return fail(PA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view of a pool tensor: rows = num_blocks * num_kv_heads * block_size, cols = head_dim;
// one box = 16 rows (times heads_per_box: the tiles of consecutive kv heads of a block are
// consecutive rows) x 128 bytes with the 128-byte swizzle.
pa_status encode_pool_map(CUtensorMap* map, const void* base, const pa_cache_desc& c,
                          int heads_per_box = 1) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const bool fp8 = c.cache_dtype == PA_FP8_E4M3;
  const cuuint64_t rows = static_cast<cuuint64_t>(c.num_blocks) * c.num_kv_heads *
                          static_cast<cuuint64_t>(c.block_size);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(c.head_dim), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(c.head_dim) * (fp8 ? 1 : 2)};
  const cuuint32_t box[2] = {fp8 ? 128u : 64u,
                             static_cast<cuuint32_t>(c.block_size * heads_per_box)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return PA_OK;
}

// 4-D view of a bf16 pool with head_dim 128 for whole-tile copies: (64 columns, 8 rows,
// 2 column halves, 8-row groups) with byte strides (-, 256, 128, 2048).  One box of
// {64, 8, 2, 2} is a (block, kv head) tile of 16 rows, landing in shared memory as
// [2 row groups][2 halves][8 rows][128 bytes] with the 128-byte swizzle.
pa_status encode_pool_tile_map(CUtensorMap* map, const void* base, const pa_cache_desc& c) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t rows = static_cast<cuuint64_t>(c.num_blocks) * c.num_kv_heads *
                          static_cast<cuuint64_t>(c.block_size);
  const cuuint64_t dims[4] = {64, 8, 2, rows / 8};
  const cuuint64_t strides[3] = {256, 128, 2048};
  const cuuint32_t box[4] = {64, 8, 2, 2};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled (pool tiles) failed (%d)", int(r));
  return PA_OK;
}

// 3-D view of q [T][Hq][D] bf16; one box = (64 columns, G heads, 128 / G tokens) = 128 rows
// of 128 bytes with the 128-byte swizzle, the q tile of one prefill work item.
pa_status encode_q_map(CUtensorMap* map, const void* q, int32_t T, int32_t Hq, int32_t D,
                       int32_t G) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                              static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(Hq) * D * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (%d)", int(r));
  return PA_OK;
}

pa_status check_cache_desc(const pa_cache_desc* c, bool for_attention) {
  if (!c) return fail(PA_ERR_INVALID_ARG, "cache descriptor is NULL");
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0 || c->block_size <= 0)
    return fail(PA_ERR_INVALID_ARG, "cache descriptor has a non-positive size");
  if (c->block_size != pa::kBlockSize)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d is not built (16 is)", c->block_size);
  if (c->cache_dtype != PA_BF16 && c->cache_dtype != PA_FP8_E4M3)
    return fail(PA_ERR_UNSUPPORTED, "cache_dtype %d is not built", c->cache_dtype);
  if (c->cache_dtype == PA_FP8_E4M3 &&
      !(std::isfinite(c->k_scale) && std::isfinite(c->v_scale) && c->k_scale > 0.f &&
        c->v_scale > 0.f))
    return fail(PA_ERR_INVALID_ARG, "E4M3 cache needs finite positive k_scale and v_scale");
  if (c->head_dim % 16 != 0)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d is not a multiple of 16", c->head_dim);
  if (for_attention) {
    const bool ok = c->cache_dtype == PA_FP8_E4M3 ? c->head_dim == 128
                                                  : (c->head_dim == 64 || c->head_dim == 128);
    if (!ok)
      return fail(PA_ERR_UNSUPPORTED,
                  "attention over head_dim %d with this cache dtype is not built", c->head_dim);
  }
  // The kernels address a pool row (block, kv head, slot) with a signed 32-bit TMA coordinate.
  const int64_t rows = int64_t(c->num_blocks) * c->num_kv_heads * c->block_size;
  if (rows > int64_t(INT32_MAX))
    return fail(PA_ERR_INVALID_ARG,
                "pool too large: %lld rows of (block, kv head, slot), at most 2^31 - 1",
                static_cast<long long>(rows));
  return PA_OK;
}

}  // namespace

namespace pa {

WsLayout workspace_layout(int32_t S, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                          int32_t max_ctx, int32_t max_q) {
  WsLayout w{};
  const int32_t G = Hkv > 0 ? Hq / Hkv : 1;
  // the partition size depends only on the shape (not on the cache dtype): sized as if chunks
  // longer than kDecodeMaxQuery queries go to the prefill path
  const int64_t tpt = std::max(1, kRowsPerTile / std::max(1, G));
  const int64_t qtiles = (std::max<int64_t>(1, std::min(max_q, kDecodeMaxQuery)) + tpt - 1) / tpt;
  const int64_t maxblk = (std::max(1, max_ctx) + kBlockSize - 1) / kBlockSize;
  // Largest partition of 32 or fewer blocks that still yields enough work items to fill the
  // GPU; a partition never has fewer than 8 blocks (2 per warp).
  int32_t pblk = 8;
  for (int32_t cand : {32, 16}) {
    const int64_t items = int64_t(S) * Hkv * qtiles * ((maxblk + cand - 1) / cand);
    if (items >= 1200) {
      pblk = cand;
      break;
    }
  }
  // Long contexts take longer partitions, up to 128 blocks (the split-KV kernel's 4 warps
  // hold one table entry per lane), while the longest sequence still has 8 of them and about
  // 1,000 items remain: 16 x 32K tokens go from 32 to 128 blocks, with a quarter of the
  // partials to write and merge.
  for (int32_t cand : {128, 64}) {
    const int64_t items = int64_t(S) * Hkv * qtiles * ((maxblk + cand - 1) / cand);
    if (cand > pblk && cand <= maxblk / 8 && items >= 1000) {
      pblk = cand;
      break;
    }
  }
  w.pblk = pblk;
  w.pmax = static_cast<int32_t>((maxblk + pblk - 1) / pblk);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = PA_WORKSPACE_HEADER_BYTES;
  w.item_start = off;
  off = up(off + sizeof(int32_t) * (size_t(std::max(S, 0)) + 1));
  w.pf_item_start = off;
  off = up(off + sizeof(int32_t) * (size_t(std::max(S, 0)) + 1));
  w.pf_order = off;
  off = up(off + sizeof(int32_t) * size_t(std::max(S, 1)));
  w.merge_start = off;
  off = up(off + sizeof(int32_t) * (size_t(std::max(S, 0)) + 1));
  const size_t rows = size_t(std::max(T, 0)) * size_t(std::max(Hq, 0));
  const size_t parts = w.pmax > 1 ? size_t(w.pmax) : 0;
  w.part_lse = off;
  off = up(off + sizeof(float) * rows * parts);
  w.part_o = off;
  off = up(off + sizeof(float) * rows * parts * size_t(std::max(D, 0)));
  w.total = off;
  return w;
}

cudaError_t launch_info_impl(const void* kern, int threads, int smem_bytes, LaunchInfo* out) {
  struct Entry {
    const void* kern;
    int dev;
    LaunchInfo info;
  };
  static std::mutex mu;
  static Entry table[64];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].kern == kern && table[i].dev == dev) {
      *out = table[i].info;
      return cudaSuccess;
    }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  LaunchInfo li;
  e = cudaDeviceGetAttribute(&li.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&li.per_sm, kern, threads, smem_bytes);
  if (e != cudaSuccess) return e;
  if (li.per_sm < 1) li.per_sm = 1;
  if (used < 64) table[used++] = Entry{kern, dev, li};
  *out = li;
  return cudaSuccess;
}

// Lets other translation units of the library report a host-side error through
// pa_last_error_string.
void set_last_error(const char* msg) { g_last_error = msg; }

pa_status check_attention_args(const void* q, int32_t num_q_tokens, const void* k_cache,
                               const void* v_cache, const pa_cache_desc* cache,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, const int32_t* query_start_loc,
                               int32_t num_seqs, int32_t max_context_len, int32_t max_query_len,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               float scale, const void* out, int32_t out_dtype, bool* nothing) {
  g_last_error.clear();
  *nothing = false;
  if (num_seqs < 0 || num_q_tokens < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
  pa_status st = check_cache_desc(cache, true);
  if (st != PA_OK) return st;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PA_ERR_INVALID_ARG, "non-positive head count or head_dim");
  if (num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                num_q_heads, num_kv_heads);
  if (num_q_heads / num_kv_heads > kDecodeMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "GQA group of %d q heads per kv head is not built (<= 16)",
                num_q_heads / num_kv_heads);
  if (head_dim != cache->head_dim || num_kv_heads != cache->num_kv_heads)
    return fail(PA_ERR_INVALID_ARG, "head_dim / num_kv_heads disagree with the cache descriptor");
  if (out_dtype != PA_FP32 && out_dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "out_dtype %d is not built", out_dtype);
  if (!(std::isfinite(scale))) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
  if (num_seqs == 0 || num_q_tokens == 0) {
    *nothing = true;
    return PA_OK;
  }
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start_loc || !out)
    return fail(PA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (max_blocks_per_seq <= 0 || max_context_len <= 0 || max_query_len <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq, max_context_len and max_query_len must "
                                    "be positive");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start_loc, 4))
    return fail(PA_ERR_INVALID_ARG, "misaligned pointer (q, out and caches need 16 bytes)");
  return PA_OK;
}

}  // namespace pa

extern "C" {

const char* pa_version(void) { return "0.1.0"; }

const char* pa_last_error_string(void) { return g_last_error.c_str(); }

void pa_set_kernel_timing_events(void* before, void* after) {
  g_before = static_cast<cudaEvent_t>(before);
  g_after = static_cast<cudaEvent_t>(after);
}

void pa_set_prefill_timing_events(void* before, void* after) {
  g_pf_before = static_cast<cudaEvent_t>(before);
  g_pf_after = static_cast<cudaEvent_t>(after);
}

void pa_set_kernel_span_buffer(uint64_t* device_buffer) { g_span = device_buffer; }

void pa_set_wait_limit_ns(uint64_t ns) { g_wait_ns = ns ? ns : pa::kWaitLimitNs; }

void pa_test_skip_one_copy(int32_t enable) { g_skip_copy = enable ? 1 : 0; }

pa_status pa_workspace_init(void* workspace, cudaStream_t stream) {
  g_last_error.clear();
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(workspace, 0, PA_WORKSPACE_HEADER_BYTES, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pa_workspace_init");
  return PA_OK;
}

pa_status pa_selftest_wait_timeout(void* workspace, uint64_t limit_ns, cudaStream_t stream) {
  g_last_error.clear();
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(workspace, 4)) return fail(PA_ERR_INVALID_ARG, "misaligned workspace");
  if (limit_ns == 0 || limit_ns > 10ull * pa::kWaitLimitNs)
    return fail(PA_ERR_INVALID_ARG, "limit_ns must be in (0, 10 s]");
  cudaError_t e =
      pa::launch_wait_timeout_selftest(static_cast<uint32_t*>(workspace), limit_ns, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pa_selftest_wait_timeout launch");
  return PA_OK;
}

pa_status pa_check_error(void* workspace, cudaStream_t stream, uint32_t* word_out) {
  g_last_error.clear();
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace is NULL");
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(word), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "pa_check_error");
  if (word_out) *word_out = word;
  if (word & PA_DEVERR_TIMEOUT)
    return fail(PA_ERR_TIMEOUT, "a device-side wait timed out (error word 0x%x)", word);
  if (word)
    return fail(PA_ERR_OUT_OF_RANGE,
                "device saw an out-of-range block id, slot or length (error word 0x%x)", word);
  return PA_OK;
}

pa_status pa_cache_append(const void* k, const void* v, const int64_t* slot_mapping,
                          int32_t num_tokens, void* k_cache, void* v_cache,
                          const pa_cache_desc* cache, void* workspace, cudaStream_t stream) {
  g_last_error.clear();
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
  pa_status st = check_cache_desc(cache, false);
  if (st != PA_OK) return st;
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace is NULL");
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8) || !aligned(workspace, 4))
    return fail(PA_ERR_INVALID_ARG, "misaligned pointer (k, v and caches need 16 bytes)");
  cudaError_t e = pa::launch_cache_append(k, v, slot_mapping, num_tokens, k_cache, v_cache,
                                          *cache, static_cast<uint32_t*>(workspace), stream);
  if (e != cudaSuccess) return cuda_fail(e, "pa_cache_append launch");
  return PA_OK;
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const pa_cache_desc* cache,
                         const int32_t* block_pairs, int32_t num_pairs, void* workspace,
                         cudaStream_t stream) {
  g_last_error.clear();
  if (num_pairs < 0 || num_pairs > 65535)
    return fail(PA_ERR_INVALID_ARG, "num_pairs must be in [0, 65535]");
  pa_status st = check_cache_desc(cache, false);
  if (st != PA_OK) return st;
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace is NULL");
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_pairs) return fail(PA_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 4) ||
      !aligned(workspace, 4))
    return fail(PA_ERR_INVALID_ARG, "misaligned pointer (caches need 16 bytes)");
  cudaError_t e = pa::launch_copy_blocks(k_cache, v_cache, *cache, block_pairs, num_pairs,
                                         static_cast<uint32_t*>(workspace), stream);
  if (e != cudaSuccess) return cuda_fail(e, "pa_copy_blocks launch");
  return PA_OK;
}

size_t pa_attention_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int32_t max_context_len, int32_t max_query_len) {
  (void)block_size;
  return pa::workspace_layout(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                              max_context_len, max_query_len)
      .total;
}

pa_status pa_attention(const void* q, int32_t num_q_tokens, const void* k_cache,
                       const void* v_cache, const pa_cache_desc* cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, const int32_t* query_start_loc,
                       int32_t num_seqs, int32_t max_context_len, int32_t max_query_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                       void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  bool nothing = false;
  pa_status st = pa::check_attention_args(
      q, num_q_tokens, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
      query_start_loc, num_seqs, max_context_len, max_query_len, num_q_heads, num_kv_heads,
      head_dim, scale, out, out_dtype, &nothing);
  if (st != PA_OK) return st;
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace is NULL");
  if (nothing) return PA_OK;
  if (!aligned(workspace, 256))
    return fail(PA_ERR_INVALID_ARG, "misaligned pointer (the workspace needs 256 bytes)");
  const pa::WsLayout ws = pa::workspace_layout(num_seqs, num_q_tokens, num_q_heads, num_kv_heads,
                                               head_dim, max_context_len, max_query_len);
  if (workspace_bytes < ws.total)
    return fail(PA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                ws.total);
  pa::PoolMaps maps;
  // boxes of one or two kv heads' rows (two only for single-token E4M3 decode, where no
  // prefill tile reads these maps)
  const int hpi = pa::decode_heads_per_item(*cache, num_q_heads, num_kv_heads, max_query_len);
  if ((st = encode_pool_map(&maps.k2, k_cache, *cache, hpi)) != PA_OK) return st;
  if ((st = encode_pool_map(&maps.v2, v_cache, *cache, hpi)) != PA_OK) return st;

  const int32_t G = num_q_heads / num_kv_heads;
  const bool use_prefill = pa::prefill_path_enabled(*cache, num_q_heads, num_kv_heads) &&
                           pa::routes_to_prefill(max_query_len, G);
  // whole (block, kv head) tiles of bf16 head_dim 128 pools in one copy: the split-KV kernel's
  // and the prefill tiles' loads
  if (cache->cache_dtype == PA_BF16 && cache->head_dim == 128) {
    if ((st = encode_pool_tile_map(&maps.k4, k_cache, *cache)) != PA_OK) return st;
    if ((st = encode_pool_tile_map(&maps.v4, v_cache, *cache)) != PA_OK) return st;
    maps.has_k4 = true;
  }
  if (use_prefill) {
    if ((st = encode_q_map(&maps.q3, q, num_q_tokens, num_q_heads, head_dim, G)) != PA_OK)
      return st;
    maps.has_q3 = true;
  }

  pa::AttnArgs a{q, num_q_tokens, k_cache, v_cache, *cache, block_tables, max_blocks_per_seq,
                 context_lens, query_start_loc, num_seqs, max_context_len, max_query_len,
                 num_q_heads, num_kv_heads, head_dim, scale, out, out_dtype, workspace,
                 workspace_bytes, stream};
  a.pf_before = g_pf_before;
  a.pf_after = g_pf_after;
  a.wait_ns = g_wait_ns;
  a.skip_copy = g_skip_copy;
  a.span = g_span;
  cudaError_t e = pa::launch_attention(a, ws, maps, use_prefill, g_before, g_after);
  if (e != cudaSuccess) return cuda_fail(e, "pa_attention launch");
  return PA_OK;
}

}  // extern "C"
