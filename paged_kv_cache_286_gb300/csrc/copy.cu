// Whole-block copies inside the pool, the device half of copy-on-write ("Serving LLMs with vLLM:
// Continuous Batching and PagedAttention Explained", section "Copy-on-Write": before a sequence
// writes into a block that other sequences share, the engine copies that block to a fresh one
// and points only this sequence's table at the copy).
//
// One CTA row per (pair, 16-byte column chunk group): 16-byte loads and stores of the
// [num_kv_heads][block_size][head_dim] image of a block, K and V.  HBM-bound.
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_cache,
                                                          uint4* __restrict__ v_cache,
                                                          const int32_t* __restrict__ pairs,
                                                          int32_t num_pairs, int32_t num_blocks,
                                                          int64_t vec_per_block,
                                                          uint32_t* __restrict__ err) {
  const int32_t pr = blockIdx.y;
  if (pr >= num_pairs) return;
  const int32_t src = __ldg(pairs + 2 * pr), dst = __ldg(pairs + 2 * pr + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, PA_DEVERR_BLOCK_ID);
    return;
  }
  const int64_t s0 = static_cast<int64_t>(src) * vec_per_block;
  const int64_t d0 = static_cast<int64_t>(dst) * vec_per_block;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < vec_per_block; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    k_cache[d0 + i] = k_cache[s0 + i];
    v_cache[d0 + i] = v_cache[s0 + i];
  }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const pa_cache_desc& c,
                               const int32_t* pairs, int32_t num_pairs, uint32_t* err,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t bytes = static_cast<int64_t>(c.num_kv_heads) * c.block_size * c.head_dim *
                        (c.cache_dtype == PA_FP8_E4M3 ? 1 : 2);
  const int64_t vecs = bytes / 16;
  const int64_t per_cta = 256;
  const unsigned gx = static_cast<unsigned>(std::min<int64_t>((vecs + per_cta - 1) / per_cta, 64));
  dim3 grid(gx, static_cast<unsigned>(num_pairs));
  copy_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4*>(k_cache),
                                               static_cast<uint4*>(v_cache), pairs, num_pairs,
                                               c.num_blocks, vecs, err);
  return cudaGetLastError();
}

}  // namespace pa
