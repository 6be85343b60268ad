// Slot-mapped cache append ("Serving LLMs with vLLM: Continuous Batching and PagedAttention
// Explained", section "Growing During Decode": each step appends the new token into the last
// block of its sequence; "Blocks and Block Tables": blocks are fixed-size and found through the
// table, which the caller folds into slot = block * block_size + offset).
//
// One thread moves 8 elements (16 bytes of bf16 input) of one (token, kv head) row for both K
// and V: coalesced 16-byte loads, 16-byte (bf16) or 8-byte (E4M3) stores into
// cache[slot / bs][head][slot % bs][:].  HBM- or launch-bound; no shared memory.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <bool kFp8>
__global__ void __launch_bounds__(256) cache_append_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    int32_t num_tokens, int32_t num_kv_heads, int32_t vec_per_row, int64_t total_slots,
    void* __restrict__ k_cache, void* __restrict__ v_cache, float k_scale, float v_scale,
    uint32_t* __restrict__ err) {
  grid_dependency_wait();    // launched early (programmatic dependent launch): inputs ready
  grid_launch_dependents();  // the step's plan kernel may launch meanwhile
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_token = static_cast<int64_t>(num_kv_heads) * vec_per_row;
  if (gid >= per_token * num_tokens) return;
  const int32_t t = static_cast<int32_t>(gid / per_token);
  const int64_t within = gid - static_cast<int64_t>(t) * per_token;  // head * vec + vec index
  const int32_t h = static_cast<int32_t>(within / vec_per_row);
  const int32_t c = static_cast<int32_t>(within - static_cast<int64_t>(h) * vec_per_row);
  const int64_t slot = __ldg(slots + t);
  if (slot < 0) return;
  if (slot >= total_slots) {
    if (c == 0 && h == 0) set_error(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / kBlockSize;
  const int64_t off = slot - blk * kBlockSize;
  // destination row (blk, h, off) of a [NB][Hkv][bs][D] pool, in 8-element units
  const int64_t row = (blk * num_kv_heads + h) * kBlockSize + off;
  const int64_t dst = row * vec_per_row + c;
  const uint4 kv = __ldg(k + gid);
  const uint4 vv = __ldg(v + gid);
  if constexpr (!kFp8) {
    reinterpret_cast<uint4*>(k_cache)[dst] = kv;
    reinterpret_cast<uint4*>(v_cache)[dst] = vv;
  } else {
    auto quant = [](uint4 x, float s) {
      // fl32(x) / s rounded to nearest (IEEE division), then E4M3 round-to-nearest-even with
      // saturation to +-448.
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t out[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_to_f32(w[2 * i]), s),
                                            __fdiv_rn(bf16hi_to_f32(w[2 * i]), s));
        const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_to_f32(w[2 * i + 1]), s),
                                            __fdiv_rn(bf16hi_to_f32(w[2 * i + 1]), s));
        out[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      return make_uint2(out[0], out[1]);
    };
    reinterpret_cast<uint2*>(k_cache)[dst] = quant(kv, k_scale);
    reinterpret_cast<uint2*>(v_cache)[dst] = quant(vv, v_scale);
  }
}

cudaError_t launch_cache_append(const void* k, const void* v, const int64_t* slots,
                                int32_t num_tokens, void* k_cache, void* v_cache,
                                const pa_cache_desc& c, uint32_t* err, cudaStream_t stream) {
  const int32_t vec_per_row = c.head_dim / 8;
  const int64_t threads = static_cast<int64_t>(num_tokens) * c.num_kv_heads * vec_per_row;
  if (threads == 0) return cudaSuccess;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  const int64_t total_slots = static_cast<int64_t>(c.num_blocks) * c.block_size;
  if (c.cache_dtype == PA_FP8_E4M3) {
    return launch_dependent(cache_append_kernel<true>, dim3(static_cast<unsigned>(grid)),
                            dim3(block), 0, stream, static_cast<const uint4*>(k),
                            static_cast<const uint4*>(v), slots, num_tokens, c.num_kv_heads,
                            vec_per_row, total_slots, k_cache, v_cache, c.k_scale, c.v_scale,
                            err);
  }
  return launch_dependent(cache_append_kernel<false>, dim3(static_cast<unsigned>(grid)),
                          dim3(block), 0, stream, static_cast<const uint4*>(k),
                          static_cast<const uint4*>(v), slots, num_tokens, c.num_kv_heads,
                          vec_per_row, total_slots, k_cache, v_cache, 1.f, 1.f, err);
}

}  // namespace pa
