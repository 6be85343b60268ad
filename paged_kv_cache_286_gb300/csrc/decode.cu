// Split-KV paged attention for decode tokens and short query runs, plus its log-sum-exp merge.
//
// What it computes ("Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained",
// section "Attention Over Scattered Blocks"): for every query token i of sequence s at position
// p_i and every q head, softmax(scale * q . k_j) over keys j <= p_i, applied to the values, where
// key/value j live in physical block block_tables[s][j / 16] at offset j % 16.
//
// Design (GB300 / sm_103a):
//  * Work item = (sequence, kv head, tile of 8 or 16 rows, KV partition of `pblk` blocks).  A row
//    is a (query token, q head of the GQA group) pair, so one item loads each K/V block once for
//    the whole group and for as many of the sequence's query tokens as the tile holds.  16-row
//    tiles (both halves of the MMA's M) serve groups above 8 and multi-token runs of up to 16
//    rows; single-token decode keeps 8-row tiles, the cheaper instance.  Runs with more rows
//    (long chunks, speculative verify with GQA) go to the tensor-core prefill tiles when those
//    are built for the pool, and otherwise take several tiles here.  Single-token E4M3 decode
//    with 4 q heads per kv head takes two kv heads per item, filling the 8 rows.
//  * A plan kernel turns context lengths into per-sequence item counts; the attention kernel is
//    persistent, takes items from an atomic counter, and starts its CTAs while the plan runs
//    (programmatic dependent launch).
//  * Each of the CTA's 4 warps owns every 4th block of the partition and streams it through its
//    own ring of shared-memory stages: one lane issues 2-D TMA tile copies of the (block, head)
//    K and V tiles (128-byte swizzle) after reading the block id from the table, completion is
//    counted on the stage's mbarrier.  The HBM stream is the whole cost of decode.
//  * Scores and P.V run on warp-level tensor-core MMAs (m16n8k16): S = Q K^T with the rows as M
//    (an 8-row tile pads M to 16), and O^T = V^T P^T so that the probabilities feed the second
//    MMA straight from the first one's accumulators.  bf16 caches: P is split into bf16 hi + lo
//    parts, which keeps P exact to ~2^-16.  E4M3 caches: K and V are converted to f16 in
//    registers (exact), q is scaled by a power of two per row into f16 range, P is f16.
//  * Online softmax in the log2 domain per warp; the 4 warps' (m, l, O) are merged in shared
//    memory; an item that covers the whole sequence writes `out`, otherwise it writes a
//    normalised partial and its log-sum-exp, which the merge kernel combines.
#include <math_constants.h>

#include <algorithm>
#include <climits>
#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

struct DecodeParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* qsl;
  int32_t* item_start;
  int32_t* pf_item_start;  // [S+1] prefill item prefix sums over the runs in claim order
  int32_t* pf_order;       // [S] the runs with prefill items, longest item first
  int32_t* merge_start;    // [S+1] prefix sums of the rows the merge combines
  float* part_lse;
  float* part_o;
  void* out;
  WsHeader* hdr;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;           // q heads per kv head
  int32_t num_blocks;
  int32_t max_context_len;
  int32_t max_query_len;
  int32_t pblk;
  int32_t pmax;
  int32_t decode_max_query;  // longer query runs go to the prefill-tile path
  int32_t decode_max_rows;   // so do runs of more (token x head) rows than one decode tile
  int32_t rows_per_tile;   // 8 * RT of the decode kernel instance
  int32_t heads_per_item;  // HPI of the decode kernel instance
  int32_t out_bf16;
  float score_log2;        // scale * log2(e) (* k_scale for E4M3)
  float v_out_scale;       // v_scale for E4M3, else 1
  uint64_t* span;          // benchmark hook: [first CTA start, last CTA end] in ns, or NULL
  int32_t wait_at_end;     // launched after the prefill kernel: wait for it only at the end
  int32_t sms;             // SMs of the device (the plan's SM split)
  int32_t kv_tile_bytes;   // bytes of one (block, kv head) tile of K plus V
  uint64_t wait_ns;        // limit of every bounded wait
  int32_t skip_copy;       // test hook: item 0 leaves out its first tile copy (see pa.h)
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Partitions of a decode-path sequence of L keys.
__device__ __forceinline__ int partitions_of(const DecodeParams& p, int L) {
  return ceil_div(ceil_div(L, kBlockSize), p.pblk);
}

// Items of one sequence on the decode path (0 if it belongs to the prefill path or is invalid).
__device__ __forceinline__ int decode_items_of(const DecodeParams& p, int n, int L, bool* bad) {
  *bad = false;
  if (n <= 0) {
    *bad = (n < 0);
    return 0;
  }
  if (n > L || L > p.max_context_len || n > p.max_query_len ||
      L > p.max_blocks_per_seq * kBlockSize) {
    *bad = true;
    return 0;
  }
  if (n > p.decode_max_query || n * p.group > p.decode_max_rows) return 0;
  const int tpt = p.rows_per_tile / (p.group * p.heads_per_item);  // query tokens per tile
  const int qtiles = ceil_div(n, tpt);
  const int nparts = partitions_of(p, L);
  return p.num_kv_heads / p.heads_per_item * qtiles * nparts;
}

// Prefill-path items of one sequence: one per (kv head, 128-row tile of tokens x heads, key
// split of the tile).
__device__ __forceinline__ int prefill_items_of(const DecodeParams& p, int n, int L) {
  bool bad;
  if (decode_items_of(p, n, L, &bad) != 0 || bad || n <= 0) return 0;
  const int tpt = 128 / p.group;
  return p.num_kv_heads * ceil_div(n, tpt) * prefill_splits(n, L, p.group, p.pmax);
}

// One CTA: exclusive prefix sums over sequences of decode items, prefill items and merge rows
// (token x q head rows of decode-path sequences split into two or more partitions); resets the
// work counters and flags inconsistent lengths.
//
// It is launched early (programmatic dependent launch) and lets the attention kernel set up its
// CTAs meanwhile, but it waits for all earlier work of the stream before it reads anything: the
// caller may have written query_start_loc or context_lens with any kernel just before, and an
// earlier step may still be reading the workspace the plan overwrites.
__global__ void __launch_bounds__(1024) plan_kernel(const DecodeParams p) {
  grid_launch_dependents();  // the attention kernel may set up its CTAs meanwhile
  grid_dependency_wait();    // every earlier kernel of the stream is complete and visible
  constexpr int kN = 4;      // decode items, prefill items, merge rows, runs with prefill items
  constexpr int kSortMax = 2048;  // runs the plan orders by length (more: sequence order)
  __shared__ int warp_sums[32][kN];
  __shared__ int sort_key[kSortMax], sort_val[kSortMax], sort_cnt[kSortMax];
  __shared__ int carry_s[kN];
  __shared__ float red_f[32][3];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kN) carry_s[tid] = 0;
  // this thread's share of the cost model: prefill SM-microseconds, the longest prefill item,
  // split-KV bytes
  float pf_us = 0.f, pf_long = 0.f, dec_bytes = 0.f;
  __syncthreads();
  for (int base = 0; base < p.num_seqs; base += 1024) {
    const int s = base + tid;
    int cnt[kN] = {0, 0, 0};
    if (s < p.num_seqs) {
      const int n = p.qsl[s + 1] - p.qsl[s];
      const int L = p.context_lens[s];
      bool bad;
      cnt[0] = decode_items_of(p, n, L, &bad);
      if (bad) set_error(&p.hdr->error, PA_DEVERR_LENGTHS);
      cnt[1] = prefill_items_of(p, n, L);
      // rows the merge combines: split-KV sequences of two or more partitions, and prefill
      // runs whose tiles are split along the keys
      cnt[2] = ((cnt[0] > 0 && partitions_of(p, L) > 1) ||
                (cnt[1] > 0 && prefill_splits(n, L, p.group, p.pmax) > 1))
                   ? n * p.num_q_heads
                   : 0;
      cnt[3] = cnt[1] > 0 ? 1 : 0;
      if (cnt[0] > 0) dec_bytes += float(ceil_div(L, kBlockSize)) * p.num_kv_heads *
                                   float(p.kv_tile_bytes);
      if (cnt[1] > 0) {
        // every prefill item of the sequence: its 128-key slices times the slice cost
        const int tpt = 128 / p.group;
        const int tiles = ceil_div(n, tpt);
        const int ns = prefill_splits(n, L, p.group, p.pmax);
        for (int t = 0; t < tiles; ++t) {
          const int pos_last = L - n + min((t + 1) * tpt, n) - 1;
          const float us = float(ceil_div(pos_last / 128 + 1, ns)) * kTileSliceUs + kTileItemUs;
          pf_us += us * ns * p.num_kv_heads;
          pf_long = fmaxf(pf_long, us);
        }
      }
    }
    int x[kN];  // inclusive warp scans
#pragma unroll
    for (int k = 0; k < kN; ++k) x[k] = cnt[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int k = 0; k < kN; ++k) {
        const int y = __shfl_up_sync(0xffffffffu, x[k], o);
        if (lane >= o) x[k] += y;
      }
    }
    if (lane == 31)
#pragma unroll
      for (int k = 0; k < kN; ++k) warp_sums[warp][k] = x[k];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int k = 0; k < kN; ++k) {
        int w = warp_sums[lane][k];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += y;
        }
        warp_sums[lane][k] = w;  // inclusive over warps
      }
    }
    __syncthreads();
    int excl[kN];
#pragma unroll
    for (int k = 0; k < kN; ++k)
      excl[k] = carry_s[k] + (warp ? warp_sums[warp - 1][k] : 0) + x[k] - cnt[k];
    if (s < p.num_seqs) {
      p.item_start[s] = excl[0];
      p.merge_start[s] = excl[2];
      if (cnt[3]) {  // runs with prefill items, in sequence order
        p.pf_order[excl[3]] = s;
        if (excl[3] < kSortMax) {  // with their sort key and item count, for the ordering
          const int n = p.qsl[s + 1] - p.qsl[s];
          const int L = p.context_lens[s];
          sort_key[excl[3]] = ceil_div((L - 1) / 128 + 1, prefill_splits(n, L, p.group, p.pmax));
          sort_val[excl[3]] = s;
          sort_cnt[excl[3]] = cnt[1];
        }
      }
    }
    __syncthreads();
    if (tid == 1023)
#pragma unroll
      for (int k = 0; k < kN; ++k) carry_s[k] = excl[k] + cnt[k];
    __syncthreads();
  }
  // Claim order of the prefill runs: longest item first (its 128-key slices; ties by sequence),
  // so that the CTAs taking items from the counter end close together.  A bitonic sort in
  // shared memory, padded to a power of two with entries that sort last.
  const int R = carry_s[3];
  if (R > 1 && R <= 256) {
    // few runs: each thread counts the runs that go before its own (larger key, or the same
    // key and a lower sequence: a strict order), one barrier instead of the sort's stages
    int key = 0, val = 0, cnt = 0, rank = 0;
    if (tid < R) {
      key = sort_key[tid];
      val = sort_val[tid];
      cnt = sort_cnt[tid];
      for (int j = 0; j < R; ++j) {
        const int kj = sort_key[j];
        rank += kj > key || (kj == key && sort_val[j] < val);
      }
    }
    __syncthreads();
    if (tid < R) {
      sort_key[rank] = key;
      sort_val[rank] = val;
      sort_cnt[rank] = cnt;
    }
    __syncthreads();
    for (int i = tid; i < R; i += 1024) p.pf_order[i] = sort_val[i];
  } else if (R > 1 && R <= kSortMax) {
    int n2 = 2;
    while (n2 < R) n2 <<= 1;
    for (int i = R + tid; i < n2; i += 1024) {
      sort_key[i] = -1;
      sort_val[i] = INT_MAX;
      sort_cnt[i] = 0;
    }
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < n2; i += 1024) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const int ka = sort_key[i], kb = sort_key[ixj], va = sort_val[i], vb = sort_val[ixj];
            const bool a_first = ka > kb || (ka == kb && va < vb);
            const bool b_first = kb > ka || (kb == ka && vb < va);
            if ((i & k) == 0 ? b_first : a_first) {
              const int ca = sort_cnt[i];
              sort_key[i] = kb;
              sort_key[ixj] = ka;
              sort_val[i] = vb;
              sort_val[ixj] = va;
              sort_cnt[i] = sort_cnt[ixj];
              sort_cnt[ixj] = ca;
            }
          }
        }
        __syncthreads();
      }
    for (int i = tid; i < R; i += 1024) p.pf_order[i] = sort_val[i];
  }
  __syncthreads();
  // prefix sums of the prefill items over the runs in that order; ranks R .. S hold the total
  {
    int carry = 0;
    for (int base = 0; base < R; base += 1024) {
      const int r = base + tid;
      int c = 0;
      if (r < R && R <= kSortMax) {
        c = sort_cnt[r];
      } else if (r < R) {
        const int s = p.pf_order[r];
        c = prefill_items_of(p, p.qsl[s + 1] - p.qsl[s], p.context_lens[s]);
      }
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) warp_sums[warp][0] = x;
      __syncthreads();
      if (warp == 0) {
        int w = warp_sums[lane][0];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += y;
        }
        warp_sums[lane][0] = w;
      }
      __syncthreads();
      const int excl = carry + (warp ? warp_sums[warp - 1][0] : 0) + x - c;
      if (r < R) p.pf_item_start[r] = excl;
      carry += warp_sums[31][0];
      __syncthreads();
    }
    for (int r = R + tid; r <= p.num_seqs; r += 1024) p.pf_item_start[r] = carry_s[1];
  }
  // block reduction of the cost model
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    pf_us += __shfl_xor_sync(0xffffffffu, pf_us, o);
    pf_long = fmaxf(pf_long, __shfl_xor_sync(0xffffffffu, pf_long, o));
    dec_bytes += __shfl_xor_sync(0xffffffffu, dec_bytes, o);
  }
  if (lane == 0) {
    red_f[warp][0] = pf_us;
    red_f[warp][1] = pf_long;
    red_f[warp][2] = dec_bytes;
  }
  __syncthreads();
  float w_pf = 0.f, longest = 0.f, bytes = 0.f;
  for (int i = 0; i < 32; ++i) {
    w_pf += red_f[i][0];
    longest = fmaxf(longest, red_f[i][1]);
    bytes += red_f[i][2];
  }
  // SMs for the prefill tiles: the P that minimises the later of the two kernels' ends, the
  // prefill taking max(work / P, longest item) and the split-KV kernel streaming its bytes on
  // the other SMs (capped by the chip's HBM rate); the smallest P within 0.1 % of the best.
  // Thread P - 1 evaluates P.
  const int items = carry_s[1];
  const int pmax = max(1, min(p.sms, items));
  const bool search = bytes > 0.f && items > 0;
  const int P = tid + 1;
  float t = CUDART_INF_F;
  if (search && P <= pmax) {
    const float tp = fmaxf(w_pf / P, longest);
    const float rate = fminf(kHbmBytesPerUs, float(p.sms - P) * kDecodeSmBytesPerUs);
    t = fmaxf(tp, rate > 0.f ? bytes / rate : CUDART_INF_F);
  }
  __shared__ float red_t[32];
  __shared__ int red_p[32];
  float tm = t;
#pragma unroll
  for (int o = 16; o; o >>= 1) tm = fminf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
  if (lane == 0) red_t[warp] = tm;
  __syncthreads();
  tm = red_t[0];
  for (int i = 1; i < 32; ++i) tm = fminf(tm, red_t[i]);
  int cand = (search && P <= pmax && t <= tm * 1.001f) ? P : INT_MAX;
#pragma unroll
  for (int o = 16; o; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
  if (lane == 0) red_p[warp] = cand;
  __syncthreads();
  if (tid == 0) {
    int best_p = INT_MAX;
    for (int i = 0; i < 32; ++i) best_p = min(best_p, red_p[i]);
    if (best_p == INT_MAX) best_p = pmax;
    p.item_start[p.num_seqs] = carry_s[0];
    p.merge_start[p.num_seqs] = carry_s[2];
    p.hdr->decode_counter = 0;
    p.hdr->prefill_counter = 0;
    p.hdr->pf_ctas = static_cast<uint32_t>(best_p);
  }
}

template <int D, bool kFp8, int HPI = 1>
struct DecodeCfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kHeadBytes = kBlockSize * D * kElem;         // one (block, head) tile
  static constexpr int kTileBytes = HPI * kHeadBytes;               // the item's heads of a block
  static constexpr int kBoxCols = kFp8 ? 128 : 64;                  // elements per 128-B row
  static constexpr int kBoxes = D / kBoxCols;                       // TMA boxes per tile
  static constexpr int kBoxBytes = HPI * kBlockSize * 128;          // 16 HPI rows x 128 B
  // bf16 head_dim 128: the whole (block, head) tile in one 4-D copy (the pool seen as 64
  // columns x 8 rows x 2 column halves x 8-row groups), laid out [row group][half][8 rows]
  // [128 B], so one SM's copy engine moves twice the bytes per copy of two 2-D boxes
  static constexpr bool kTile4d = !kFp8 && D == 128;
  // shared-memory byte offset of 16-byte chunk `chunk` of key row `row` of a tile (swizzled)
  __device__ static uint32_t offset(int row, int chunk) {
    const uint32_t sw = static_cast<uint32_t>(((chunk & 7) ^ (row & 7)) << 4);
    if constexpr (kTile4d)
      return (row >> 3) * 2048 + (chunk >> 3) * 1024 + (row & 7) * 128 + sw;
    else
      return (chunk >> 3) * kBoxBytes + row * 128 + sw;
  }
  static constexpr int kStageBytes = 2 * kTileBytes;                // K tiles + V tiles
  static constexpr int kKSteps = D / 16;
  // consecutive kv heads of a block are consecutive rows of the pool, so one box of 16 HPI rows
  // holds all of them only when a head's tile is one 128-byte column box (E4M3, D 128)
  static_assert(HPI == 1 || kBoxes == 1, "several heads per item need one box per head tile");
};

template <int D, bool kFp8, int NST, int HPI>
constexpr int decode_smem_bytes() {
  using C = DecodeCfg<D, kFp8, HPI>;
  return 1024 /*alignment slack*/ + kDecodeWarps * NST * C::kStageBytes +
         kDecodeWarps * NST * 8 /*mbarriers*/ + 2 * 64 /*item slots*/;
}

struct ItemInfo {
  int s, h, qt, part, t0, n, L, nparts, blk_begin, blk_end, pos_base, rows, valid, idx;
};

// Instances with 2-stage rings are held to 3 CTAs per SM (at most 170 registers a thread): the
// kernel is latency-bound per SM, and the third CTA's warps, which the smaller rings leave room
// for in shared memory, keep more blocks in flight.
template <int D, bool kFp8, int NST, int RT, int HPI>
__global__ void __launch_bounds__(kDecodeWarps * 32, NST == 2 ? 3 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  // RT row tiles of 8 rows: rows quad and quad + 8 of the m16 MMA (RT = 2 uses both halves).
  // HPI kv heads per item (single-token decode only): row r is q head h0 * G + r, and the rows
  // of head h0 + i take their scores from, and add P V into O from, head i's tiles alone.
  using C = DecodeCfg<D, kFp8, HPI>;
  constexpr int R = 8 * RT;
  static_assert(HPI == 1 || RT == 1, "several heads per item use one 8-row tile");
  static_assert(sizeof(ItemInfo) <= 64 && C::kStageBytes * NST >= 16 * D * 4 + 2 * 16 * 4,
                "merge scratch must fit in a warp's stage buffers");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecodeWarps * NST * C::kStageBytes);
  ItemInfo* s_item = reinterpret_cast<ItemInfo*>(bars + kDecodeWarps * NST);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int quad = lane >> 2;  // fragment row group
  const int qc = lane & 3;     // position within the quad
  uint8_t* wbuf = smem + warp * NST * C::kStageBytes;
  uint64_t* wbars = bars + warp * NST;

  if (lane == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(&wbars[st], 1);
    fence_barrier_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncthreads();
  // Launched right after the plan, the kernel waits for it here.  Launched after the prefill
  // tiles (which waited for the plan before letting this kernel launch), the plan is already
  // complete: the kernel starts on the SMs the prefill left free and waits for the prefill
  // only before it exits, so that whatever follows on the stream sees both done.
  if (!p.wait_at_end) grid_dependency_wait();
  if (p.span && threadIdx.x == 0) atomicMin(reinterpret_cast<unsigned long long*>(p.span),
                                            static_cast<unsigned long long>(global_ns()));

  // (the plan's arrays are complete before this grid launches in either case, and L1 holds
  // nothing older than the launch, so plain loads read them)
  const int total_items = p.item_start[p.num_seqs];
  uint32_t it = 0;          // blocks this warp has consumed so far (stage / phase tracking)
  bool timed_out = false;

  // Thread 0 claims and decodes the CTA's next item while the current one streams, so the
  // atomic and the search over item_start stay off the critical path.
  auto fetch_item = [&](ItemInfo* dst) {
    ItemInfo info;
    const int item = static_cast<int>(atomicAdd(&p.hdr->decode_counter, 1u));
    info.valid = item < total_items;
    info.idx = item;
    if (info.valid) {
      int lo = 0, hi = p.num_seqs;  // largest s with item_start[s] <= item
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.item_start[mid] <= item) lo = mid; else hi = mid;
      }
      const int s = lo;
      const int t0 = p.qsl[s];
      const int n = p.qsl[s + 1] - t0;
      const int L = p.context_lens[s];
      const int tpt = R / (p.group * HPI);
      const int istart = p.item_start[s];
      const int qtiles = ceil_div(n, tpt);
      const int nblk = ceil_div(L, kBlockSize);
      const int nparts = ceil_div(nblk, p.pblk);
      int local = item - istart;
      const int part = local % nparts;
      local /= nparts;
      const int qt = local % qtiles;
      const int h = (local / qtiles) * HPI;                // first kv head of the item
      const int tok_begin = qt * tpt;
      const int tok_end = min(n, tok_begin + tpt);
      const int pos_max = L - n + tok_end - 1;           // last position in the tile
      const int blk_tile = pos_max / kBlockSize + 1;     // blocks the tile can see
      info.s = s; info.h = h; info.qt = qt; info.part = part; info.t0 = t0 + tok_begin;
      info.n = tok_end - tok_begin; info.L = L; info.nparts = nparts;
      info.blk_begin = min(part * p.pblk, blk_tile);
      info.blk_end = min((part + 1) * p.pblk, blk_tile);
      info.pos_base = L - n + tok_begin;                 // position of the tile's first token
      info.rows = info.n * p.group * HPI;
    }
    *dst = info;
  };
  if (threadIdx.x == 0) fetch_item(&s_item[0]);
  int cur = 0;

  while (true) {
    const bool any_timeout = __syncthreads_or(timed_out) != 0;
    const ItemInfo I = s_item[cur];
    if (!I.valid || any_timeout) break;
    const uint32_t it0 = it;  // blocks consumed before this item

    // ---- rows held by this lane: S rows quad + 8r; O^T columns 2qc, 2qc+1 of each tile --
    bool row_ok[RT];
    int row_tok[RT], row_pos[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int row = quad + 8 * r;
      row_ok[r] = row < I.rows;
      row_tok[r] = row_ok[r] ? row / (p.group * HPI) : 0;
      row_pos[r] = I.pos_base + row_tok[r];
    }
    const int my_head = HPI > 1 ? quad / p.group : 0;  // head of the item this lane's row uses
    const int pos_last = I.pos_base + I.n - 1;

    // ---- table entries of this warp's blocks, one per lane -----------------------------
    const int my_first = I.blk_begin + warp;
    const int nb_w = my_first < I.blk_end ? ceil_div(I.blk_end - my_first, kDecodeWarps) : 0;
    int phys_lane = -1;
    if (lane < nb_w) {
      const int b = my_first + lane * kDecodeWarps;
      phys_lane = __ldg(p.block_tables + static_cast<int64_t>(I.s) * p.max_blocks_per_seq + b);
      if (phys_lane < 0 || phys_lane >= p.num_blocks) {
        set_error(&p.hdr->error, PA_DEVERR_BLOCK_ID);
        phys_lane = -1;
      }
    }

    auto issue = [&](int k) {  // stage load for the warp's k-th block (all lanes call)
      const int phys = __shfl_sync(0xffffffffu, phys_lane, k);
      if (lane == 0) {
        const uint32_t st = (it0 + k) % NST;
        uint64_t* bar = &wbars[st];
        if (phys >= 0) {
          uint8_t* kt = wbuf + st * C::kStageBytes;
          uint8_t* vt = kt + C::kTileBytes;
          const int y = (phys * p.num_kv_heads + I.h) * kBlockSize;
          mbar_arrive_expect_tx(bar, C::kStageBytes);
          // test hook: the first stage of the first item claimed (whichever CTA claims it)
          // expects its bytes but gets no copy, so that the bounded wait on it expires
          const bool skip = p.skip_copy && I.idx == 0 && warp == 0 && k == 0;
          if (!skip) {
            if constexpr (C::kTile4d) {
              const int y4 = (phys * p.num_kv_heads + I.h) * 2;  // its first 8-row group
              tma_load_4d(kt, &kmap, 0, 0, 0, y4, bar);
              tma_load_4d(vt, &vmap, 0, 0, 0, y4, bar);
            } else {
#pragma unroll
              for (int bx = 0; bx < C::kBoxes; ++bx) {
                tma_load_2d(kt + bx * C::kBoxBytes, &kmap, bx * C::kBoxCols, y, bar);
                tma_load_2d(vt + bx * C::kBoxBytes, &vmap, bx * C::kBoxCols, y, bar);
              }
            }
          }
        } else {
          mbar_arrive(bar);
        }
      }
    };

    const int npre = min(NST, nb_w);
    for (int k = 0; k < npre; ++k) issue(k);
    if (threadIdx.x == 0) fetch_item(&s_item[cur ^ 1]);  // read after the next loop-top barrier

    // ---- q fragments (A operand of S = Q K^T): a0/a2 row quad, a1/a3 row quad + 8 -------
    uint32_t qa[C::kKSteps][4];
    float row_scale[RT];
#pragma unroll
    for (int ks = 0; ks < C::kKSteps; ++ks) qa[ks][1] = qa[ks][3] = 0u;  // rows 8..15 (RT = 1)
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int row = quad + 8 * r;
      const __nv_bfloat16* qrow =
          p.q + (static_cast<int64_t>(I.t0 + row_tok[r]) * p.num_q_heads + I.h * p.group +
                 (row_ok[r] ? row % (p.group * HPI) : 0)) * D;
      if constexpr (!kFp8) {
        row_scale[r] = p.score_log2;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          const uint32_t* src = reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * qc);
          qa[ks][r] = row_ok[r] ? __ldg(src) : 0u;
          qa[ks][2 + r] = row_ok[r] ? __ldg(src + 4) : 0u;
        }
      } else {
        // k index 2c,2c+1 of a k-step <-> d 4c,4c+1; k index 2c+8,2c+9 <-> d 4c+2,4c+3
        uint2 raw[C::kKSteps];
        float amax = 0.f;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          raw[ks] = row_ok[r] ? __ldg(reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * qc))
                              : make_uint2(0u, 0u);
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16lo_to_f32(raw[ks].x)),
                                         fabsf(bf16hi_to_f32(raw[ks].x))),
                                   fmaxf(fabsf(bf16lo_to_f32(raw[ks].y)),
                                         fabsf(bf16hi_to_f32(raw[ks].y)))));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // power of two e with amax * 2^e < 2^15 (f16 range), exact scaling
        int ex = 0;
        if (amax > 0.f) frexpf(amax, &ex);
        const int e = max(-100, min(100, 15 - ex));
        const float up = ldexpf(1.f, e);
        row_scale[r] = p.score_log2 * ldexpf(1.f, -e);
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          qa[ks][r] = pack_f16x2(bf16lo_to_f32(raw[ks].x) * up, bf16hi_to_f32(raw[ks].x) * up);
          qa[ks][2 + r] =
              pack_f16x2(bf16lo_to_f32(raw[ks].y) * up, bf16hi_to_f32(raw[ks].y) * up);
        }
      }
    }

    float m_run[RT], l_run[RT];  // running max (log2 domain) and this lane's share of the sum
    float oacc[RT][C::kKSteps][4];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      m_run[r] = -CUDART_INF_F;
      l_run[r] = 0.f;
#pragma unroll
      for (int j = 0; j < C::kKSteps; ++j)
        oacc[r][j][0] = oacc[r][j][1] = oacc[r][j][2] = oacc[r][j][3] = 0.f;
    }

    for (int k = 0; k < nb_w; ++k) {
      const uint32_t st = it % NST;
      const uint32_t parity = (it / NST) & 1u;
      // every lane polls; the outcome is made warp-uniform before any lane acts on it
      if (!__all_sync(0xffffffffu, mbar_wait(&wbars[st], parity, p.wait_ns))) {
        if (lane == 0) set_error(&p.hdr->error, PA_DEVERR_TIMEOUT);
        timed_out = true;
        // drain the other loads in flight, each with its own bounded wait
        for (int k2 = k + 1; k2 < min(nb_w, k + NST); ++k2)
          mbar_wait(&wbars[(it + (k2 - k)) % NST], ((it + (k2 - k)) / NST) & 1u, p.wait_ns);
        break;
      }
      const int phys = __shfl_sync(0xffffffffu, phys_lane, k);
      if (phys >= 0) {
        const int blk = my_first + k * kDecodeWarps;
        const int key0 = blk * kBlockSize;
        const uint32_t kbase = smem_u32(wbuf + st * C::kStageBytes);
        const uint32_t vbase = kbase + C::kTileBytes;

        // ---- S = Q K^T for the block's 16 keys (two n-tiles of 8 keys) -------------------
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
          const int krow = 8 * nt + (lane & 7);
          if constexpr (!kFp8) {
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              const int chunk = 4 * kk + (lane >> 3);  // 16-byte chunk = 8 d
              const uint32_t addr = kbase + C::offset(krow, chunk);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(addr, b0, b1, b2, b3);
              mma_bf16(sacc[nt], qa[2 * kk], b0, b1);
              mma_bf16(sacc[nt], qa[2 * kk + 1], b2, b3);
            }
          } else {
#pragma unroll
            for (int hi = 0; hi < HPI; ++hi) {
              // head hi's scores; a lane keeps those of its own row's head
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int kk = 0; kk < D / 64; ++kk) {
                const int chunk = 4 * kk + (lane >> 3);  // 16-byte chunk = 16 d = one k-step
                const uint32_t addr = kbase + hi * C::kHeadBytes + krow * 128 +
                                      (((chunk & 7) ^ (krow & 7)) << 4);
                uint32_t rr[4];
                ldsm_x4(addr, rr[0], rr[1], rr[2], rr[3]);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                  uint32_t b0, b1;
                  e4m3x4_to_f16x2x2(rr[m], b0, b1);
                  mma_f16(acc, qa[4 * kk + m], b0, b1);
                }
              }
              if (hi == 0 || my_head == hi) {
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[nt][i] = acc[i];
              }
            }
          }
        }

        // keys past the tile's last position hold stale slots: zero their V (may be NaN)
        const int nvalid = min(kBlockSize, pos_last + 1 - key0);
        uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;  // keys 2qc.., keys 8+2qc..
        if (nvalid < kBlockSize) {
          vm_lo = (2 * qc < nvalid ? 0x0000ffffu : 0u) | (2 * qc + 1 < nvalid ? 0xffff0000u : 0u);
          vm_hi = (8 + 2 * qc < nvalid ? 0x0000ffffu : 0u) |
                  (9 + 2 * qc < nvalid ? 0xffff0000u : 0u);
        }

        // ---- online softmax for rows quad + 8r over keys 8nt + 2qc + e ------------------
        uint32_t pb[RT][4];  // P^T fragments: bf16 hi pair 0, hi pair 1, lo 0, lo 1 (or f16)
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          float sv[4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int kidx = key0 + 8 * nt + 2 * qc + e;
              const bool ok = row_ok[r] && kidx <= row_pos[r];
              sv[2 * nt + e] = ok ? sacc[nt][2 * r + e] * row_scale[r] : -CUDART_INF_F;
            }
          float mloc = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
          mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
          mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
          // Lazy rescale: the exponent base m_run moves only when a row's max exceeds it by
          // more than 2^8 (p stays <= 256, exact in the P formats used); the final division
          // uses the same base, so the result is unchanged.
          const bool grow = mloc > m_run[r] + kLazyRescaleLog2;
          float alpha = 1.f;
          if (grow) {
            alpha = (m_run[r] == -CUDART_INF_F) ? 0.f : fast_exp2(m_run[r] - mloc);
            m_run[r] = mloc;
          }
          const float m_use = (m_run[r] == -CUDART_INF_F) ? 0.f : m_run[r];
          float pr[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) pr[i] = fast_exp2(sv[i] - m_use);
          l_run[r] = l_run[r] * alpha + (pr[0] + pr[1]) + (pr[2] + pr[3]);
          if (__any_sync(0xffffffffu, grow)) {
            // O^T columns 2qc, 2qc+1 of tile r belong to rows 8r + 2qc (+1): held by lanes
            // 8qc and 8qc + 4
            const float alpha_a = __shfl_sync(0xffffffffu, alpha, 8 * qc);
            const float alpha_b = __shfl_sync(0xffffffffu, alpha, 8 * qc + 4);
#pragma unroll
            for (int j = 0; j < C::kKSteps; ++j) {
              oacc[r][j][0] *= alpha_a;
              oacc[r][j][1] *= alpha_b;
              oacc[r][j][2] *= alpha_a;
              oacc[r][j][3] *= alpha_b;
            }
          }
          if constexpr (!kFp8) {
            pb[r][0] = pack_bf16x2(pr[0], pr[1]);
            pb[r][1] = pack_bf16x2(pr[2], pr[3]);
            pb[r][2] = pack_bf16x2(pr[0] - bf16lo_to_f32(pb[r][0]),
                                   pr[1] - bf16hi_to_f32(pb[r][0]));
            pb[r][3] = pack_bf16x2(pr[2] - bf16lo_to_f32(pb[r][1]),
                                   pr[3] - bf16hi_to_f32(pb[r][1]));
          } else {
            pb[r][0] = pack_f16x2(pr[0], pr[1]);
            pb[r][1] = pack_f16x2(pr[2], pr[3]);
          }
        }

        // ---- O^T += V^T P^T (one V^T fragment feeds every row tile) ----------------------
        if constexpr (!kFp8) {
          const int vrow = ((lane >> 4) << 3) + (lane & 7);  // key row of this lane's address
#pragma unroll
          for (int j = 0; j < C::kKSteps; ++j) {
            const int chunk = 2 * j + ((lane >> 3) & 1);
            const uint32_t addr = vbase + C::offset(vrow, chunk);
            uint32_t a[4];
            ldsm_x4_t(addr, a[0], a[1], a[2], a[3]);
            if (nvalid < kBlockSize) {
              a[0] &= vm_lo;
              a[1] &= vm_lo;
              a[2] &= vm_hi;
              a[3] &= vm_hi;
            }
#pragma unroll
            for (int r = 0; r < RT; ++r) {
              mma_bf16(oacc[r][j], a, pb[r][0], pb[r][1]);
              mma_bf16(oacc[r][j], a, pb[r][2], pb[r][3]);
            }
          }
        } else {
          const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
          for (int hi = 0; hi < HPI; ++hi) {
          // P^T columns of rows of other heads are zero for head hi's V
          uint32_t pbh[RT][2];
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            pbh[r][0] = (HPI == 1 || my_head == hi) ? pb[r][0] : 0u;
            pbh[r][1] = (HPI == 1 || my_head == hi) ? pb[r][1] : 0u;
          }
#pragma unroll
          for (int jj = 0; jj < D / 32; ++jj) {
            const int chunk = 2 * jj + (lane >> 4);
            const uint32_t addr = vbase + hi * C::kHeadBytes + vrow * 128 +
                                  (((chunk & 7) ^ (vrow & 7)) << 4);
            uint32_t rr[4];  // (keys 0-7, chunk 2jj), (8-15, 2jj), (0-7, 2jj+1), (8-15, 2jj+1)
            ldsm_x4_t(addr, rr[0], rr[1], rr[2], rr[3]);
            if (nvalid < kBlockSize) {
              rr[0] &= vm_lo;
              rr[1] &= vm_hi;
              rr[2] &= vm_lo;
              rr[3] &= vm_hi;
            }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              // bytes (b0, b2) -> keys 2qc, 2qc+1 at d 2u; (b1, b3) -> the same keys at d 2u+1
              uint32_t a[4];
              e4m3x4_to_f16x2x2(prmt(rr[2 * h2], 0u, 0x3120u), a[0], a[1]);
              e4m3x4_to_f16x2x2(prmt(rr[2 * h2 + 1], 0u, 0x3120u), a[2], a[3]);
#pragma unroll
              for (int r = 0; r < RT; ++r) mma_f16(oacc[r][2 * jj + h2], a, pbh[r][0], pbh[r][1]);
            }
          }
          }
        }
      }
      __syncwarp();
      ++it;
      if (k + NST < nb_w) issue(k + NST);
    }
    if (timed_out) it = 0;  // results are void; phase tracking no longer matters

    // ---- per-warp state -> shared memory (this warp's own stage buffers) -----------------
    float* so = reinterpret_cast<float*>(wbuf);           // [16][D]
    float* sm = so + 16 * D;                               // [16]
    float* sl = sm + 16;                                   // [16]
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      float l_row = l_run[r];
      l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
      l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
#pragma unroll
      for (int j = 0; j < C::kKSteps; ++j) {
        int da, db;
        if constexpr (!kFp8) {
          da = 16 * j + quad;
          db = da + 8;
        } else {
          da = 16 * j + 2 * quad;
          db = da + 1;
        }
        const int ra = 8 * r + 2 * qc;
        so[ra * D + da] = oacc[r][j][0];
        so[(ra + 1) * D + da] = oacc[r][j][1];
        so[ra * D + db] = oacc[r][j][2];
        so[(ra + 1) * D + db] = oacc[r][j][3];
      }
      if (qc == 0) {
        sm[quad + 8 * r] = m_run[r];
        sl[quad + 8 * r] = l_row;
      }
    }
    __syncthreads();

    // ---- merge the 4 warps and write the output or the partial ---------------------------
    for (int e = threadIdx.x; e < I.rows * D; e += kDecodeWarps * 32) {
      const int r = e / D, d = e - r * D;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float* wsm = reinterpret_cast<const float*>(smem + w * NST * C::kStageBytes) +
                           16 * D;
        M = fmaxf(M, wsm[r]);
      }
      float Lsum = 0.f, O = 0.f;
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) {
          const float* wso = reinterpret_cast<const float*>(smem + w * NST * C::kStageBytes);
          const float mw = wso[16 * D + r];
          const float f = fast_exp2(mw - M);
          Lsum += wso[16 * D + 16 + r] * f;
          O += wso[r * D + d] * f;
        }
      }
      const float val = Lsum > 0.f ? O / Lsum * p.v_out_scale : 0.f;
      const int t = I.t0 + r / (p.group * HPI);
      const int hq = I.h * p.group + r % (p.group * HPI);
      const int64_t orow = static_cast<int64_t>(t) * p.num_q_heads + hq;
      if (I.nparts == 1) {
        if (p.out_bf16)
          reinterpret_cast<__nv_bfloat16*>(p.out)[orow * D + d] = __float2bfloat16_rn(val);
        else
          reinterpret_cast<float*>(p.out)[orow * D + d] = val;
      } else {
        const int64_t prow = orow * p.pmax + I.part;
        p.part_o[prow * D + d] = val;
        if (d == 0) p.part_lse[prow] = Lsum > 0.f ? M + __log2f(Lsum) : -CUDART_INF_F;
      }
    }
    __syncthreads();
    fence_proxy_async_smem();  // generic accesses to the stage buffers before the next TMA
    cur ^= 1;
  }
  if (p.span && threadIdx.x == 0)
    atomicMax(reinterpret_cast<unsigned long long*>(p.span) + 1,
              static_cast<unsigned long long>(global_ns()));
  if (p.wait_at_end) grid_dependency_wait();  // the prefill tiles of the step are complete
}

// Eight loads of kPer consecutive floats each, issued back to back in one asm block (so that
// they are in flight together whatever the register allocator prefers) before the merge uses
// any of the results.
template <int kPer>
__device__ __forceinline__ void load_batch8(const float* const (&src)[8], float (&v)[8][kPer]);

template <>
__device__ __forceinline__ void load_batch8<4>(const float* const (&src)[8], float (&v)[8][4]) {
  asm volatile(
      "ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%32];\n\t"
      "ld.global.nc.v4.f32 {%4, %5, %6, %7}, [%33];\n\t"
      "ld.global.nc.v4.f32 {%8, %9, %10, %11}, [%34];\n\t"
      "ld.global.nc.v4.f32 {%12, %13, %14, %15}, [%35];\n\t"
      "ld.global.nc.v4.f32 {%16, %17, %18, %19}, [%36];\n\t"
      "ld.global.nc.v4.f32 {%20, %21, %22, %23}, [%37];\n\t"
      "ld.global.nc.v4.f32 {%24, %25, %26, %27}, [%38];\n\t"
      "ld.global.nc.v4.f32 {%28, %29, %30, %31}, [%39];"
      : "=f"(v[0][0]), "=f"(v[0][1]), "=f"(v[0][2]), "=f"(v[0][3]), "=f"(v[1][0]),
        "=f"(v[1][1]), "=f"(v[1][2]), "=f"(v[1][3]), "=f"(v[2][0]), "=f"(v[2][1]),
        "=f"(v[2][2]), "=f"(v[2][3]), "=f"(v[3][0]), "=f"(v[3][1]), "=f"(v[3][2]),
        "=f"(v[3][3]), "=f"(v[4][0]), "=f"(v[4][1]), "=f"(v[4][2]), "=f"(v[4][3]),
        "=f"(v[5][0]), "=f"(v[5][1]), "=f"(v[5][2]), "=f"(v[5][3]), "=f"(v[6][0]),
        "=f"(v[6][1]), "=f"(v[6][2]), "=f"(v[6][3]), "=f"(v[7][0]), "=f"(v[7][1]),
        "=f"(v[7][2]), "=f"(v[7][3])
      : "l"(src[0]), "l"(src[1]), "l"(src[2]), "l"(src[3]), "l"(src[4]), "l"(src[5]),
        "l"(src[6]), "l"(src[7]));
}

template <>
__device__ __forceinline__ void load_batch8<2>(const float* const (&src)[8], float (&v)[8][2]) {
  asm volatile(
      "ld.global.nc.v2.f32 {%0, %1}, [%16];\n\t"
      "ld.global.nc.v2.f32 {%2, %3}, [%17];\n\t"
      "ld.global.nc.v2.f32 {%4, %5}, [%18];\n\t"
      "ld.global.nc.v2.f32 {%6, %7}, [%19];\n\t"
      "ld.global.nc.v2.f32 {%8, %9}, [%20];\n\t"
      "ld.global.nc.v2.f32 {%10, %11}, [%21];\n\t"
      "ld.global.nc.v2.f32 {%12, %13}, [%22];\n\t"
      "ld.global.nc.v2.f32 {%14, %15}, [%23];"
      : "=f"(v[0][0]), "=f"(v[0][1]), "=f"(v[1][0]), "=f"(v[1][1]), "=f"(v[2][0]),
        "=f"(v[2][1]), "=f"(v[3][0]), "=f"(v[3][1]), "=f"(v[4][0]), "=f"(v[4][1]),
        "=f"(v[5][0]), "=f"(v[5][1]), "=f"(v[6][0]), "=f"(v[6][1]), "=f"(v[7][0]),
        "=f"(v[7][1])
      : "l"(src[0]), "l"(src[1]), "l"(src[2]), "l"(src[3]), "l"(src[4]), "l"(src[5]),
        "l"(src[6]), "l"(src[7]));
}

// Combines the partials of one row: out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M).
template <int D>
__device__ __forceinline__ void merge_row(const DecodeParams& p, int64_t rid, int nparts,
                                          int lane) {
  const float* lse = p.part_lse + rid * p.pmax;
  float M = -CUDART_INF_F;
  for (int i = lane; i < nparts; i += 32) M = fmaxf(M, lse[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int kPer = D / 32;  // columns per lane
  constexpr int kBatch = 8;     // partitions whose loads are in flight together
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float wsum = 0.f;  // this lane's share; summed over the warp below
  const float* po = p.part_o + rid * p.pmax * D + lane * kPer;
  for (int base = 0; base < nparts; base += 32) {
    const int i = base + lane;
    const float w = (i < nparts && M != -CUDART_INF_F) ? fast_exp2(lse[i] - M) : 0.f;
    wsum += w;
    const int cnt = min(32, nparts - base);
#pragma unroll 1
    for (int j0 = 0; j0 < cnt; j0 += kBatch) {
      // issue the batch's loads first, then fold them in: a dependent load per partition
      // would leave one load in flight per warp
      float v[kBatch][kPer];
      // past the last partition a load repeats it (a written, finite partial) under a zero
      // weight, so the batch's loads are unconditional and go out back to back
      const float* src[8];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        src[u] = po + static_cast<int64_t>(base + min(j0 + u, cnt - 1)) * D;
      load_batch8<kPer>(src, v);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float wj = __shfl_sync(0xffffffffu, w, j0 + u);  // 0 past nparts
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] += wj * v[u][e];
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int64_t o = rid * D + lane * kPer + i;
    if (p.out_bf16)
      reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(acc[i] * inv);
    else
      reinterpret_cast<float*>(p.out)[o] = acc[i] * inv;
  }
}

// One warp per row (token, q head) of a sequence that was split into several partitions: the
// plan lists those rows (merge_start), and a grid of at most one resident wave strides over
// them.
template <int D>
// (At least 4 CTAs per SM, i.e. up to 64 registers a thread: room for the eight loads in flight
// of a row, with twice the rows in flight of two CTAs per SM and sixteen loads.)
__global__ void __launch_bounds__(256, 4) merge_kernel(const DecodeParams p) {
  grid_dependency_wait();  // the attention kernel's partials (and the plan) are complete
  const int lane = threadIdx.x & 31;
  const int total = p.merge_start[p.num_seqs];
  const int stride = gridDim.x * 8;
#pragma unroll 1
  for (int c = blockIdx.x * 8 + (threadIdx.x >> 5); c < total; c += stride) {
    // sequence of merge row c, the largest s with merge_start[s] <= c (merge_start is
    // non-decreasing from 0; a sequence without rows has an empty range): a 32-way search by
    // the warp, one coalesced load per round
    int lo = 0, span = p.num_seqs;
    while (span > 32) {
      const int step = (span + 31) >> 5;
      const int idx = lo + lane * step;
      const int start = idx < lo + span ? p.merge_start[idx] : INT_MAX;
      const int last = 31 - __clz(__ballot_sync(0xffffffffu, start <= c));
      lo += last * step;
      span = min(step, span - last * step);
    }
    const int start = lane < span ? p.merge_start[lo + lane] : INT_MAX;
    const int s = lo + 31 - __clz(__ballot_sync(0xffffffffu, start <= c));
    const int local = c - p.merge_start[s];
    const int t0 = p.qsl[s];
    const int n = p.qsl[s + 1] - t0, L = p.context_lens[s];
    const int64_t rid = static_cast<int64_t>(t0) * p.num_q_heads + local;
    bool bad;
    const int nparts = decode_items_of(p, n, L, &bad) > 0 ? partitions_of(p, L)
                                                         : prefill_splits(n, L, p.group, p.pmax);
    merge_row<D>(p, rid, nparts, lane);
  }
}

template <int D, bool kFp8, int NST, int RT, int HPI = 1>
static cudaError_t run_decode(const AttnArgs& a, const WsLayout& ws, const DecodeParams& p,
                              const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaEvent_t before, cudaEvent_t after) {
  constexpr int smem = decode_smem_bytes<D, kFp8, NST, HPI>();
  auto kern = decode_kernel<D, kFp8, NST, RT, HPI>;
  LaunchInfo li;
  cudaError_t e = launch_info(kern, kDecodeWarps * 32, smem, &li);
  if (e != cudaSuccess) return e;
  const int sms = li.sms, per_sm = li.per_sm;
  const int tpt = std::max(1, 8 * RT / (p.group * HPI));
  const int64_t qtiles_max = (std::min(a.max_query_len, p.decode_max_query) + tpt - 1) / tpt;
  const int64_t upper =
      static_cast<int64_t>(a.num_seqs) * (a.num_kv_heads / HPI) * qtiles_max * ws.pmax;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(upper, int64_t(sms) * per_sm));
  if (before) cudaEventRecord(before, a.stream);
  e = launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(kDecodeWarps * 32), smem,
                       a.stream, kmap, vmap, p);
  if (after) cudaEventRecord(after, a.stream);
  if (e != cudaSuccess) return e;
  if (ws.pmax > 1) {
    // at most one resident wave of 8-warp CTAs; the merge rows are fewer than all rows
    LaunchInfo mi;
    if ((e = launch_info(merge_kernel<D>, 256, 0, &mi)) != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(a.num_q_tokens) * a.num_q_heads;
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, int64_t(mi.sms) * mi.per_sm);
    if (blocks > 0)
      e = launch_dependent(merge_kernel<D>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                           a.stream, p);
  }
  return e;
}

int decode_heads_per_item(const pa_cache_desc& c, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t max_query_len) {
  // single-token E4M3 decode with 4 q heads per kv head fills an 8-row tile with two kv heads,
  // whose tiles are adjacent in the pool: one 4 KiB copy each for K and V per block
  const int G = num_kv_heads > 0 ? num_q_heads / num_kv_heads : 0;
  return (c.cache_dtype == PA_FP8_E4M3 && c.head_dim == 128 && G == 4 && num_kv_heads % 2 == 0 &&
          max_query_len == 1)
             ? 2
             : 1;
}

bool prefill_path_enabled(const pa_cache_desc& c, int32_t num_q_heads, int32_t num_kv_heads) {
  const int G = num_q_heads / num_kv_heads;
  const bool built = (c.cache_dtype == PA_BF16 && (c.head_dim == 128 || c.head_dim == 64)) ||
                     (c.cache_dtype == PA_FP8_E4M3 && c.head_dim == 128);
  return built && G >= 1 && G <= kRowsPerTile && 128 % G == 0;
}

cudaError_t launch_attention(const AttnArgs& a, const WsLayout& ws, const PoolMaps& maps,
                             bool use_prefill, cudaEvent_t before, cudaEvent_t after) {
  const CUtensorMap& kmap = maps.k2;
  const CUtensorMap& vmap = maps.v2;
  uint8_t* wsb = static_cast<uint8_t*>(a.workspace);
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.qsl = a.query_start_loc;
  p.item_start = reinterpret_cast<int32_t*>(wsb + ws.item_start);
  p.pf_item_start = reinterpret_cast<int32_t*>(wsb + ws.pf_item_start);
  p.pf_order = reinterpret_cast<int32_t*>(wsb + ws.pf_order);
  p.merge_start = reinterpret_cast<int32_t*>(wsb + ws.merge_start);
  p.part_lse = reinterpret_cast<float*>(wsb + ws.part_lse);
  p.part_o = reinterpret_cast<float*>(wsb + ws.part_o);
  p.out = a.out;
  p.hdr = reinterpret_cast<WsHeader*>(wsb);
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.cache.num_blocks;
  p.max_context_len = a.max_context_len;
  p.max_query_len = a.max_query_len;
  // An E4M3 block is half the bytes of a bf16 one: give E4M3 items twice the blocks (the
  // workspace, sized for the bf16 choice, then holds fewer partitions than it has room for;
  // pmax stays the row stride of the partial arrays).  Fewer, longer partitions also make the
  // merge cheaper.
  const bool fp8_cache = a.cache.cache_dtype == PA_FP8_E4M3;
  const int hpi = decode_heads_per_item(a.cache, a.num_q_heads, a.num_kv_heads,
                                        a.max_query_len);
  p.heads_per_item = hpi;
  p.pblk = (fp8_cache && ws.pblk <= 32) ? ws.pblk * 2 : ws.pblk;
  // a warp holds the table entries of its blocks of a partition one per lane
  if (p.pblk > kDecodeWarps * 32) return cudaErrorInvalidValue;
  p.pmax = ws.pmax;
  const bool prefill = use_prefill && prefill_path_enabled(a.cache, a.num_q_heads,
                                                          a.num_kv_heads);
  p.decode_max_query = prefill ? kDecodeMaxQuery : INT32_MAX;
  p.decode_max_rows = prefill ? kDecodeMaxRows : INT32_MAX;
  p.out_bf16 = a.out_dtype == PA_BF16;
  p.wait_ns = a.wait_ns;
  p.skip_copy = a.skip_copy;
  const float log2e = 1.4426950408889634f;
  const bool fp8 = a.cache.cache_dtype == PA_FP8_E4M3;
  p.score_log2 = a.scale * log2e * (fp8 ? a.cache.k_scale : 1.f);
  p.v_out_scale = fp8 ? a.cache.v_scale : 1.f;

  // 16-row tiles when a tile of 8 rows cannot hold the group, or when the decode-path query
  // runs (multi-token verify, short chunks) fill more than 8 rows; a mixed batch whose chunks
  // go to the prefill path keeps 8-row tiles for its single-token decodes.
  const int dec_q = std::min(a.max_query_len, p.decode_max_query);
  const bool mixed = prefill && routes_to_prefill(a.max_query_len, p.group);
  const bool rt2 = p.group > 8 || (!mixed && static_cast<int64_t>(dec_q) * p.group > 8);
  p.rows_per_tile = rt2 ? 16 : 8;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  p.kv_tile_bytes = 2 * kBlockSize * a.head_dim * (fp8 ? 1 : 2);
  p.span = a.span;

  e = launch_dependent(plan_kernel, dim3(1), dim3(1024), 0, a.stream, p);
  if (e != cudaSuccess) return e;
  // The prefill tiles (tensor pipe, key slices mostly from L2) and the split-KV decode (HBM)
  // share the GPU, one stream, each kernel launched early (programmatic dependent launch):
  // the prefill kernel waits for the plan, which has given it part of the SMs, and then lets
  // the split-KV kernel launch; its CTAs fill the SMs the prefill left free at once (and the
  // others as prefill CTAs end), and wait for the prefill kernel only before they exit.  Both
  // only read what the plan and the append wrote, and write disjoint output rows.
  if (prefill) {
    PrefillScratch scratch{p.part_lse, p.part_o, p.pmax};
    if ((e = launch_prefill(a, p.pf_item_start, p.pf_order, p.hdr, maps, scratch)) !=
        cudaSuccess)
      return e;
    p.wait_at_end = 1;
  }
  if (fp8 && hpi == 2)
    e = run_decode<128, true, 2, 1, 2>(a, ws, p, kmap, vmap, before, after);
  else if (fp8)
    e = rt2 ? run_decode<128, true, 4, 2>(a, ws, p, kmap, vmap, before, after)
            : run_decode<128, true, 4, 1>(a, ws, p, kmap, vmap, before, after);
  else if (a.head_dim == 128)  // whole-tile 4-D copies
    e = rt2 ? run_decode<128, false, 3, 2>(a, ws, p, maps.k4, maps.v4, before, after)
            : run_decode<128, false, 2, 1>(a, ws, p, maps.k4, maps.v4, before, after);
  else
    e = rt2 ? run_decode<64, false, 4, 2>(a, ws, p, kmap, vmap, before, after)
            : run_decode<64, false, 4, 1>(a, ws, p, kmap, vmap, before, after);
  return e;
}

}  // namespace pa
