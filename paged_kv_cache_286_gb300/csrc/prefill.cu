// Causal chunked-prefill tiles on tcgen05 tensor cores.
//
// What it computes ("Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained",
// sections "Chunked Prefill", "Prefill Versus Decode", "Attention Over Scattered Blocks"): a
// prompt chunk of n tokens whose sequence holds L keys after this step's append sits at
// positions p_i = L - n + i; token i attends keys 0..p_i, fetched through the block table.
// The same causal run serves the verify step of speculative decoding (section "Speculative
// Decoding": the draft tokens are checked in one pass); every run of more than 16 tokens or
// more than 16 (token x head) rows comes here.
//
// Design (GB300 / sm_103a; written for bf16 K/V of head_dim 128, with instances for head_dim 64
// and for E4M3 pools described at the end):
//  * A tile is 128 rows, a row being (query token, q head of the GQA group), so the tile's
//    queries share every K/V tile they read.  One work item is a tile over a range of 128-key
//    slices: the tiles of very long runs are cut along the keys into several items
//    (prefill_splits), each writing a normalised partial and its log-sum-exp into the
//    workspace's split-KV arrays, which the merge kernel combines like the split-KV
//    partitions.  Persistent CTAs (one per SM, as many as the plan gives this kernel) take
//    items from an atomic counter in the order the plan gives (runs by their longest item,
//    longest first; within a run the last, longest tiles first); warp 0 claims the CTA's next
//    item while the current one runs.
//  * The pool is viewed by a 4-D tensor map as (64 columns, 8 rows, 2 column halves, 8-row
//    groups), so that one TMA copy brings a whole 16 x 128 (block, kv head) tile: 8 copies per
//    128 keys for K (lanes of warp 0, which also loads the q tile) and 8 for V (warp 6), into
//    two-stage rings.  One SM's TMA unit is limited by the number of copies rather than their
//    bytes, so whole-tile copies halve the copy time of a slice.  In shared memory a block's
//    tile is [2 row groups][2 halves][8 rows][128 bytes] with the 128-byte swizzle, i.e. 8-key
//    groups 2 KiB apart and the column halves 1 KiB apart, which the MMA descriptors express
//    as strides.
//  * tcgen05.mma, each issued from one thread: warp 1 S = Q K^T into one of three TMEM buffers
//    (128 x 128 fp32), warp 7 O += P V, with P read from TMEM and V from shared memory
//    (MN-major).  With one issuing thread for both, every wait of that thread sat between
//    two groups of MMAs while the tensor pipe ran dry; with two, each waits on its own.  The
//    softmax threads write P over the S they have read, as bf16 hi and lo parts (keys 0-63: hi
//    in columns 0-31, lo in 32-63; keys 64-127 likewise in 64-127; P V is exact to ~2^-16 like
//    the decode path), and S of slice j+3 goes into a buffer once the P V of slice j has read
//    it, so the S MMAs run up to three slices ahead of the softmax.  TMEM: S / P 3 x 128
//    columns, O 128.
//  * Softmax, two threads per row (TMEM lane), one for keys (and O columns) 0-63 in warps 2-5
//    and one for 64-127 in warps 8-11: each reads its half row of S from TMEM once, masks keys
//    beyond the row's position, keeps the running max in the log2 domain (set by the first
//    slice that shows the row a key) and rescales O in TMEM only when the max grows by more
//    than 2^8 (the final division uses the same max, so the result is exact), and finally
//    divides O by the row sum.  The two threads of a row agree on its max, and at the end add
//    their sums, through a shared-memory slot and an mbarrier of the pair.  A warp can only
//    reach the lane quarter of its own SM sub-partition; the per-slice work of a row is
//    bound by instruction latency rather than issue, and the second warp on each
//    sub-partition hides it (whole rows on one warp each took a quarter longer per slice).
//  * Pool slots past the sequence's end (stale, possibly NaN) in its last loaded block are
//    zeroed in shared memory before P V reads them (by the P V issuer's warp); blocks past the
//    tile's last position are not loaded, and their rows keep older, finite V data (the ring
//    starts zeroed) under P = 0.  K there only feeds masked scores.
//  * The epilogue stages each warp's rows in a region of its own (swizzled) and writes whole
//    rows per instruction, instead of one scattered 16-byte piece per row and instruction.
//  * Items follow one another without a block-wide barrier: warp 0 claims the next item while
//    the current one runs and loads its q tile and first K/V slices as soon as the S MMAs and
//    stages of the current one are done with theirs, so the next item's first S is computed
//    while the softmax warps write the current one's output; only its first P V waits for
//    them to have read O.  (K and V rings of two stages make room for the staging region; the
//    slice period did not change with the ring depth.)
//  * Launched right after the plan (programmatic dependent launch): the CTAs beyond the SMs
//    the plan gives this kernel end at once, and the split-KV kernel launches onto the rest.
//  * Every wait is bounded; on expiry the CTA records PA_DEVERR_TIMEOUT, stops, lets the copies
//    and MMAs it issued finish (bounded waits again) and frees its tensor memory.
//  * head_dim 64: one 64-column q half, the (block, kv head) tiles of 2 KiB by one 2-D box of the
//    pool (16 rows x 128 bytes) each, S from four MMAs, P V with N = 64 into 64 O columns.
//  * E4M3 pools (head_dim 128): the MMAs are kind::f8f6f4, whose operands are both 8-bit, so
//    K and V are read as stored (2 KiB tiles, one 2-D box each) while q and P are split into
//    E4M3 parts.  The softmax warps turn the bf16 q tile into three parts (hi, mid, lo of q
//    times a per-row power of two that puts the row's max in [128, 256)), whose three S MMAs
//    per 32 dims accumulate into one S; P, made 2^8 times larger to keep small values clear of
//    E4M3's subnormal floor, is written as hi and lo parts, and the lazy rescale threshold is
//    2^0.5 so that it stays under 448.  k_scale and the row's q scale go into the scores,
//    v_scale into the output.
#include <math_constants.h>

#include <algorithm>
#include <climits>
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace pf {
constexpr int kRows = 128;
constexpr int kKeys = 128;
constexpr int kStages = 2;   // K and V ring depth
constexpr int kPBufs = 3;    // S / P buffers in TMEM (a slice's P is written over its S)
constexpr int kHalf = 16384;  // one 64-column half of the q tile (bf16), or one E4M3 q part
constexpr int kStageBytes = 65536;
constexpr int kXBufs = 3;
// Shared memory, by the pool's element type: the q tile (bf16: two 64-column halves; E4M3 pools:
// the bf16 tile lands there and becomes three E4M3 parts), the K and V rings (a stage is the 8
// (block, kv head) tiles of 128 keys: 32 KiB bf16, 16 KiB E4M3), the epilogue's staging of the
// softmax warps' rows, the control block, the row exchanges' mbarriers (one per lane quarter)
// and slots.
struct Layout {
  int q_bytes, stage_stride, k, v, stage, ctl, xbar, xslot, smem;
  __host__ __device__ constexpr Layout(bool fp8)
      : q_bytes(fp8 ? 3 * kHalf : 2 * kHalf),
        stage_stride(fp8 ? 16384 : 32768),
        k(q_bytes),
        v(k + kStages * stage_stride),
        stage(v + kStages * stage_stride),
        ctl(stage + kStageBytes),
        xbar(ctl + 384),
        xslot(xbar + 32),
        smem(1024 + xslot + kXBufs * kRows * 4) {}
};
constexpr int kQ = 0;
constexpr int kVWarp = 6;     // V producer (warp 0 loads q and K)
constexpr int kPvWarp = 7;    // P V issuer (warp 1 issues S)
// The softmax: warps 2-5 take keys 0-63 of their rows and warps 8-11 keys 64-127, and the
// pairs exchange row sums and maxima through shared memory.
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;

constexpr uint32_t kTmemCols = 512;
// S / P buffer b at columns 128 b; then the O accumulator
constexpr uint32_t kOCol = kPBufs * 128;
static_assert(kOCol + 128 == kTmemCols, "TMEM columns");
constexpr float kRescaleLog2 = 8.f;
constexpr float kRescaleLog2Fp8 = 0.5f;  // E4M3 P (times 2^8) stays under 2^8.5 < 448
}  // namespace pf

struct PfItem {
  int s, h, t0, ntok, pos0, L, nblk_tile, valid, first;
  int j0, nj;       // the item's slices of the tile: j0 .. j0 + nj - 1
  int ns, k;        // splits of the tile and this item's split
};

struct PfCtl {
  uint64_t q_full, k_full[pf::kStages], k_empty[pf::kStages], v_full[pf::kStages],
      v_empty[pf::kStages], s_full[pf::kPBufs], p_full[pf::kPBufs], o_done[pf::kPBufs], drain[2],
      q_empty, o_free, item_full[2], item_empty[2], q_ready;
  uint32_t tmem_base;
  int abort_flag;
  int v_zero_from[pf::kStages], v_zero_to[pf::kStages];
  uint32_t v_bad[pf::kStages];
  PfItem item[2];  // by the parity of the item count: warp 0 fills one while the other is read
};
static_assert(sizeof(PfCtl) <= 384, "control block too large");
static_assert(pf::Layout(false).smem <= 232448 && pf::Layout(true).smem <= 232448,
              "more shared memory than a CTA may have");

// Floats mapped to ints of the same order (an involution), so that integer atomicMax takes the
// max of floats.  The empty slot INT_MIN is below every mapped float and reads as -0.0f.
__device__ __forceinline__ int float_order_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float order_key_float(int k) {
  return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff));
}

// A thread's kC consecutive 32-bit TMEM columns from `cols` (its lane) into registers.
template <int kC>
__device__ __forceinline__ void tmem_ld_row(uint32_t cols, uint32_t (&v)[kC]) {
#pragma unroll
  for (int c = 0; c < kC / 32; ++c)
    tmem_ld32(cols + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
  tmem_wait_ld();
}

// Claims the next item from the counter and decodes it.  The plan ordered the runs longest
// item first; within a run the items go from its last (longest) tile back.
__device__ __forceinline__ PfItem claim_item(const PrefillParams& p, int total) {
  PfItem it;
  const int item = static_cast<int>(atomicAdd(&p.hdr->prefill_counter, 1u));
  it.valid = item < total;
  it.first = item == 0;
  if (!it.valid) return it;
  int lo = 0, hi = p.num_seqs;  // the last rank whose first item is at or before this one
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.item_start[mid] <= item) lo = mid; else hi = mid;
  }
  const int s = p.order[lo];
  const int t0 = p.qsl[s];
  const int n = p.qsl[s + 1] - t0;
  const int L = p.context_lens[s];
  const int tpt = pf::kRows / p.group;
  const int ns = prefill_splits(n, L, p.group, p.pmax);
  // counted from the run's last item: the q tile is the outer index, so the last (longest)
  // tiles of every kv head come first
  const int local = p.item_start[lo + 1] - 1 - item;
  const int k = local % ns;
  const int ti = local / ns;
  const int h = ti % p.num_kv_heads;
  const int qt = ti / p.num_kv_heads;
  const int i0 = qt * tpt;
  it.s = s;
  it.h = h;
  it.t0 = t0 + i0;
  it.ntok = min(tpt, n - i0);
  it.pos0 = L - n + i0;
  it.L = L;
  it.ns = ns;
  it.k = k;
  const int pmax = it.pos0 + it.ntok - 1;
  const int nkv = pmax / pf::kKeys + 1;  // slices of the tile
  const int per = (nkv + ns - 1) / ns;
  it.j0 = min(nkv, k * per);
  it.nj = min(nkv, it.j0 + per) - it.j0;
  it.nblk_tile = pmax / kBlockSize + 1;
  return it;
}

template <int D, bool kFp8>
__global__ void __launch_bounds__(pf::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(!kFp8 || D == 128, "E4M3 tiles have head_dim 128");
  constexpr pf::Layout kL(kFp8);
  constexpr int kBlk = 16 * D * (kFp8 ? 1 : 2);  // bytes of one (block, kv head) tile
  constexpr int kOC = D / 2;     // O columns of a softmax thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PfCtl* ctl = reinterpret_cast<PfCtl*>(smem + kL.ctl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launched right after the plan (programmatic dependent launch): wait for its items and SM
  // budget, let the split-KV kernel launch onto the SMs this kernel leaves, and end the CTAs
  // beyond the budget at once.
  grid_dependency_wait();
  grid_launch_dependents();
  if (blockIdx.x >= ld_cg(&p.hdr->pf_ctas)) return;
  if (p.span && threadIdx.x == 0) atomicMin(reinterpret_cast<unsigned long long*>(p.span),
                                            static_cast<unsigned long long>(global_ns()));
  const int total = p.item_start[p.num_seqs];

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int i = 0; i < pf::kStages; ++i) {
      mbar_init(&ctl->k_full[i], 1);
      mbar_init(&ctl->k_empty[i], 1);
      mbar_init(&ctl->v_full[i], 1);
      mbar_init(&ctl->v_empty[i], 1);
    }
    // S of slice g goes into buffer g % 3 once the P V of slice g - 3 has read the P there
    // (o_done); the softmax writes the slice's P over its S (p_full).  One s_full / p_full /
    // o_done per buffer keeps every waiter within one phase of its barrier.
    for (int i = 0; i < pf::kPBufs; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], pf::kSoftmaxThreads);
      mbar_init(&ctl->o_done[i], 1);
    }
    mbar_init(&ctl->drain[0], 1);
    mbar_init(&ctl->drain[1], 1);
    // Items flow through the roles without a block-wide barrier between them: warp 0 claims
    // the next item into the other slot once the other warps have read the item that was
    // there (item_empty: one lane of each of the 11), loads its q tile once the S MMAs of the
    // item before have read theirs (q_empty), and the P V issuer starts the next item's O once
    // the softmax warps have read the last one (o_free: one lane of each of the 8).
    mbar_init(&ctl->q_empty, 1);
    mbar_init(&ctl->q_ready, pf::kSoftmaxThreads / 32);  // E4M3 pools: q parts written
    mbar_init(&ctl->o_free, pf::kSoftmaxThreads / 32);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->item_full[i], 1);
      mbar_init(&ctl->item_empty[i], pf::kThreads / 32 - 1);
    }
    for (int q = 0; q < 4; ++q)
        mbar_init(reinterpret_cast<uint64_t*>(smem + kL.xbar) + q, 2);  // one lane a warp
    ctl->abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    ctl->item[0] = claim_item(p, total);
    mbar_arrive(&ctl->item_full[0]);
  }
  int* xslot = reinterpret_cast<int*>(smem + kL.xslot);  // [kXBufs][kRows]
  for (int i = tid; i < pf::kXBufs * pf::kRows; i += pf::kThreads) xslot[i] = INT_MIN;
  // the V ring starts zeroed: rows of blocks a slice does not load are then always finite
  for (int i = tid; i < pf::kStages * kL.stage_stride / 16; i += pf::kThreads)
    reinterpret_cast<uint4*>(smem + kL.v)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc(&ctl->tmem_base, pf::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  uint32_t tc = 0;  // KV slices processed by this CTA so far (ring / phase tracking)
  uint32_t ic = 0;  // items processed by this CTA so far
  uint32_t xc = 0;  // exchanges of this softmax thread's pair so far (slot / phase tracking)
  uint32_t kiss = 0, viss = 0, qiss = 0;  // producers: K, V and q fills issued (final drain)
  const int G = p.group;

  auto fail = [&](uint32_t bits) {
    set_error(&p.hdr->error, bits);
    ctl->abort_flag = 1;
  };
  // all lanes wait; the outcome is warp-uniform
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, p.wait_ns));
    if (!ok && lane == 0) fail(PA_DEVERR_TIMEOUT);
    return ok;
  };

  while (true) {
    // warp 0 wrote the item itself; the others wait for it and hand the slot back once read
    if (warp != 0 && !wait(&ctl->item_full[ic & 1u], (ic >> 1) & 1u)) break;
    const PfItem I = ctl->item[ic & 1u];
    if (warp != 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->item_empty[ic & 1u]);
    }
    if (!I.valid || *reinterpret_cast<volatile int*>(&ctl->abort_flag)) break;

    if (warp == 0 || warp == pf::kVWarp) {
      // ------------------------------------------------------- producers (TMA): warp 0 q and K,
      // warp 6 V.  Two issuing warps double the rate at which tile copies enter the TMA unit.
      // The q tile of an item goes in once the S MMAs of the item before are done with theirs.
      const bool k_side = warp == 0;
      bool ok = !k_side || ic == 0 || wait(&ctl->q_empty, (ic - 1) & 1u);
      if (ok && k_side && lane == 0) {
        mbar_arrive_expect_tx(&ctl->q_full, pf::kRows * D * 2);
        tma_load_3d(smem + pf::kQ, &qmap, 0, I.h * G, I.t0, &ctl->q_full);
        if constexpr (D == 128)
          tma_load_3d(smem + pf::kQ + pf::kHalf, &qmap, 64, I.h * G, I.t0, &ctl->q_full);
      }
      if (ok && k_side) ++qiss;
      // Block-table entries are read 32 at a time (lane l holds block 32 * grp + l) with the
      // next group prefetched, so no TMA issue waits on a dependent table load.
      const int32_t* trow = p.block_tables + static_cast<int64_t>(I.s) * p.max_blocks_per_seq;
      auto tab_load = [&](int grp) -> int {
        const int jb = 32 * grp + lane;
        return jb < I.nblk_tile ? __ldg(trow + jb) : -1;
      };
      int grp_cur = I.j0 >> 2;
      int tab_cur = tab_load(grp_cur);
      int tab_next = tab_load(grp_cur + 1);
      const int yrow0 = I.h * 2;  // 8-row group of (block 0, this kv head)
      // this lane's (block, kv head) tile of a slice into its place in a stage: one 4-D copy
      // for bf16 head_dim 128 (the whole tile), one 2-D box of 16 rows x 128 B otherwise
      auto tile_copy = [&](int stage_off, const CUtensorMap* map, int group, uint64_t* bar) {
        uint8_t* dst = smem + stage_off + lane * kBlk;
        if constexpr (D == 128 && !kFp8) tma_load_4d(dst, map, 0, 0, 0, group, bar);
        else tma_load_2d(dst, map, 0, group * 8, bar);
      };
      for (int jj = 0; ok && jj < I.nj; ++jj) {
        const int j = I.j0 + jj;
        const int grp = j >> 2;
        if (grp != grp_cur) {
          tab_cur = tab_next;
          tab_next = tab_load(grp + 1);
          grp_cur = grp;
        }
        // block ids of slice j for lanes 0-7 (-1 = not loaded), plus masks of loadable / bad
        // ones
        const int e = __shfl_sync(0xffffffffu, tab_cur, 8 * (j & 3) + (lane & 7));
        const int jb = 8 * j + lane;
        int phys = -1;
        bool bad = false;
        if (lane < 8 && jb < I.nblk_tile) {
          if (e < 0 || e >= p.num_blocks) {
            set_error(&p.hdr->error, PA_DEVERR_BLOCK_ID);
            bad = true;
          } else {
            phys = e;
          }
        }
        const uint32_t okm = __ballot_sync(0xffffffffu, phys >= 0);
        const uint32_t badm = __ballot_sync(0xffffffffu, bad);
        const uint32_t bytes = __popc(okm) * static_cast<uint32_t>(kBlk);
        const int ycoord = (phys * p.num_kv_heads) * 2 + yrow0;
        const uint32_t g = tc + jj, st = g % pf::kStages;
        if (k_side) {
          if (!(ok = wait(&ctl->k_empty[st], ((g / pf::kStages) & 1u) ^ 1u))) break;
          if (lane == 0) {
            if (bytes) mbar_arrive_expect_tx(&ctl->k_full[st], bytes);
            else mbar_arrive(&ctl->k_full[st]);
          }
          __syncwarp();
          // test hook: lane 0's copy of the first slice of the first item claimed is left
          // out (its bytes are still expected), so that the bounded waits on that stage expire
          const bool skip = p.skip_copy && I.first && jj == 0 && lane == 0;
          if (phys >= 0 && !skip)
            tile_copy(kL.k + st * kL.stage_stride, &kmap, ycoord, &ctl->k_full[st]);
          ++kiss;
        } else {
          if (!(ok = wait(&ctl->v_empty[st], ((g / pf::kStages) & 1u) ^ 1u))) break;
          if (lane == 0) {
            // rows the P V issuer clears: keys past the last valid one, and bad blocks
            const int valid_end = min(I.L, I.nblk_tile * kBlockSize) - j * pf::kKeys;
            ctl->v_zero_from[st] = max(0, min(pf::kKeys, valid_end));
            ctl->v_zero_to[st] =
                max(0, min(pf::kKeys, I.nblk_tile * kBlockSize - j * pf::kKeys));
            ctl->v_bad[st] = badm;
            if (bytes) mbar_arrive_expect_tx(&ctl->v_full[st], bytes);
            else mbar_arrive(&ctl->v_full[st]);
          }
          __syncwarp();
          if (phys >= 0) tile_copy(kL.v + st * kL.stage_stride, &vmap, ycoord, &ctl->v_full[st]);
          ++viss;
        }
      }
      // warp 0 claims the next item into the other slot, once the other warps have read the
      // item that was last there
      if (k_side && ok) {
        const uint32_t next = ic + 1;
        if (next >= 2 && !wait(&ctl->item_empty[next & 1u], ((next >> 1) - 1) & 1u)) break;
        if (lane == 0) {
          ctl->item[next & 1u] = claim_item(p, total);
          mbar_arrive(&ctl->item_full[next & 1u]);
        }
        __syncwarp();
      }
      if (!ok) break;
    } else if (warp == 1) {
      // ------------------------------------------------------------- S issuer -----------
      // S of slice g into buffer g % 3 once the P V of slice g - 3 has read its P there.
      const uint32_t id_s = kFp8 ? idesc_e4m3_f32(128, 128, false) : idesc_bf16_f32(128, 128, false);
      const uint32_t q_addr = smem_u32(smem + pf::kQ);
      // E4M3 pools: the softmax warps turn the bf16 q tile into three E4M3 parts first
      bool ok = wait(kFp8 ? &ctl->q_ready : &ctl->q_full, ic & 1u);
      for (int jj = 0; ok && jj < I.nj; ++jj) {
        const uint32_t g = tc + jj, st = g % pf::kStages, b = g % pf::kPBufs;
        if (g >= pf::kPBufs &&
            !(ok = wait(&ctl->o_done[b], ((g - pf::kPBufs) / pf::kPBufs) & 1u)))
          break;
        if (!(ok = wait(&ctl->k_full[st], (g / pf::kStages) & 1u))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_addr = smem_u32(smem + kL.k + st * kL.stage_stride);
          if constexpr (kFp8) {
            // S = (q_hi + q_mid + q_lo) K^T, 32 dims a step: q parts 16 KiB apart, K and q rows
            // of 128 bytes (8-row groups 1 KiB apart)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
#pragma unroll
              for (int part = 0; part < 3; ++part)
                tc_mma_f8(tmem + b * 128u,
                          smem_desc_sw128(q_addr + part * pf::kHalf + ks * 32, 16, 1024),
                          smem_desc_sw128(k_addr + ks * 32, 16, 1024), id_s, ks > 0 || part > 0);
          } else {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            // 64-column halves of q 16 KiB apart; of a K block 1 KiB apart (head_dim 128: 8-key
            // groups 2 KiB apart), or one half (64: 8-key groups 1 KiB apart)
            const uint32_t qa = q_addr + (ks >> 2) * pf::kHalf + (ks & 3) * 32;
            const uint32_t kb = k_addr + (ks >> 2) * 1024 + (ks & 3) * 32;
            tc_mma_bf16(tmem + b * 128u, smem_desc_sw128(qa, 16, 1024),
                        smem_desc_sw128(kb, 16, D == 128 ? 2048 : 1024), id_s, ks > 0);
          }
          }
          tc_commit(&ctl->s_full[b]);
          tc_commit(&ctl->k_empty[st]);
        }
        __syncwarp();
      }
      // the q tile is free for the next item once these S MMAs have run
      if (ok && lane == 0) tc_commit(&ctl->q_empty);
      __syncwarp();
    } else if (warp == pf::kPvWarp) {
      // ------------------------------------------------------------- P V issuer ---------
      // O += P V of slice jj once its V has landed (rows without a valid key cleared) and the
      // softmax has handed over its P.  A warp of its own, so that neither issuer's waits hold
      // back the other's MMAs.
      const uint32_t id_pv = kFp8 ? idesc_e4m3_f32(128, D, true) : idesc_bf16_f32(128, D, true);
      // O starts over once the softmax warps have read the last item's
      if (ic > 0) {
        if (!wait(&ctl->o_free, (ic - 1) & 1u)) break;
        tc_fence_after();
      }
      for (int jj = 0; jj < I.nj; ++jj) {
        const uint32_t g = tc + jj, st = g % pf::kStages, b = g % pf::kPBufs;
        if (!wait(&ctl->v_full[st], (g / pf::kStages) & 1u)) break;
        uint8_t* vt = smem + kL.v + st * kL.stage_stride;
        const int zf = ctl->v_zero_from[st], zt = ctl->v_zero_to[st];
        const uint32_t badm = ctl->v_bad[st];
        if (zf < zt || badm) {
          // clear the 128-byte rows (every column half) of keys that hold no valid value: the
          // pool slots past the sequence's end in its last loaded block, and the blocks with
          // a bad id.  (Blocks past the tile's last position are not loaded; their rows keep
          // older V data, finite since the ring starts zeroed and every stale slot that lands
          // is cleared here, and P is 0 there.)  Key kk of the slice: block kk / 16, row group
          // (kk / 8) % 2, row kk % 8.
          constexpr int kHalves = kBlk / 2048;  // 128-byte column halves of a key's row
          auto clear_key = [&](int key, int e) {
            const int half = (e >> 3) % kHalves, c16 = e & 7;
            *reinterpret_cast<uint4*>(vt + (key >> 3) * (kHalves * 1024) + half * 1024 +
                                      (key & 7) * 128 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
          };
          for (int e = lane; e < (zt - zf) * kHalves * 8; e += 32) clear_key(zf + e / (kHalves * 8), e);
          if (badm)
            for (int e = lane; e < pf::kKeys * kHalves * 8; e += 32) {
              const int key = e / (kHalves * 8);
              if ((badm >> (key >> 4)) & 1u) clear_key(key, e);
            }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (!wait(&ctl->p_full[b], (g / pf::kPBufs) & 1u)) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t v_addr = smem_u32(vt);
          // P of keys 16 ks .. 16 ks + 15: the hi parts of keys 0-63 in columns 0-31 of the
          // buffer and their lo parts in 32-63; keys 64-127 the same in columns 64-127.  V of
          // those keys: block ks of the stage, MN-major (head_dim 128: the column halves 1 KiB
          // apart, 8-key groups 2 KiB apart; 64: one half, 8-key groups 1 KiB apart).
          auto p_col = [&](int ks) { return tmem + b * 128u + (ks >> 2) * 64u + (ks & 3) * 8u; };
          const uint32_t o_acc = tmem + pf::kOCol;
          if constexpr (kFp8) {
            // P as E4M3 hi and lo parts, 4 keys a column: keys 32 ks .. 32 ks + 31 in columns
            // 64 (ks / 2) + 8 (ks % 2) .. + 7 (hi) and 16 further (lo), inside the columns of
            // their half's S; V of those keys: blocks 2 ks and 2 ks + 1 of the stage, MN-major
            // rows of 128 bytes (8-key groups 1 KiB apart)
            const uint32_t pb = tmem + b * 128u;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t vd = smem_desc_sw128(v_addr + ks * 2 * kBlk, 1024, 1024);
              const uint32_t pc = pb + (ks >> 1) * 64u + (ks & 1) * 8u;
              tc_mma_f8_ts(o_acc, pc, vd, id_pv, jj > 0 || ks > 0);
              tc_mma_f8_ts(o_acc, pc + 16u, vd, id_pv, true);
            }
          } else {
          auto v_desc = [&](int ks) {
            return smem_desc_sw128(v_addr + ks * kBlk, 1024, D == 128 ? 2048 : 1024);
          };
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(o_acc, p_col(ks), v_desc(ks), id_pv, jj > 0 || ks > 0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(o_acc, p_col(ks) + 32u, v_desc(ks), id_pv, true);
          }
          tc_commit(&ctl->o_done[b]);
          tc_commit(&ctl->v_empty[st]);
        }
        __syncwarp();
      }
    } else {
      // ------------------------------------------------------------- softmax rows -------
      constexpr int kC = 64;  // keys (and O columns) of a thread
      const int half = warp > pf::kPvWarp ? 1 : 0;
      const int quarter = warp & 3;        // TMEM lane quarter this warp may access
      const int r = quarter * 32 + lane;   // tile row = TMEM lane
      const int tok = r / G;
      const bool row_ok = tok < I.ntok;
      const int row_pos = I.pos0 + tok;
      const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      const uint32_t hc = half * 64u;      // first S / P column of this thread
      const uint32_t oc = half * kOC;      // and its first O column
      uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + kL.xbar) + quarter;
      // Combine v with the other half of the row (max, or sum): both threads fold v into the
      // row's slot, the two warps meet at the pair's barrier (lane 0 of each arrives once the
      // warp's updates are ordered before it) and read the slot; then the slot that the
      // exchange after next uses is cleared (its last readers have passed this barrier).
      auto exchange = [&](float v, bool sum, float* out) -> bool {
        int* slot = xslot + (xc % pf::kXBufs) * pf::kRows + r;
        if (sum) atomicAdd(reinterpret_cast<float*>(slot), v);  // -0.0f + a + b, either order
        else atomicMax(slot, float_order_key(v));
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar);
        if (!wait(xbar, xc & 1u)) return false;
        const int k = *reinterpret_cast<volatile int*>(slot);
        *out = sum ? __int_as_float(k) : order_key_float(k);
        xslot[((xc + 2) % pf::kXBufs) * pf::kRows + r] = INT_MIN;
        ++xc;
        return true;
      };
      // a quarter with no row of the run writes P = 0 and skips the exchanges (both warps of
      // a pair see the same rows)
      const bool live = __any_sync(0xffffffffu, row_ok);
      float m_used = 0.f, l = 0.f;
      bool seen = false;  // whether m_used comes from a visible key yet
      bool ok = true;
      // Scores of this row are multiplied by sl_row: scale * log2 e (* k_scale for E4M3),
      // and for E4M3 by the row's q scale as well.
      float sl_row = p.score_log2;
      if constexpr (kFp8) {
        // The bf16 q tile (two 64-column halves, each row 128 swizzled bytes) becomes three
        // E4M3 parts of the same layout (one 128-byte row each, parts 16 KiB apart): q is
        // scaled per row by 2^e, with the row's max magnitude in [128, 256); hi = e4m3(q 2^e),
        // mid = e4m3 of the rest, lo = e4m3 of what is left, so q 2^e = hi + mid + lo to about
        // 2^-12 of the row max.  This thread converts its half of the row; the two threads of a
        // row agree on its max first, which also orders their reads of the bf16 halves before
        // either writes over them.
        if (!(ok = wait(&ctl->q_full, ic & 1u))) break;
        const uint32_t qrow = smem_u32(smem + pf::kQ) + r * 128;
        const int sw = r & 7;
        float qv[64];
        float qmax = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w0, w1, w2, w3;
          ld_shared_v4(qrow + half * pf::kHalf + ((c ^ sw) << 4), w0, w1, w2, w3);
          const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            qv[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
            qv[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            qmax = fmax3(qmax, fabsf(qv[8 * c + 2 * i]), fabsf(qv[8 * c + 2 * i + 1]));
          }
        }
        float rmax;
        if (!(ok = exchange(qmax, false, &rmax))) break;
        // 2^e with rmax 2^e in [128, 256); 1 for a row of zeros (or of non-finite values)
        int e = 0;
        if (rmax > 0.f && rmax <= 3.0e38f) e = 7 - (((__float_as_uint(rmax) >> 23) & 0xff) - 127);
        e = max(-100, min(100, e));
        const float sc = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
        sl_row = p.score_log2 * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 16-dim chunks 4 half + c of the three part rows
          uint32_t hw[4], mw[4], lw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t hh = 0, mm = 0, ll = 0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float a0 = qv[16 * c + 4 * i + 2 * j] * sc;
              const float a1 = qv[16 * c + 4 * i + 2 * j + 1] * sc;
              const uint16_t h2 = f32x2_to_e4m3x2(a0, a1);
              float h0, h1;
              e4m3x2_to_f32x2(h2, h0, h1);
              const float r0 = a0 - h0, r1 = a1 - h1;
              const uint16_t m2 = f32x2_to_e4m3x2(r0, r1);
              float m0, m1;
              e4m3x2_to_f32x2(m2, m0, m1);
              const uint16_t l2 = f32x2_to_e4m3x2(r0 - m0, r1 - m1);
              hh |= static_cast<uint32_t>(h2) << (16 * j);
              mm |= static_cast<uint32_t>(m2) << (16 * j);
              ll |= static_cast<uint32_t>(l2) << (16 * j);
            }
            hw[i] = hh;
            mw[i] = mm;
            lw[i] = ll;
          }
          const uint32_t off = (((4 * half + c) ^ sw) << 4);
          st_shared_v4(qrow + off, hw[0], hw[1], hw[2], hw[3]);
          st_shared_v4(qrow + pf::kHalf + off, mw[0], mw[1], mw[2], mw[3]);
          st_shared_v4(qrow + 2 * pf::kHalf + off, lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async_smem();  // before the S MMAs read the parts
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->q_ready);
      }
      // This thread's columns of S are read into registers and its P is written over them; a
      // quarter with no row of the run reads nothing and leaves its rows of P alone (their O
      // rows are never read).
      for (int jj = 0; ok && jj < I.nj; ++jj) {
        const uint32_t g = tc + jj, b = g % pf::kPBufs;
        if (!(ok = wait(&ctl->s_full[b], (g / pf::kPBufs) & 1u))) break;
        tc_fence_after();
        if (!live) {
          mbar_arrive(&ctl->p_full[b]);
          continue;
        }
        const uint32_t s_cols = tl + b * 128u + hc;
        uint32_t sv[kC];
        tmem_ld_row<kC>(s_cols, sv);
        // keys 0..kmax of this thread's columns are visible
        const int kmax = row_ok ? row_pos - (I.j0 + jj) * pf::kKeys - half * 64 : -1;
        // raw scores, masked keys -inf; the row max is taken on them (the scale is positive)
        // and moved to the log2 domain once.  Eight independent max / sum accumulators keep
        // the dependency chains short.
        float x[kC];
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -CUDART_INF_F;
        if (__all_sync(0xffffffffu, kmax >= kC - 1)) {  // warp-uniform branch
#pragma unroll
          for (int i = 0; i < kC; ++i) x[i] = __uint_as_float(sv[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kC; ++i) x[i] = (i <= kmax) ? __uint_as_float(sv[i]) : -CUDART_INF_F;
        }
#pragma unroll
        for (int i = 0; i < kC; i += 2) mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], x[i], x[i + 1]);
        float mt;
        if (!(ok = exchange(fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))),
                            false, &mt)))
          break;
        if (mt != -CUDART_INF_F) mt *= sl_row;
        bool rescale = false;
        float m_new = m_used;
        if (!seen) {
          // O and l of the row are still zero: the first visible key sets the base
          if (mt != -CUDART_INF_F) {
            m_new = mt;
            seen = true;
          }
        } else if (mt > m_used + (kFp8 ? pf::kRescaleLog2Fp8 : pf::kRescaleLog2)) {
          m_new = mt;
          rescale = true;
        }
        const float alpha = rescale ? fast_exp2(m_used - m_new) : 1.f;
        // probabilities 2^(s * scale * log2 e - m); for the thread's 64 keys, bf16 hi parts
        // into its columns 0..31 and lo parts into 32..63.  The split is by truncation, on the integer
        // pipes: hi keeps the upper 16 bits of p, lo = p - hi exactly in fp32, and lo is
        // truncated in turn, so hi + lo = p within 2^-14 relative.
        // The pairs of keys go through Blackwell's two-wide fp32 instructions (the scale-and-shift,
        // the row sums, the lo parts), each lane rounded as the scalar one would be.
        const uint32_t p_cols = s_cols;
        // E4M3: P is made 2^8 times larger (kept under 448 by the rescale threshold), so that
        // its small values stay clear of E4M3's subnormal floor; l carries the same factor.
        constexpr float kPShift = kFp8 ? 8.f : 0.f;
        const f32x2 sl2 = f2_pack(sl_row, sl_row),
                    mn2 = f2_pack(kPShift - m_new, kPShift - m_new);
        f32x2 rsum[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rsum[i] = f2_pack(0.f, 0.f);
        if constexpr (kFp8) {
          // hi = e4m3(p), lo = e4m3(p - hi): for the thread's 64 keys, 16 columns of hi (four
          // keys a column) at its columns 0..15, and of lo at 16..31
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            uint32_t hh = 0, ll = 0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int k0 = 4 * q4 + 2 * j;
              float a0, a1;
              f2_unpack(f2_fma(f2_pack(x[k0], x[k0 + 1]), sl2, mn2), a0, a1);
              const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
              rsum[(2 * q4 + j) & 3] = f2_add(rsum[(2 * q4 + j) & 3], f2_pack(p0, p1));
              const uint16_t h2 = f32x2_to_e4m3x2(p0, p1);
              float h0, h1;
              e4m3x2_to_f32x2(h2, h0, h1);
              const uint16_t l2 = f32x2_to_e4m3x2(p0 - h0, p1 - h1);
              hh |= static_cast<uint32_t>(h2) << (16 * j);
              ll |= static_cast<uint32_t>(l2) << (16 * j);
            }
            hi[q4] = hh;
            lo[q4] = ll;
          }
          tmem_st16(p_cols, hi);
          tmem_st16(p_cols + 16, lo);
        } else {
#pragma unroll
        for (int c = 0; c < kC / 32; ++c) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(x[c * 32 + 2 * e], x[c * 32 + 2 * e + 1]), sl2, mn2), a0, a1);
            const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
            const f32x2 pp = f2_pack(p0, p1);
            rsum[e & 3] = f2_add(rsum[e & 3], pp);
            const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
            hi[e] = prmt(b0, b1, 0x7632u);
            float l0, l1;
            f2_unpack(f2_sub(pp, f2_pack(__uint_as_float(b0 & 0xffff0000u),
                                         __uint_as_float(b1 & 0xffff0000u))),
                      l0, l1);
            lo[e] = prmt(__float_as_uint(l0), __float_as_uint(l1), 0x7632u);
          }
          const uint32_t pc = p_cols + (c >> 1) * 64 + (c & 1) * 16;
          tmem_st16(pc, hi);
          tmem_st16(pc + 32, lo);
        }
        }
        float rs0, rs1, rs2, rs3, rs4, rs5, rs6, rs7;
        f2_unpack(rsum[0], rs0, rs1);
        f2_unpack(rsum[1], rs2, rs3);
        f2_unpack(rsum[2], rs4, rs5);
        f2_unpack(rsum[3], rs6, rs7);
        const float rs = ((rs0 + rs1) + (rs2 + rs3)) + ((rs4 + rs5) + (rs6 + rs7));
        l = l * alpha + rs;
        if (__any_sync(0xffffffffu, rescale)) {
          // this thread's columns of O move to the new base once the previous P V has landed
          // in it (a rescale needs a visible key in an earlier slice of the item, so jj > 0)
          if (!(ok = wait(&ctl->o_done[(g - 1) % pf::kPBufs], ((g - 1) / pf::kPBufs) & 1u)))
            break;
          tc_fence_after();
          uint32_t o[kOC];
#pragma unroll
          for (int c = 0; c < kOC / 32; ++c)
            tmem_ld32(tl + pf::kOCol + oc + c * 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kOC; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
#pragma unroll
          for (int c = 0; c < kOC / 32; ++c)
            tmem_st32(tl + pf::kOCol + oc + c * 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
        }
        tmem_wait_st();
        m_used = m_new;
        tc_fence_before();
        mbar_arrive(&ctl->p_full[b]);
      }
      // Epilogue: the thread's columns of O divided by the row sum (of both halves), to the
      // output, or (a split tile) to the item's partial with its log-sum-exp in the log2
      // domain, which the merge kernel combines after the split-KV kernel.
      if (ok && live) {
        float lt;
        ok = exchange(l, true, &lt);
        l = lt;
      }
      // Each warp stages its 32 rows in the (now idle) K stages, swizzled by row so that
      // neither the row-wise writes nor the chunk-wise reads conflict on banks, and then
      // writes them back a whole row (or two, four) per instruction, coalesced.
      const bool split = I.ns > 1;
      const uint32_t g_last = tc + I.nj - 1;
      const int sw = half ? warp - 4 : warp - 2;  // softmax warp index 0..7
      uint8_t* stage = smem + kL.stage + sw * (32 * kOC * 4);
      const bool have =
          ok && live && wait(&ctl->o_done[g_last % pf::kPBufs], (g_last / pf::kPBufs) & 1u);
      // O may take the next item's P V once every softmax warp has read it.  A warp with no
      // row of this item gets here without waiting on any reader of the item before, so it
      // first waits for that item's phase to complete: its arrival must not count there.
      auto release_o = [&] {
        if (ic > 0 && !wait(&ctl->o_free, (ic - 1) & 1u)) return;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->o_free);
      };
      if (!have) {  // warp-uniform
        release_o();
      } else {
        tc_fence_after();
        uint32_t o[kOC];
#pragma unroll
        for (int c = 0; c < kOC / 32; ++c)
          tmem_ld32(tl + pf::kOCol + oc + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
        tmem_wait_ld();
        release_o();
        // E4M3: O and l both carry P's factor 2^8, and V its scale
        const float inv = (row_ok && l > 0.f) ? (kFp8 ? p.v_out_scale : 1.f) / l : 0.f;
        const bool bf16 = p.out_bf16 && !split;   // partials are fp32
        if (split && half == 0 && row_ok)
          p.part_lse[(static_cast<int64_t>(I.t0 + tok) * p.num_q_heads + I.h * G + r % G) *
                         p.pmax + I.k] =
              (seen && l > 0.f) ? m_used + __log2f(l) - (kFp8 ? 8.f : 0.f) : -CUDART_INF_F;
        if (!bf16) {
          constexpr int CH = kOC / 4;   // 16-byte chunks of the thread's row part
#pragma unroll
          for (int c = 0; c < CH; ++c)
            *reinterpret_cast<uint4*>(stage + lane * CH * 16 + ((c ^ lane) & (CH - 1)) * 16) =
                make_uint4(__float_as_uint(__uint_as_float(o[4 * c]) * inv),
                           __float_as_uint(__uint_as_float(o[4 * c + 1]) * inv),
                           __float_as_uint(__uint_as_float(o[4 * c + 2]) * inv),
                           __float_as_uint(__uint_as_float(o[4 * c + 3]) * inv));
        } else {
          constexpr int CH = kOC / 8;
#pragma unroll
          for (int c = 0; c < CH; ++c)
            *reinterpret_cast<uint4*>(stage + lane * CH * 16 + ((c ^ lane) & (CH - 1)) * 16) =
                make_uint4(pack_bf16x2(__uint_as_float(o[8 * c]) * inv,
                                       __uint_as_float(o[8 * c + 1]) * inv),
                           pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv,
                                       __uint_as_float(o[8 * c + 3]) * inv),
                           pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv,
                                       __uint_as_float(o[8 * c + 5]) * inv),
                           pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv,
                                       __uint_as_float(o[8 * c + 7]) * inv));
        }
        __syncwarp();
        // this lane's row: its destination (NULL past the run), handed to the other lanes by
        // shuffles in the write loop
        const int64_t orow = static_cast<int64_t>(I.t0 + tok) * p.num_q_heads + I.h * G + r % G;
        uint8_t* my_dst =
            !row_ok ? nullptr
            : split ? reinterpret_cast<uint8_t*>(p.part_o + (orow * p.pmax + I.k) * D + oc)
            : bf16  ? reinterpret_cast<uint8_t*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                 orow * D + oc)
                    : reinterpret_cast<uint8_t*>(reinterpret_cast<float*>(p.out) + orow * D + oc);
        const uint32_t stage_s = smem_u32(stage);
        auto write_rows = [&](auto ch_tag) {
          constexpr int CH = decltype(ch_tag)::value;
          constexpr int RPI = 32 / CH;  // rows per instruction
#pragma unroll 8
          for (int it = 0; it < CH; ++it) {
            const int rr = it * RPI + lane / CH, c = lane % CH;
            uint4 v;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(stage_s + rr * CH * 16 + ((c ^ rr) & (CH - 1)) * 16));
            uint8_t* dst = reinterpret_cast<uint8_t*>(__shfl_sync(
                0xffffffffu, reinterpret_cast<unsigned long long>(my_dst), rr));
            if (dst) *reinterpret_cast<uint4*>(dst + c * 16) = v;
          }
        };
        if (!bf16) write_rows(std::integral_constant<int, kOC / 4>());
        else write_rows(std::integral_constant<int, kOC / 8>());
      }
    }
    tc += I.nj;
    ++ic;
    if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) break;
  }
  // Exit, normal or after an expired wait: no copy may still be landing in shared memory and
  // no MMA may still be using tensor memory when the CTA ends.
  if (warp == 0 || warp == pf::kVWarp) {
    // the latest fill of each stage is the only one that can still be in flight
    const uint32_t iss = warp == 0 ? kiss : viss;
    uint64_t* full = warp == 0 ? ctl->k_full : ctl->v_full;
    for (uint32_t g = iss > pf::kStages ? iss - pf::kStages : 0; g < iss; ++g)
      mbar_wait(&full[g % pf::kStages], (g / pf::kStages) & 1u, p.wait_ns);
    if (warp == 0 && qiss) mbar_wait(&ctl->q_full, (qiss - 1) & 1u, p.wait_ns);
  } else if (warp == 1 || warp == pf::kPvWarp) {
    // each issuer's own MMAs (a commit tracks those of the issuing thread)
    uint64_t* drain = &ctl->drain[warp == 1 ? 0 : 1];
    if (lane == 0) tc_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, p.wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, pf::kTmemCols);
  if (p.span && threadIdx.x == 0)
    atomicMax(reinterpret_cast<unsigned long long*>(p.span) + 1,
              static_cast<unsigned long long>(global_ns()));
}

namespace {

template <int D, bool kFp8>
cudaError_t launch_prefill_grid(const AttnArgs& a, const PrefillParams& p, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const CUtensorMap& vmap) {
  constexpr pf::Layout kL(kFp8);
  LaunchInfo li;
  cudaError_t e = launch_info(prefill_kernel<D, kFp8>, pf::kThreads, kL.smem, &li);
  if (e != cudaSuccess) return e;
  // at most one CTA per SM (shared memory); the plan decides how many of them work
  const int64_t upper =
      static_cast<int64_t>(a.num_kv_heads) * kMaxSplits *
      ((static_cast<int64_t>(a.num_q_tokens) * p.group + pf::kRows - 1) / pf::kRows +
       a.num_seqs);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(upper, li.sms));
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_before, a.stream);
  e = launch_dependent(prefill_kernel<D, kFp8>, dim3(static_cast<unsigned>(grid)),
                       dim3(pf::kThreads), kL.smem, a.stream, qmap, kmap, vmap, p);
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_after, a.stream);
  return e;
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a, const int32_t* item_start, const int32_t* order,
                           WsHeader* hdr,
                           const PoolMaps& maps, const PrefillScratch& scratch) {
  PrefillParams p{};
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.qsl = a.query_start_loc;
  p.item_start = item_start;
  p.order = order;
  p.out = a.out;
  p.hdr = hdr;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.cache.num_blocks;
  p.out_bf16 = a.out_dtype == PA_BF16;
  const bool fp8 = a.cache.cache_dtype == PA_FP8_E4M3;
  // E4M3 pools: K's scale folds into the scores, V's into the output
  p.score_log2 = a.scale * 1.4426950408889634f * (fp8 ? a.cache.k_scale : 1.f);
  p.v_out_scale = fp8 ? a.cache.v_scale : 1.f;
  p.wait_ns = a.wait_ns;
  p.skip_copy = a.skip_copy;
  p.span = a.span ? a.span + 2 : nullptr;
  p.part_lse = scratch.part_lse;
  p.part_o = scratch.part_o;
  p.pmax = scratch.pmax;
  // bf16 head_dim 128: whole-tile 4-D copies; 64 and E4M3: the 2-D pool view, whose 16-row box
  // is the tile
  if (fp8) return launch_prefill_grid<128, true>(a, p, maps.q3, maps.k2, maps.v2);
  if (a.head_dim == 64) return launch_prefill_grid<64, false>(a, p, maps.q3, maps.k2, maps.v2);
  return launch_prefill_grid<128, false>(a, p, maps.q3, maps.k4, maps.v4);
}

}  // namespace pa
