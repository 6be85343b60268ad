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
// Design (GB300 / sm_103a; bf16 K/V, head_dim 128):
//  * One work item = (sequence, kv head, tile of 128 rows), a row being (query token, q head of
//    the GQA group), so the tile's queries share every K/V tile they read.  Items are taken
//    longest-first from an atomic counter by persistent CTAs (one per SM).
//  * Warp 0 issues TMA copies of the q tile once (a 3-D box of tokens x heads x 64 columns, two
//    boxes), then for every 128 keys the 8 (block, kv head) K tiles of the block table; warp 6
//    does the same for the V tiles.  Eight lanes of each issue one block's boxes apiece, into
//    three-stage K and V rings (128-byte swizzle, completion on mbarriers).
//  * Warp 1 issues tcgen05.mma from one thread: S = Q K^T into one of three TMEM buffers
//    (128 x 128 fp32), and O += P V into a fourth, with P read from TMEM and V from shared
//    memory (MN-major).  The softmax threads write P back over their S columns as bf16 hi and
//    lo parts (keys 0-63: hi in columns 0-31, lo in 32-63; keys 64-127 likewise in 64-127), so
//    P V is exact to ~2^-16 like the decode path, and the next tile's softmax can run while
//    this tile's P V is in flight.
//  * Softmax, one thread per row (TMEM lane): it reads its row of S from TMEM once, masks keys
//    beyond the row's position, keeps the running max in the log2 domain and rescales O in
//    TMEM only when the max grows by more than 2^8 (the final division uses the same max, so
//    the result is exact), and finally divides O by the row sum and stores it.  Warps 2-5 do
//    this for whole rows.  When every run has at most 64 rows (speculative verify), at most
//    two of the four lane quarters hold rows, and the kernel instance with the row split runs
//    instead: warps 2-5 take keys (and O columns) 0-63 and warps 7-10 keys 64-127, the two
//    threads of a row agreeing on its max, and at the end adding their sums, through a
//    shared-memory slot and an mbarrier of the pair.  A warp can only reach the lane quarter
//    of its own SM sub-partition, so the split puts a second warp on each busy sub-partition
//    to hide the latency of the exponentials and TMEM traffic.
//  * V rows past the last valid key (stale slots, possibly NaN) are zeroed in shared memory
//    before P V reads them; K there only feeds masked scores.
#include <math_constants.h>

#include <algorithm>
#include <climits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace pf {
constexpr int kRows = 128;
constexpr int kKeys = 128;
constexpr int kStages = 3;   // K and V ring depth
constexpr int kSBufs = 3;    // S/P buffers in TMEM (3 x 128 columns) ahead of O
constexpr int kHalf = 16384;  // one 64-column region of a 128-row bf16 tile
constexpr int kTile = 32768;  // 128 x 128 bf16
constexpr int kQ = 0, kK = kTile, kV = kK + kStages * kTile;
constexpr int kCtl = kV + kStages * kTile;  // control block (barriers, item, flags)
constexpr int kXBar = kCtl + 256;           // 4 mbarriers: one per pair of softmax warps
constexpr int kXSlot = kXBar + 32;          // 3 x 128 row slots of the pairs' exchanges
constexpr int kXBufs = 3;
constexpr int kVWarp = 6;     // V producer (warp 0 loads q and K)
// Without the row split: warps 2-5 are the softmax, a thread a whole row.  With it: warps 2-5
// take keys 0-63 of their rows and warps 7-10 keys 64-127, and the pairs exchange row sums
// and maxima through shared memory.
__host__ __device__ constexpr int threads(bool split) { return split ? 352 : 224; }
__host__ __device__ constexpr int softmax_threads(bool split) { return split ? 256 : 128; }
__host__ __device__ constexpr int smem_bytes(bool split) {
  return 1024 + (split ? kXSlot + kXBufs * kRows * 4 : kCtl + 256);
}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = kSBufs * 128;
constexpr float kRescaleLog2 = 8.f;
}  // namespace pf


struct PfItem {
  int s, h, t0, ntok, pos0, L, nkv, nblk_tile, valid, first;
};

struct PfCtl {
  uint64_t q_full, k_full[pf::kStages], k_empty[pf::kStages], v_full[pf::kStages],
      v_empty[pf::kStages], s_full[pf::kSBufs], p_full[pf::kSBufs], o_done[pf::kSBufs];
  uint32_t tmem_base;
  int abort_flag;
  int v_zero_from[pf::kStages];
  uint32_t v_bad[pf::kStages];
  PfItem item;
};
static_assert(sizeof(PfCtl) <= 256, "control block too large");
static_assert(pf::smem_bytes(true) <= 232448, "more shared memory than a CTA may have");

// Floats mapped to ints of the same order (an involution), so that integer atomicMax takes the
// max of floats.  The empty slot INT_MIN is below every mapped float and reads as -0.0f.
__device__ __forceinline__ int float_order_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float order_key_float(int k) {
  return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff));
}

template <bool kSplit>
__global__ void __launch_bounds__(pf::threads(kSplit), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PfCtl* ctl = reinterpret_cast<PfCtl*>(smem + pf::kCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int i = 0; i < pf::kStages; ++i) {
      mbar_init(&ctl->k_full[i], 1);
      mbar_init(&ctl->k_empty[i], 1);
      mbar_init(&ctl->v_full[i], 1);
      mbar_init(&ctl->v_empty[i], 1);
    }
    // one of each per S/P buffer, so that every waiter is within one phase of its barrier:
    // S of tile g+3 is issued only after P V of tile g, which waits for P of tile g
    for (int i = 0; i < pf::kSBufs; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], pf::softmax_threads(kSplit));
      mbar_init(&ctl->o_done[i], 1);
    }
    if (kSplit)
      for (int q = 0; q < 4; ++q)
        mbar_init(reinterpret_cast<uint64_t*>(smem + pf::kXBar) + q, 2);  // one lane a warp
    ctl->abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  int* xslot = reinterpret_cast<int*>(smem + pf::kXSlot);  // [kXBufs][kRows], split only
  if (kSplit)
    for (int i = tid; i < pf::kXBufs * pf::kRows; i += pf::threads(true)) xslot[i] = INT_MIN;
  if (warp == 1) tmem_alloc(&ctl->tmem_base, pf::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int total = p.item_start[p.num_seqs];
  uint32_t tc = 0;  // KV tiles processed by this CTA so far (ring / phase tracking)
  uint32_t ic = 0;  // items processed by this CTA so far
  uint32_t xc = 0;  // exchanges of this softmax thread's pair so far (slot / phase tracking)
  const int G = p.group;
  const int tpt = pf::kRows / G;  // query tokens per tile

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
    if (tid == 0) {
      PfItem it;
      const int rev = static_cast<int>(atomicAdd(&p.hdr->prefill_counter, 1u));
      const int item = total - 1 - rev;  // longest items (last tiles of a chunk) first
      it.valid = item >= 0;
      it.first = rev == 0;
      if (it.valid) {
        int lo = 0, hi = p.num_seqs;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (p.item_start[mid] <= item) lo = mid; else hi = mid;
        }
        const int s = lo;
        const int t0 = p.qsl[s];
        const int n = p.qsl[s + 1] - t0;
        const int L = p.context_lens[s];
        const int qtiles = (n + tpt - 1) / tpt;
        const int local = item - p.item_start[s];
        const int h = local / qtiles;
        const int qt = local - h * qtiles;
        const int i0 = qt * tpt;
        it.s = s;
        it.h = h;
        it.t0 = t0 + i0;
        it.ntok = min(tpt, n - i0);
        it.pos0 = L - n + i0;
        it.L = L;
        const int pmax = it.pos0 + it.ntok - 1;
        it.nkv = pmax / pf::kKeys + 1;
        it.nblk_tile = pmax / kBlockSize + 1;
      }
      ctl->item = it;
    }
    __syncthreads();
    const PfItem I = ctl->item;
    if (!I.valid || ctl->abort_flag) break;

    if (warp == 0 || warp == pf::kVWarp) {
      // ------------------------------------------------------- producers (TMA): warp 0 q and K,
      // warp 6 V.  Two issuing warps double the rate at which tile copies enter the TMA unit.
      const bool k_side = warp == 0;
      if (k_side && lane == 0) {
        mbar_arrive_expect_tx(&ctl->q_full, pf::kTile);
        tma_load_3d(smem + pf::kQ, &qmap, 0, I.h * G, I.t0, &ctl->q_full);
        tma_load_3d(smem + pf::kQ + pf::kHalf, &qmap, 64, I.h * G, I.t0, &ctl->q_full);
      }
      // Block-table entries are read 32 at a time (lane l holds block 32 * grp + l) with the
      // next group prefetched, so no TMA issue waits on a dependent table load.
      const int32_t* trow = p.block_tables + static_cast<int64_t>(I.s) * p.max_blocks_per_seq;
      auto tab_load = [&](int grp) -> int {
        const int jb = 32 * grp + lane;
        return jb < I.nblk_tile ? __ldg(trow + jb) : -1;
      };
      int grp_cur = 0;
      int tab_cur = tab_load(0);
      int tab_next = tab_load(1);
      // block ids of slice j for lanes 0-7 (-1 = not loaded), plus masks of loadable / bad ones
      auto slice = [&](int j, int& phys, uint32_t& ok_mask, uint32_t& bad_mask) {
        const int grp = j >> 2;
        if (grp != grp_cur) {
          tab_cur = tab_next;
          tab_next = tab_load(grp + 1);
          grp_cur = grp;
        }
        const int e = __shfl_sync(0xffffffffu, tab_cur, 8 * (j & 3) + (lane & 7));
        const int jb = 8 * j + lane;
        phys = -1;
        bool bad = false;
        if (lane < 8 && jb < I.nblk_tile) {
          if (e < 0 || e >= p.num_blocks) {
            set_error(&p.hdr->error, PA_DEVERR_BLOCK_ID);
            bad = true;
          } else {
            phys = e;
          }
        }
        ok_mask = __ballot_sync(0xffffffffu, phys >= 0);
        bad_mask = __ballot_sync(0xffffffffu, bad);
      };
      auto load_k = [&](int j, int phys, uint32_t okm) -> bool {
        const uint32_t g = tc + j, st = g % pf::kStages;
        const uint32_t bytes = __popc(okm) * 2u * 2048u;
        if (!wait(&ctl->k_empty[st], ((g / pf::kStages) & 1u) ^ 1u)) return false;
        if (lane == 0) {
          if (bytes) mbar_arrive_expect_tx(&ctl->k_full[st], bytes);
          else mbar_arrive(&ctl->k_full[st]);
        }
        __syncwarp();
        // test hook: lane 0's copy of the first slice of the first item claimed is left out
        // (its bytes are still expected), so that the bounded waits on that stage expire
        const bool skip = p.skip_copy && I.first && j == 0 && lane == 0;
        if (phys >= 0 && !skip) {
          const int yrow = (phys * p.num_kv_heads + I.h) * kBlockSize;
          uint8_t* kt = smem + pf::kK + st * pf::kTile + lane * 2048;
          tma_load_2d(kt, &kmap, 0, yrow, &ctl->k_full[st]);
          tma_load_2d(kt + pf::kHalf, &kmap, 64, yrow, &ctl->k_full[st]);
        }
        return true;
      };
      auto load_v = [&](int j, int phys, uint32_t okm, uint32_t badm) -> bool {
        const uint32_t g = tc + j, st = g % pf::kStages;
        const uint32_t bytes = __popc(okm) * 2u * 2048u;
        if (!wait(&ctl->v_empty[st], ((g / pf::kStages) & 1u) ^ 1u)) return false;
        if (lane == 0) {
          // rows the MMA warp has to clear: keys past the last valid one, and bad blocks
          const int valid_end = min(I.L, I.nblk_tile * kBlockSize) - j * pf::kKeys;
          ctl->v_zero_from[st] = max(0, min(pf::kKeys, valid_end));
          ctl->v_bad[st] = badm;
          if (bytes) mbar_arrive_expect_tx(&ctl->v_full[st], bytes);
          else mbar_arrive(&ctl->v_full[st]);
        }
        __syncwarp();
        if (phys >= 0) {
          const int yrow = (phys * p.num_kv_heads + I.h) * kBlockSize;
          uint8_t* vt = smem + pf::kV + st * pf::kTile + lane * 2048;
          tma_load_2d(vt, &vmap, 0, yrow, &ctl->v_full[st]);
          tma_load_2d(vt + pf::kHalf, &vmap, 64, yrow, &ctl->v_full[st]);
        }
        return true;
      };
      for (int j = 0; j < I.nkv; ++j) {
        int ph;
        uint32_t okm, badm;
        slice(j, ph, okm, badm);
        if (!(k_side ? load_k(j, ph, okm) : load_v(j, ph, okm, badm))) break;
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------- MMA issuer ---------
      const uint32_t id_s = idesc_bf16_f32(128, 128, false);
      const uint32_t id_pv = idesc_bf16_f32(128, 128, true);
      const uint32_t q_addr = smem_u32(smem + pf::kQ);
      auto issue_s = [&](int j) -> bool {
        const uint32_t g = tc + j, st = g % pf::kStages, b = g % pf::kSBufs;
        if (!wait(&ctl->k_full[st], (g / pf::kStages) & 1u)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_addr = smem_u32(smem + pf::kK + st * pf::kTile);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * pf::kHalf + (ks & 3) * 32;
            tc_mma_bf16(tmem + b * 128u, smem_desc_sw128(q_addr + off, 16, 1024),
                        smem_desc_sw128(k_addr + off, 16, 1024), id_s, ks > 0);
          }
          tc_commit(&ctl->s_full[b]);
          tc_commit(&ctl->k_empty[st]);
        }
        __syncwarp();
        return true;
      };
      bool ok = wait(&ctl->q_full, ic & 1u);
      if (ok) tc_fence_after();
      for (int j = 0; ok && j < min(pf::kSBufs, I.nkv); ++j) ok = issue_s(j);
      for (int j = 0; ok && j < I.nkv; ++j) {
        const uint32_t g = tc + j, st = g % pf::kStages, b = g % pf::kSBufs;
        if (!(ok = wait(&ctl->v_full[st], (g / pf::kStages) & 1u))) break;
        uint8_t* vt = smem + pf::kV + st * pf::kTile;
        const int zf = ctl->v_zero_from[st];
        const uint32_t badm = ctl->v_bad[st];
        if (zf < pf::kKeys || badm) {
          // clear the 128-byte rows (both column halves) of keys that hold no valid value
          for (int e = lane; e < pf::kKeys * 2 * 8; e += 32) {
            const int key = e >> 4, half = (e >> 3) & 1, c16 = e & 7;
            if (key >= zf || ((badm >> (key >> 4)) & 1u))
              *reinterpret_cast<uint4*>(vt + half * pf::kHalf + key * 128 + c16 * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (!(ok = wait(&ctl->p_full[b], (g / pf::kSBufs) & 1u))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t v_addr = smem_u32(vt);
          // P of keys 16 ks .. 16 ks + 15: the hi parts of keys 0-63 in columns 0-31 of the
          // buffer and their lo parts in 32-63; keys 64-127 the same in columns 64-127
          auto p_col = [&](int ks) { return tmem + b * 128u + (ks >> 2) * 64u + (ks & 3) * 8u; };
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(tmem + pf::kOCol, p_col(ks),
                           smem_desc_sw128(v_addr + ks * 2048, pf::kHalf, 1024), id_pv,
                           j > 0 || ks > 0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(tmem + pf::kOCol, p_col(ks) + 32u,
                           smem_desc_sw128(v_addr + ks * 2048, pf::kHalf, 1024), id_pv, true);
          tc_commit(&ctl->o_done[b]);
          tc_commit(&ctl->v_empty[st]);
        }
        __syncwarp();
        // S of tile j+3 reuses this tile's S/P buffer: it is issued after (and runs after) the
        // P V that reads P from it
        if (j + pf::kSBufs < I.nkv) ok = issue_s(j + pf::kSBufs);
      }
    } else {
      // ------------------------------------------------------------- softmax rows -------
      constexpr int kC = kSplit ? 64 : 128;  // keys (and O columns) of a thread
      const int half = (kSplit && warp > pf::kVWarp) ? 1 : 0;
      const int quarter = warp & 3;        // TMEM lane quarter this warp may access
      const int r = quarter * 32 + lane;   // tile row = TMEM lane
      const int tok = r / G;
      const bool row_ok = tok < I.ntok;
      const int row_pos = I.pos0 + tok;
      const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      const uint32_t hc = half * 64u;      // first S / P / O column of this thread
      uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + pf::kXBar) + quarter;
      // Combine v with the other half of the row (max, or sum): both threads fold v into the
      // row's slot, the two warps meet at the pair's barrier (lane 0 of each arrives once the
      // warp's updates are ordered before it) and read the slot; then the slot that the
      // exchange after next uses is cleared (its last readers have passed this barrier).
      auto exchange = [&](float v, bool sum, float* out) -> bool {
        if (!kSplit) {
          *out = v;
          return true;
        }
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
      bool ok = true;
      for (int j = 0; j < I.nkv; ++j) {
        const uint32_t g = tc + j, b = g % pf::kSBufs;
        if (!(ok = wait(&ctl->s_full[b], (g / pf::kSBufs) & 1u))) break;
        tc_fence_after();
        const uint32_t sb = tl + b * 128u + hc;  // this thread's columns of S, then of P
        if (!live) {
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
          for (int c = 0; c < kC / 16; ++c) tmem_st16(sb + c * 16, z);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&ctl->p_full[b]);
          continue;
        }
        // keys 0..kmax of this thread's columns are visible
        const int kmax = row_ok ? row_pos - j * pf::kKeys - half * 64 : -1;
        uint32_t sv[kC];
#pragma unroll
        for (int c = 0; c < kC / 32; ++c)
          tmem_ld32(sb + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
        tmem_wait_ld();
        // scores in the log2 domain; masked keys become -inf.  Eight independent max / sum
        // accumulators keep the dependency chains short.
        float x[kC];
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -CUDART_INF_F;
        if (__all_sync(0xffffffffu, kmax >= kC - 1)) {  // warp-uniform branch
#pragma unroll
          for (int i = 0; i < kC; ++i) {
            x[i] = __uint_as_float(sv[i]) * p.score_log2;
            mx[i & 7] = fmaxf(mx[i & 7], x[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kC; ++i) {
            x[i] = (i <= kmax) ? __uint_as_float(sv[i]) * p.score_log2 : -CUDART_INF_F;
            mx[i & 7] = fmaxf(mx[i & 7], x[i]);
          }
        }
        float mt;
        if (!(ok = exchange(fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))),
                            false, &mt)))
          break;
        bool rescale = false;
        float m_new = m_used;
        if (j == 0) {
          m_new = (mt == -CUDART_INF_F) ? 0.f : mt;
        } else if (mt > m_used + pf::kRescaleLog2) {
          m_new = mt;
          rescale = true;
        }
        const float alpha = rescale ? fast_exp2(m_used - m_new) : 1.f;
        // probabilities; for every 64 keys, bf16 hi parts into their columns 0..31 and lo
        // parts into 32..63
        float rsum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rsum[i] = 0.f;
#pragma unroll
        for (int c = 0; c < kC / 32; ++c) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = fast_exp2(x[c * 32 + 2 * e] - m_new);
            const float p1 = fast_exp2(x[c * 32 + 2 * e + 1] - m_new);
            rsum[e & 7] += p0 + p1;
            hi[e] = pack_bf16x2(p0, p1);
            lo[e] = pack_bf16x2(p0 - bf16lo_to_f32(hi[e]), p1 - bf16hi_to_f32(hi[e]));
          }
          const uint32_t pc = sb + (c >> 1) * 64 + (c & 1) * 16;
          tmem_st16(pc, hi);
          tmem_st16(pc + 32, lo);
        }
        const float rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) +
                         ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
        l = l * alpha + rs;
        if (__any_sync(0xffffffffu, rescale)) {
          // O may be rescaled only once the previous P V has landed in it
          if (j > 0 &&
              !(ok = wait(&ctl->o_done[(g - 1) % pf::kSBufs], ((g - 1) / pf::kSBufs) & 1u)))
            break;
          tc_fence_after();
          uint32_t o[kC];
#pragma unroll
          for (int c = 0; c < kC / 32; ++c)
            tmem_ld32(tl + pf::kOCol + hc + c * 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kC; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
#pragma unroll
          for (int c = 0; c < kC / 32; ++c)
            tmem_st32(tl + pf::kOCol + hc + c * 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
        }
        tmem_wait_st();
        m_used = m_new;
        tc_fence_before();
        mbar_arrive(&ctl->p_full[b]);
      }
      // epilogue: the thread's columns of O divided by the row sum (of both halves)
      if (ok && live) {
        float lt;
        ok = exchange(l, true, &lt);
        l = lt;
      }
      const uint32_t g_last = tc + I.nkv - 1;
      if (ok && live && wait(&ctl->o_done[g_last % pf::kSBufs], (g_last / pf::kSBufs) & 1u)) {
        tc_fence_after();
        const float inv = (row_ok && l > 0.f) ? 1.f / l : 0.f;
        const int64_t orow = static_cast<int64_t>(I.t0 + tok) * p.num_q_heads + I.h * G + r % G;
        uint32_t o[kC];
#pragma unroll
        for (int c = 0; c < kC / 32; ++c)
          tmem_ld32(tl + pf::kOCol + hc + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
        tmem_wait_ld();
        if (row_ok) {
          if (p.out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                  orow * 128 + hc);
#pragma unroll
            for (int i = 0; i < kC / 8; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(__uint_as_float(o[8 * i + 2 * e]) * inv,
                                   __uint_as_float(o[8 * i + 2 * e + 1]) * inv);
              dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst =
                reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * 128 + hc);
#pragma unroll
            for (int i = 0; i < kC / 4; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv,
                                   __uint_as_float(o[4 * i + 1]) * inv,
                                   __uint_as_float(o[4 * i + 2]) * inv,
                                   __uint_as_float(o[4 * i + 3]) * inv);
          }
        }
      }
      tc_fence_before();
    }
    tc += I.nkv;
    ++ic;
    __syncthreads();
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, pf::kTmemCols);
}

namespace {

template <bool kSplit>
cudaError_t launch_prefill_as(const AttnArgs& a, const PrefillParams& p, const CUtensorMap& qmap,
                              const CUtensorMap& kmap, const CUtensorMap& vmap) {
  constexpr int kThreads = pf::threads(kSplit), kSmem = pf::smem_bytes(kSplit);
  LaunchInfo li;
  cudaError_t e = launch_info(prefill_kernel<kSplit>, kThreads, kSmem, &li);
  if (e != cudaSuccess) return e;
  const int64_t upper =
      static_cast<int64_t>(a.num_kv_heads) *
      ((static_cast<int64_t>(a.num_q_tokens) * p.group + pf::kRows - 1) / pf::kRows +
       a.num_seqs);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(upper, li.sms));
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_before, a.stream);
  prefill_kernel<kSplit>
      <<<static_cast<unsigned>(grid), kThreads, kSmem, a.stream>>>(qmap, kmap, vmap, p);
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_after, a.stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a, const int32_t* item_start, WsHeader* hdr,
                           const PoolMaps& maps) {
  PrefillParams p{};
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.qsl = a.query_start_loc;
  p.item_start = item_start;
  p.out = a.out;
  p.hdr = hdr;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.cache.num_blocks;
  p.out_bf16 = a.out_dtype == PA_BF16;
  p.score_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = a.wait_ns;
  p.skip_copy = a.skip_copy;
  // Runs of at most 64 rows (tokens x group heads: speculative verify) leave at least two of
  // a tile's four lane quarters empty; splitting each row over two warps then puts a second
  // warp on the busy quarters' SM sub-partitions.  Fuller tiles gain nothing from the split.
  if (!prefill_uses_pairs(a.max_query_len, p.group))
    return launch_prefill_as<true>(a, p, maps.q3, maps.k2, maps.v2);
  return launch_chunk(a, p, maps.q3, maps.k4, maps.v4);
}

}  // namespace pa
