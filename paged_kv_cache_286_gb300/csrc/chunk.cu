// Causal chunked-prefill tiles on tcgen05 tensor cores, two query tiles per CTA.
//
// What it computes ("Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained",
// sections "Chunked Prefill", "Prefill Versus Decode", "Attention Over Scattered Blocks"): a
// prompt chunk of n tokens whose sequence holds L keys after this step's append sits at
// positions p_i = L - n + i; token i attends keys 0..p_i, fetched through the block table.
// Every query run with more than 64 (token x q head) rows of a step comes here.
//
// Design (GB300 / sm_103a; bf16 K/V, head_dim 128):
//  * A tile is 128 rows, a row being (query token, q head of the GQA group).  One work item is
//    a pair of consecutive tiles (A, B) of one (sequence, kv head): both read every K/V slice of
//    128 keys from the same shared-memory stage, which halves the tile copies per flop.  The
//    copy count, not the bytes, is what one SM's TMA unit is limited by.
//  * The pool is viewed by a 4-D tensor map as (64 columns, 8 rows, 2 column halves, 8-row
//    groups), so that one TMA copy brings a whole 16 x 128 (block, kv head) tile: 8 copies per
//    slice for K and 8 for V, issued by eight lanes of the producer warp (warp 0), into a
//    3-stage K ring and a 2-stage V ring.  In shared memory a block's tile is
//    [2 row groups][2 halves][8 rows][128 bytes] with the 128-byte swizzle, i.e. 8-key groups
//    2 KiB apart and the two column halves 1 KiB apart, which the MMA descriptors express as
//    strides.
//  * Warp 1 issues tcgen05.mma from one thread.  Tensor memory holds S/P of A and B (columns
//    0-127 and 128-255) and O of A and B (256-383, 384-511).  Per slice j the order is
//    PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while the softmax warps of A work on S_A(j+1), the
//    pipe runs PV_B(j) and S_B(j+1), and the other way round, so the exponentials of one tile
//    overlap the MMAs of the other.  Since the pipe runs one thread's MMAs in order, S_X(j+1)
//    overwrites P_X(j) only after PV_X(j) has read it, and the commit that signals S_X(j+1)
//    also covers PV_X(j) (so O_X may be rescaled once S_X(j+1) is seen).
//  * Softmax: warps 2-5 take the rows of tile A and warps 6-9 those of B, one thread per row
//    (TMEM lane).  A thread reads its row of S once, masks keys beyond the row's position,
//    keeps the running max in the log2 domain and rescales O only when the max grows by more
//    than 2^8 (the final division uses the same max), and writes P back over S as bf16 hi and
//    lo parts (for every 32 keys: hi in their first 16 columns, lo in the next 16), so P V is
//    exact to ~2^-16.  It reads S twice, 32 columns at a time (the row max, then the
//    probabilities), to keep few registers live; each 32-key chunk of P overwrites only the
//    chunk of S just read.  At the end it divides its row of O by the row sum and stores it.
//  * V rows past the last valid key (stale slots, possibly NaN) and of bad block ids are
//    zeroed in shared memory before P V reads them; K there only feeds masked scores.
//  * Every wait is bounded; on expiry the CTA records PA_DEVERR_TIMEOUT, stops, lets the copies
//    and MMAs it issued finish (bounded waits again) and frees its tensor memory.
#include <math_constants.h>

#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace ck {
constexpr int kRows = 128;               // rows of one tile
constexpr int kKeys = 128;               // keys of one slice
constexpr int kKStages = 3, kVStages = 2;
constexpr int kTile = 32768;             // 128 x 128 bf16
constexpr int kHalf = 16384;             // one 64-column half of a q tile
constexpr int kBlockBytes = 4096;        // one (block, kv head) tile in shared memory
constexpr int kQ = 0;                    // q of tile A; tile B follows at kTile
constexpr int kK = 2 * kTile;
constexpr int kV = kK + kKStages * kTile;
constexpr int kCtl = kV + kVStages * kTile;
constexpr int kThreads = 320;            // warp 0 TMA, warp 1 MMA, warps 2-9 softmax
constexpr int kSmem = 1024 + kCtl + 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;
constexpr float kRescaleLog2 = 8.f;
}  // namespace ck

static_assert(ck::kSmem <= 232448, "more shared memory than a CTA may have");

struct CkItem {
  int s, h, L, nkv, nblk, valid, has_b, first;
  int t0[2], ntok[2], pos0[2];
};

struct CkCtl {
  uint64_t q_full, k_full[ck::kKStages], k_empty[ck::kKStages], v_full[ck::kVStages],
      v_empty[ck::kVStages], s_full[2], p_full[2], o_done[2], drain;
  uint32_t tmem_base;
  int abort_flag;
  int v_zero_from[ck::kVStages];
  uint32_t v_bad[ck::kVStages];
  CkItem item;
};
static_assert(sizeof(CkCtl) <= 512, "control block too large");

__global__ void __launch_bounds__(ck::kThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  CkCtl* ctl = reinterpret_cast<CkCtl*>(smem + ck::kCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int i = 0; i < ck::kKStages; ++i) {
      mbar_init(&ctl->k_full[i], 1);
      mbar_init(&ctl->k_empty[i], 1);
    }
    for (int i = 0; i < ck::kVStages; ++i) {
      mbar_init(&ctl->v_full[i], 1);
      mbar_init(&ctl->v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ctl->s_full[t], 1);
      mbar_init(&ctl->p_full[t], 128);
      mbar_init(&ctl->o_done[t], 1);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, ck::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int total = p.item_start[p.num_seqs];
  const int G = p.group;
  const int tpt = ck::kRows / G;  // query tokens per tile
  // Fills and phases so far, per ring / barrier (every role counts the same way).
  uint32_t kc = 0, vc = 0;         // K and V slices streamed by this CTA
  uint32_t sc[2] = {0u, 0u};       // slices of tile A / B computed
  uint32_t ic = 0;                 // items
  uint32_t kiss = 0, viss = 0;     // producer: K / V fills issued (for the final drain)
  uint32_t qiss = 0;               // producer: q fills issued

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
      CkItem it;
      const int rev = static_cast<int>(atomicAdd(&p.hdr->prefill_counter, 1u));
      const int item = total - 1 - rev;  // last items (latest tiles of the last runs) first
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
        const int npairs = (qtiles + 1) / 2;
        const int local = item - p.item_start[s];
        const int h = local / npairs;
        const int pi = local - h * npairs;
        it.s = s;
        it.h = h;
        it.L = L;
        for (int x = 0; x < 2; ++x) {
          const int i0 = (2 * pi + x) * tpt;
          it.t0[x] = t0 + i0;
          it.ntok[x] = max(0, min(tpt, n - i0));
          it.pos0[x] = L - n + i0;
        }
        it.has_b = it.ntok[1] > 0;
        const int xl = it.has_b ? 1 : 0;
        const int pmax = it.pos0[xl] + it.ntok[xl] - 1;
        it.nkv = pmax / ck::kKeys + 1;
        it.nblk = pmax / kBlockSize + 1;
      }
      ctl->item = it;
    }
    __syncthreads();
    const CkItem I = ctl->item;
    if (!I.valid || ctl->abort_flag) break;

    if (warp == 0) {
      // ---------------------------------------------------------------- producer (TMA) ----
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->q_full, ck::kTile * (I.has_b ? 2 : 1));
        for (int x = 0; x < (I.has_b ? 2 : 1); ++x) {
          uint8_t* q = smem + ck::kQ + x * ck::kTile;
          tma_load_3d(q, &qmap, 0, I.h * G, I.t0[x], &ctl->q_full);
          tma_load_3d(q + ck::kHalf, &qmap, 64, I.h * G, I.t0[x], &ctl->q_full);
        }
      }
      ++qiss;
      // Block-table entries are read 32 at a time (lane l holds block 32 * grp + l) with the
      // next group prefetched, so no copy waits on a dependent table load.
      const int32_t* trow = p.block_tables + static_cast<int64_t>(I.s) * p.max_blocks_per_seq;
      auto tab_load = [&](int grp) -> int {
        const int jb = 32 * grp + lane;
        return jb < I.nblk ? __ldg(trow + jb) : -1;
      };
      int grp_cur = 0;
      int tab_cur = tab_load(0);
      int tab_next = tab_load(1);
      const int yrow0 = I.h * 2;  // 8-row group of (block 0, this kv head)
      for (int j = 0; j < I.nkv; ++j) {
        const int grp = j >> 2;
        if (grp != grp_cur) {
          tab_cur = tab_next;
          tab_next = tab_load(grp + 1);
          grp_cur = grp;
        }
        const int e = __shfl_sync(0xffffffffu, tab_cur, 8 * (j & 3) + (lane & 7));
        const int jb = 8 * j + lane;
        int phys = -1;
        bool bad = false;
        if (lane < 8 && jb < I.nblk) {
          if (e < 0 || e >= p.num_blocks) {
            set_error(&p.hdr->error, PA_DEVERR_BLOCK_ID);
            bad = true;
          } else {
            phys = e;
          }
        }
        const uint32_t okm = __ballot_sync(0xffffffffu, phys >= 0);
        const uint32_t badm = __ballot_sync(0xffffffffu, bad);
        const uint32_t bytes = __popc(okm) * static_cast<uint32_t>(ck::kBlockBytes);
        const int ycoord = (phys * p.num_kv_heads) * 2 + yrow0;
        // K slice j
        {
          const uint32_t g = kc + j, st = g % ck::kKStages;
          if (!wait(&ctl->k_empty[st], ((g / ck::kKStages) & 1u) ^ 1u)) break;
          if (lane == 0) {
            if (bytes) mbar_arrive_expect_tx(&ctl->k_full[st], bytes);
            else mbar_arrive(&ctl->k_full[st]);
          }
          __syncwarp();
          // test hook: lane 0's copy of the first slice of the first item claimed is left out
          // (its bytes are still expected), so that the bounded waits on that stage expire
          const bool skip = p.skip_copy && I.first && j == 0 && lane == 0;
          if (phys >= 0 && !skip)
            tma_load_4d(smem + ck::kK + st * ck::kTile + lane * ck::kBlockBytes, &kmap, 0, 0,
                        0, ycoord, &ctl->k_full[st]);
          ++kiss;
        }
        // V slice j
        {
          const uint32_t g = vc + j, st = g % ck::kVStages;
          if (!wait(&ctl->v_empty[st], ((g / ck::kVStages) & 1u) ^ 1u)) break;
          if (lane == 0) {
            // rows the MMA warp has to clear: keys past the last valid one, and bad blocks
            const int valid_end = min(I.L, I.nblk * kBlockSize) - j * ck::kKeys;
            ctl->v_zero_from[st] = max(0, min(ck::kKeys, valid_end));
            ctl->v_bad[st] = badm;
            if (bytes) mbar_arrive_expect_tx(&ctl->v_full[st], bytes);
            else mbar_arrive(&ctl->v_full[st]);
          }
          __syncwarp();
          if (phys >= 0)
            tma_load_4d(smem + ck::kV + st * ck::kTile + lane * ck::kBlockBytes, &vmap, 0, 0,
                        0, ycoord, &ctl->v_full[st]);
          ++viss;
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer -------
      const uint32_t id_s = idesc_bf16_f32(128, 128, false);
      const uint32_t id_pv = idesc_bf16_f32(128, 128, true);
      const uint32_t q_addr = smem_u32(smem + ck::kQ);
      // S_X(j) = Q_X K(j)^T into the S/P columns of tile X
      auto issue_s = [&](int x, int j) {
        const uint32_t st = (kc + j) % ck::kKStages;
        if (lane == 0) {
          const uint32_t k_addr = smem_u32(smem + ck::kK + st * ck::kTile);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t qa = q_addr + x * ck::kTile + (ks >> 2) * ck::kHalf + (ks & 3) * 32;
            const uint32_t kb = k_addr + (ks >> 2) * 1024 + (ks & 3) * 32;
            tc_mma_bf16(tmem + x * 128u, smem_desc_sw128(qa, 16, 1024),
                        smem_desc_sw128(kb, 16, 2048), id_s, ks > 0);
          }
          tc_commit(&ctl->s_full[x]);
        }
        __syncwarp();
      };
      // O_X += P_X(j) V(j), P from tensor memory (bf16 hi then lo parts)
      auto issue_pv = [&](int x, int j) -> bool {
        if (!wait(&ctl->p_full[x], ((x ? sc[1] : sc[0]) + j) & 1u)) return false;
        tc_fence_after();
        const uint32_t st = (vc + j) % ck::kVStages;
        if (lane == 0) {
          const uint32_t v_addr = smem_u32(smem + ck::kV + st * ck::kTile);
          // keys 16 ks .. 16 ks + 15: hi parts in columns 32 (ks / 2) + 8 (ks % 2) + 0..7, lo
          // parts 16 columns further
          auto p_col = [&](int ks) {
            return tmem + x * 128u + (ks >> 1) * 32u + (ks & 1) * 8u;
          };
          const uint32_t o_col = tmem + ck::kOCol + x * 128u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(o_col, p_col(ks), smem_desc_sw128(v_addr + ks * 4096, 1024, 2048),
                           id_pv, j > 0 || ks > 0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(o_col, p_col(ks) + 16u,
                           smem_desc_sw128(v_addr + ks * 4096, 1024, 2048), id_pv, true);
          tc_commit(&ctl->o_done[x]);
        }
        __syncwarp();
        return true;
      };
      auto k_ready = [&](int j) -> bool {
        const uint32_t g = kc + j;
        if (!wait(&ctl->k_full[g % ck::kKStages], (g / ck::kKStages) & 1u)) return false;
        tc_fence_after();
        return true;
      };
      auto k_release = [&](int j) {
        if (lane == 0) tc_commit(&ctl->k_empty[(kc + j) % ck::kKStages]);
        __syncwarp();
      };
      bool ok = wait(&ctl->q_full, ic & 1u);
      if (ok) tc_fence_after();
      if (ok && (ok = k_ready(0))) {
        issue_s(0, 0);
        if (I.has_b) issue_s(1, 0);
        k_release(0);
      }
      for (int j = 0; ok && j < I.nkv; ++j) {
        const uint32_t g = vc + j, st = g % ck::kVStages;
        if (!(ok = wait(&ctl->v_full[st], (g / ck::kVStages) & 1u))) break;
        uint8_t* vt = smem + ck::kV + st * ck::kTile;
        const int zf = ctl->v_zero_from[st];
        const uint32_t badm = ctl->v_bad[st];
        if (zf < ck::kKeys || badm) {
          // clear the 128-byte rows (both column halves) of keys that hold no valid value;
          // key kk of the slice: block kk / 16, row group (kk / 8) % 2, row kk % 8
          for (int e = lane; e < ck::kKeys * 2 * 8; e += 32) {
            const int key = e >> 4, half = (e >> 3) & 1, c16 = e & 7;
            if (key >= zf || ((badm >> (key >> 4)) & 1u))
              *reinterpret_cast<uint4*>(vt + (key >> 3) * 2048 + half * 1024 + (key & 7) * 128 +
                                        c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (!(ok = issue_pv(0, j))) break;
        const bool more = j + 1 < I.nkv;
        if (more) {
          if (!(ok = k_ready(j + 1))) break;
          issue_s(0, j + 1);
          if (!I.has_b) k_release(j + 1);
        }
        if (I.has_b && !(ok = issue_pv(1, j))) break;
        if (lane == 0) tc_commit(&ctl->v_empty[st]);
        __syncwarp();
        if (I.has_b && more) {
          issue_s(1, j + 1);
          k_release(j + 1);
        }
      }
    } else {
      // ---------------------------------------------------------------- softmax rows -----
      const int x = (warp - 2) >> 2;       // tile: warps 2-5 A, 6-9 B
      const int quarter = warp & 3;        // TMEM lane quarter this warp may access
      const int r = quarter * 32 + lane;   // tile row = TMEM lane
      const int tok = r / G;
      const bool has_x = x == 0 || I.has_b;
      // (selects rather than indexing by x, which would put the arrays in local memory)
      const int ntok_x = x ? I.ntok[1] : I.ntok[0];
      const int t0_x = x ? I.t0[1] : I.t0[0];
      const uint32_t sc_x = x ? sc[1] : sc[0];
      const bool row_ok = has_x && tok < ntok_x;
      const int row_pos = (x ? I.pos0[1] : I.pos0[0]) + tok;
      const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      const uint32_t sb = tl + x * 128u;               // this row's S, then P
      const uint32_t ob = tl + ck::kOCol + x * 128u;   // this row's O
      const bool live = __any_sync(0xffffffffu, row_ok);
      float m_used = 0.f, l = 0.f;
      bool ok = true;
      for (int j = 0; has_x && j < I.nkv; ++j) {
        if (!(ok = wait(&ctl->s_full[x], (sc_x + j) & 1u))) break;
        tc_fence_after();
        // keys 0..kmax of the slice are visible to this row
        const int kmax = row_ok ? row_pos - j * ck::kKeys : -1;
        if (!live || __all_sync(0xffffffffu, kmax < 0)) {
          // no key of this slice is visible to any row of the warp: P = 0
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
          for (int c = 0; c < 8; ++c) tmem_st16(sb + c * 16, z);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&ctl->p_full[x]);
          continue;
        }
        // Two passes over the row of S in tensor memory (reads there are cheap), 32 columns
        // at a time, so that few registers stay live: the row max of the visible keys, then
        // the probabilities.  Scores are used in the log2 domain (times scale * log2 e).
        const bool full = __all_sync(0xffffffffu, kmax >= ck::kKeys - 1);  // warp-uniform
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t sv[32];
          tmem_ld32(sb + c * 32, sv);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float v = __uint_as_float(sv[i]);
            mx[i & 7] = fmaxf(mx[i & 7], (full || c * 32 + i <= kmax) ? v : -CUDART_INF_F);
          }
        }
        float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        mt = mt == -CUDART_INF_F ? mt : mt * p.score_log2;  // scale > 0 keeps the order
        bool rescale = false;
        float m_new = m_used;
        if (j == 0) {
          m_new = (mt == -CUDART_INF_F) ? 0.f : mt;
        } else if (mt > m_used + ck::kRescaleLog2) {
          m_new = mt;
          rescale = true;
        }
        const float alpha = rescale ? fast_exp2(m_used - m_new) : 1.f;
        // probabilities 2^(s * c - m); for every 32 keys, bf16 hi parts into their columns
        // 0..15 and lo parts into 16..31 (so a chunk overwrites only the scores it has read)
        float rsum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rsum[i] = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t sv[32];
          tmem_ld32(sb + c * 32, sv);
          tmem_wait_ld();
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i0 = c * 32 + 2 * e;
            const float x0 = (full || i0 <= kmax)
                                 ? fmaf(__uint_as_float(sv[2 * e]), p.score_log2, -m_new)
                                 : -CUDART_INF_F;
            const float x1 = (full || i0 + 1 <= kmax)
                                 ? fmaf(__uint_as_float(sv[2 * e + 1]), p.score_log2, -m_new)
                                 : -CUDART_INF_F;
            const float p0 = fast_exp2(x0);
            const float p1 = fast_exp2(x1);
            rsum[e & 7] += p0 + p1;
            hi[e] = pack_bf16x2(p0, p1);
            lo[e] = pack_bf16x2(p0 - bf16lo_to_f32(hi[e]), p1 - bf16hi_to_f32(hi[e]));
          }
          // the chunk's own 32 columns, already read: hi parts first, then lo parts
          tmem_st16(sb + c * 32, hi);
          tmem_st16(sb + c * 32 + 16, lo);
        }
        const float rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) +
                         ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
        l = l * alpha + rs;
        if (__any_sync(0xffffffffu, rescale)) {
          // the commit of S_X(j) also covered PV_X(j - 1): O_X is complete and may be scaled
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_ld32(ob + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(ob + c * 32, o);
          }
        }
        tmem_wait_st();
        m_used = m_new;
        tc_fence_before();
        mbar_arrive(&ctl->p_full[x]);
      }
      // epilogue: the row of O divided by the row sum
      const uint32_t g_last = sc_x + I.nkv - 1;
      if (ok && has_x && live && wait(&ctl->o_done[x], g_last & 1u)) {
        tc_fence_after();
        const float inv = (row_ok && l > 0.f) ? 1.f / l : 0.f;
        const int64_t orow =
            static_cast<int64_t>(t0_x + tok) * p.num_q_heads + I.h * G + r % G;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(ob + c * 32, o);
          tmem_wait_ld();
          if (row_ok) {
            if (p.out_bf16) {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                    orow * 128 + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  w[e] = pack_bf16x2(__uint_as_float(o[8 * i + 2 * e]) * inv,
                                     __uint_as_float(o[8 * i + 2 * e + 1]) * inv);
                dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) +
                                                      orow * 128 + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv,
                                     __uint_as_float(o[4 * i + 1]) * inv,
                                     __uint_as_float(o[4 * i + 2]) * inv,
                                     __uint_as_float(o[4 * i + 3]) * inv);
            }
          }
        }
      }
    }
    tc_fence_before();
    kc += I.nkv;
    vc += I.nkv;
    sc[0] += I.nkv;
    sc[1] += I.has_b ? I.nkv : 0;
    ++ic;
    __syncthreads();
    tc_fence_after();
  }
  // Exit, normal or after an expired wait: no copy may still be landing in shared memory and
  // no MMA may still be using tensor memory when the CTA ends.
  if (warp == 0) {
    // the latest fill of each stage is the only one that can still be in flight
    for (uint32_t g = kiss > ck::kKStages ? kiss - ck::kKStages : 0; g < kiss; ++g)
      mbar_wait(&ctl->k_full[g % ck::kKStages], (g / ck::kKStages) & 1u, p.wait_ns);
    for (uint32_t g = viss > ck::kVStages ? viss - ck::kVStages : 0; g < viss; ++g)
      mbar_wait(&ctl->v_full[g % ck::kVStages], (g / ck::kVStages) & 1u, p.wait_ns);
    if (qiss) mbar_wait(&ctl->q_full, (qiss - 1) & 1u, p.wait_ns);
  } else if (warp == 1) {
    if (lane == 0) tc_commit(&ctl->drain);
    __syncwarp();
    mbar_wait(&ctl->drain, 0, p.wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, ck::kTmemCols);
}

cudaError_t launch_chunk(const AttnArgs& a, const PrefillParams& p, const CUtensorMap& qmap,
                         const CUtensorMap& kmap4, const CUtensorMap& vmap4) {
  LaunchInfo li;
  cudaError_t e = launch_info(chunk_kernel, ck::kThreads, ck::kSmem, &li);
  if (e != cudaSuccess) return e;
  // pairs of 128-row tiles: at most one per 256 rows of the step plus one per sequence
  const int64_t upper =
      static_cast<int64_t>(a.num_kv_heads) *
      ((static_cast<int64_t>(a.num_q_tokens) * p.group + 2 * ck::kRows - 1) / (2 * ck::kRows) +
       a.num_seqs);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(upper, li.sms));
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_before, a.stream);
  chunk_kernel<<<static_cast<unsigned>(grid), ck::kThreads, ck::kSmem, a.stream>>>(qmap, kmap4,
                                                                                  vmap4, p);
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_after, a.stream);
  return cudaGetLastError();
}

}  // namespace pa
