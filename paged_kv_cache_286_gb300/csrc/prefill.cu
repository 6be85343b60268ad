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
//  * Warp 1 issues tcgen05.mma from one thread: S = Q K^T into one of two TMEM buffers
//    (128 x 128 fp32), and O += P V into a third, with P read from TMEM and V from shared
//    memory (MN-major).  The softmax threads write P back over their S buffer as bf16 hi and lo
//    halves (64 columns each), so P V is exact to ~2^-16 like the decode path, and the next
//    tile's softmax can run while this tile's P V is in flight.
//  * Warps 2-5 own one row each: they read the row of S from TMEM once, mask keys beyond the
//    row's position, keep the running max in the log2 domain and rescale O in TMEM only when
//    the max grows by more than 2^8 (the final division uses the same max, so the result is
//    exact), and finally divide O by the row sum and store it.
//  * V rows past the last valid key (stale slots, possibly NaN) are zeroed in shared memory
//    before P V reads them; K there only feeds masked scores.
#include <math_constants.h>

#include <algorithm>

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
constexpr int kSmem = 1024 + kCtl + 256;
constexpr int kThreads = 224;
constexpr int kVWarp = 6;     // V producer (warp 0 loads q and K)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = kSBufs * 128;
constexpr float kRescaleLog2 = 8.f;
}  // namespace pf

struct PrefillParams {
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* qsl;
  const int32_t* item_start;  // [S+1] prefix sums of prefill items
  void* out;
  WsHeader* hdr;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t num_blocks;
  int32_t out_bf16;
  float score_log2;
};

struct PfItem {
  int s, h, t0, ntok, pos0, L, nkv, nblk_tile, valid;
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

__global__ void __launch_bounds__(pf::kThreads, 1)
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
      mbar_init(&ctl->p_full[i], pf::kRows);
      mbar_init(&ctl->o_done[i], 1);
    }
    ctl->abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, pf::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int total = p.item_start[p.num_seqs];
  uint32_t tc = 0;  // KV tiles processed by this CTA so far (ring / phase tracking)
  uint32_t ic = 0;  // items processed by this CTA so far
  const int G = p.group;
  const int tpt = pf::kRows / G;  // query tokens per tile

  auto fail = [&](uint32_t bits) {
    set_error(&p.hdr->error, bits);
    ctl->abort_flag = 1;
  };
  // all lanes wait; the outcome is warp-uniform
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity));
    if (!ok && lane == 0) fail(PA_DEVERR_TIMEOUT);
    return ok;
  };

  while (true) {
    if (tid == 0) {
      PfItem it;
      const int rev = static_cast<int>(atomicAdd(&p.hdr->prefill_counter, 1u));
      const int item = total - 1 - rev;  // longest items (last tiles of a chunk) first
      it.valid = item >= 0;
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
        if (phys >= 0) {
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
          const uint32_t p_hi = tmem + b * 128u, p_lo = p_hi + 64u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(tmem + pf::kOCol, p_hi + ks * 8,
                           smem_desc_sw128(v_addr + ks * 2048, pf::kHalf, 1024), id_pv,
                           j > 0 || ks > 0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_bf16_ts(tmem + pf::kOCol, p_lo + ks * 8,
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
      const int quarter = warp & 3;        // TMEM lane quarter this warp may access
      const int r = quarter * 32 + lane;   // tile row = TMEM lane
      const int tok = r / G;
      const bool row_ok = tok < I.ntok;
      const int row_pos = I.pos0 + tok;
      const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      float m_used = 0.f, l = 0.f;
      bool ok = true;
      for (int j = 0; j < I.nkv; ++j) {
        const uint32_t g = tc + j, b = g % pf::kSBufs;
        if (!(ok = wait(&ctl->s_full[b], (g / pf::kSBufs) & 1u))) break;
        tc_fence_after();
        const int kmax = row_ok ? row_pos - j * pf::kKeys : -1;  // keys 0..kmax are visible
        if (!__any_sync(0xffffffffu, row_ok)) {  // a quarter of rows past the run: P = 0
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
          for (int c = 0; c < 8; ++c) tmem_st16(tl + b * 128u + c * 16, z);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&ctl->p_full[b]);
          continue;
        }
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tl + b * 128u + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
        tmem_wait_ld();
        // scores in the log2 domain; masked keys become -inf.  Eight independent max / sum
        // accumulators keep the dependency chains short.
        float x[128];
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -CUDART_INF_F;
        if (__all_sync(0xffffffffu, kmax >= pf::kKeys - 1)) {  // warp-uniform branch
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            x[i] = __uint_as_float(sv[i]) * p.score_log2;
            mx[i & 7] = fmaxf(mx[i & 7], x[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            x[i] = (i <= kmax) ? __uint_as_float(sv[i]) * p.score_log2 : -CUDART_INF_F;
            mx[i & 7] = fmaxf(mx[i & 7], x[i]);
          }
        }
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        bool rescale = false;
        float m_new = m_used;
        if (j == 0) {
          m_new = (mt == -CUDART_INF_F) ? 0.f : mt;
        } else if (mt > m_used + pf::kRescaleLog2) {
          m_new = mt;
          rescale = true;
        }
        const float alpha = rescale ? fast_exp2(m_used - m_new) : 1.f;
        // probabilities; bf16 hi halves into columns 0..63 of the buffer, lo into 64..127
        float rsum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rsum[i] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = fast_exp2(x[c * 32 + 2 * e] - m_new);
            const float p1 = fast_exp2(x[c * 32 + 2 * e + 1] - m_new);
            rsum[e & 7] += p0 + p1;
            hi[e] = pack_bf16x2(p0, p1);
            lo[e] = pack_bf16x2(p0 - bf16lo_to_f32(hi[e]), p1 - bf16hi_to_f32(hi[e]));
          }
          tmem_st16(tl + b * 128u + c * 16, hi);
          tmem_st16(tl + b * 128u + 64 + c * 16, lo);
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
          uint32_t o[128];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld32(tl + pf::kOCol + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 128; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_st32(tl + pf::kOCol + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
        }
        tmem_wait_st();
        m_used = m_new;
        tc_fence_before();
        mbar_arrive(&ctl->p_full[b]);
      }
      // epilogue: O / l
      const uint32_t g_last = tc + I.nkv - 1;
      if (ok && wait(&ctl->o_done[g_last % pf::kSBufs], (g_last / pf::kSBufs) & 1u)) {
        tc_fence_after();
        const float inv = (row_ok && l > 0.f) ? 1.f / l : 0.f;
        const int64_t orow = static_cast<int64_t>(I.t0 + tok) * p.num_q_heads + I.h * G + r % G;
        uint32_t o[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tl + pf::kOCol + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
        tmem_wait_ld();
        if (row_ok) {
          if (p.out_bf16) {
            uint4* dst =
                reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * 128);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(__uint_as_float(o[8 * i + 2 * e]) * inv,
                                   __uint_as_float(o[8 * i + 2 * e + 1]) * inv);
              dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * 128);
#pragma unroll
            for (int i = 0; i < 32; ++i)
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

size_t prefill_smem_bytes() { return pf::kSmem; }

cudaError_t launch_prefill(const AttnArgs& a, const int32_t* item_start, WsHeader* hdr,
                           const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap) {
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
  LaunchInfo li;
  cudaError_t e = launch_info(prefill_kernel, pf::kThreads, pf::kSmem, &li);
  if (e != cudaSuccess) return e;
  const int sms = li.sms;
  const int G = p.group;
  const int64_t upper =
      static_cast<int64_t>(a.num_kv_heads) *
      ((static_cast<int64_t>(a.num_q_tokens) * G + pf::kRows - 1) / pf::kRows + a.num_seqs);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(upper, sms));
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_before, a.stream);
  prefill_kernel<<<static_cast<unsigned>(grid), pf::kThreads, pf::kSmem, a.stream>>>(qmap, kmap,
                                                                                     vmap, p);
  if (a.pf_before && a.pf_after) cudaEventRecord(a.pf_after, a.stream);
  return cudaGetLastError();
}

}  // namespace pa
