// Host-side block manager of the paged KV pool: free list, per-sequence block tables, reference
// counts with copy-on-write, and a prefix cache of full blocks keyed by a chained hash with
// least-recently-used eviction.  See include/pa_block_manager.h for the contract and the pages'
// sections each piece follows.
#include "pa_block_manager.h"

#include <cstring>
#include <deque>
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

namespace {

constexpr uint64_t kRootHash = 0x9E3779B97F4A7C15ull;

// 64-bit hash of a block's token ids chained with the hash of everything before it.
uint64_t chain_hash(uint64_t parent, const int32_t* tokens, int32_t n) {
  uint64_t h = parent ^ 0xD6E8FEB86659FD93ull;
  for (int32_t i = 0; i < n; ++i) {
    h ^= static_cast<uint32_t>(tokens[i]);
    h *= 0x9FB21C651E98DF25ull;
    h ^= h >> 29;
  }
  h ^= static_cast<uint64_t>(n);
  h *= 0xBF58476D1CE4E5B9ull;
  return h ^ (h >> 31);
}

struct Seq {
  std::vector<int32_t> blocks;
  int64_t ntok = 0;
  bool hashing = true;             // every token so far came with its id
  uint64_t chain = kRootHash;      // hash through the last full block
  std::vector<int32_t> tail;       // token ids of the partly filled last block
};

}  // namespace

struct pa_block_manager {
  int32_t nb = 0, bs = 0;
  std::vector<int32_t> ref;
  std::deque<int32_t> free_list;
  std::vector<char> hashed;
  std::vector<uint64_t> block_hash;
  std::vector<std::vector<int32_t>> block_tokens;
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::list<int32_t> lru;  // evictable cached blocks, least recently released first
  std::vector<std::list<int32_t>::iterator> lru_pos;
  std::vector<char> in_lru;
  std::unordered_map<int64_t, Seq> seqs;

  int32_t available() const { return static_cast<int32_t>(free_list.size() + lru.size()); }

  int32_t take() {  // caller has checked availability
    int32_t b;
    if (!free_list.empty()) {
      b = free_list.front();
      free_list.pop_front();
    } else {
      b = lru.front();
      lru.pop_front();
      in_lru[b] = 0;
      auto it = by_hash.find(block_hash[b]);
      if (it != by_hash.end() && it->second == b) by_hash.erase(it);
      hashed[b] = 0;
      block_tokens[b].clear();
    }
    ref[b] = 1;
    return b;
  }

  void drop(int32_t b) {
    if (--ref[b] > 0) return;
    if (hashed[b]) {
      lru.push_back(b);
      lru_pos[b] = std::prev(lru.end());
      in_lru[b] = 1;
    } else {
      free_list.push_back(b);
    }
  }

  void revive(int32_t b) {
    if (ref[b] == 0 && in_lru[b]) {
      lru.erase(lru_pos[b]);
      in_lru[b] = 0;
    }
    ++ref[b];
  }

  // Cached block holding exactly `tokens` after the prefix with hash `parent`, or -1.
  int32_t lookup(uint64_t parent, const int32_t* tokens, uint64_t* h_out) const {
    const uint64_t h = chain_hash(parent, tokens, bs);
    *h_out = h;
    auto it = by_hash.find(h);
    if (it == by_hash.end()) return -1;
    const int32_t b = it->second;
    if (!hashed[b] || std::memcmp(block_tokens[b].data(), tokens, sizeof(int32_t) * bs) != 0)
      return -1;
    return b;
  }

  int32_t append(int64_t seq, const int32_t* tokens, int32_t n, int64_t* slots,
                 int32_t* pairs, int32_t cap, int32_t* cached_out) {
    if (n < 0 || (n > 0 && !slots)) return PA_BM_BAD_ARG;
    if (cached_out) *cached_out = 0;
    auto found = seqs.find(seq);
    const bool fresh = found == seqs.end();
    Seq scratch;
    Seq& s = fresh ? scratch : found->second;

    // leading cached blocks (only for a sequence with no tokens yet, tokens known)
    std::vector<int32_t> hits;
    std::vector<uint64_t> hit_hash;
    if (tokens && s.ntok == 0) {
      uint64_t parent = s.chain;
      for (int32_t off = 0; off + bs <= n; off += bs) {
        uint64_t h;
        const int32_t b = lookup(parent, tokens + off, &h);
        if (b < 0) break;
        hits.push_back(b);
        hit_hash.push_back(h);
        parent = h;
      }
    }
    int32_t revived_from_lru = 0;
    for (int32_t b : hits)
      if (ref[b] == 0 && in_lru[b]) ++revived_from_lru;
    const int64_t cur = s.ntok + static_cast<int64_t>(hits.size()) * bs;
    const int32_t rest = n - static_cast<int32_t>(hits.size()) * bs;
    const bool partial_last = (cur % bs) != 0;
    const bool cow = rest > 0 && partial_last && !s.blocks.empty() && ref[s.blocks.back()] > 1;
    const int64_t room = partial_last ? bs - cur % bs : 0;
    const int64_t new_blocks = rest > room ? (rest - room + bs - 1) / bs : 0;
    const int64_t need = new_blocks + (cow ? 1 : 0);
    if (need > available() - revived_from_lru) return PA_BM_NO_SPACE;
    if (cow && cap < 1) return PA_BM_BAD_ARG;

    Seq& t = fresh ? seqs[seq] : s;
    int32_t npairs = 0;
    int64_t slot_i = 0;
    for (size_t i = 0; i < hits.size(); ++i) {
      revive(hits[i]);
      t.blocks.push_back(hits[i]);
      for (int32_t o = 0; o < bs; ++o) slots[slot_i++] = static_cast<int64_t>(hits[i]) * bs + o;
      t.ntok += bs;
      t.chain = hit_hash[i];
    }
    if (cached_out) *cached_out = static_cast<int32_t>(hits.size()) * bs;
    if (cow) {
      const int32_t old = t.blocks.back();
      const int32_t nbk = take();
      pairs[0] = old;
      pairs[1] = nbk;
      npairs = 1;
      drop(old);
      t.blocks.back() = nbk;
    }
    if (!tokens && rest > 0) t.hashing = false;
    for (int32_t i = 0; i < rest; ++i) {
      if (t.ntok % bs == 0) t.blocks.push_back(take());
      const int32_t b = t.blocks[t.ntok / bs];
      slots[slot_i++] = static_cast<int64_t>(b) * bs + t.ntok % bs;
      ++t.ntok;
      if (t.hashing && tokens) {
        t.tail.push_back(tokens[static_cast<int32_t>(hits.size()) * bs + i]);
        if (t.ntok % bs == 0) {  // block full: register it in the prefix cache
          const uint64_t h = chain_hash(t.chain, t.tail.data(), bs);
          if (by_hash.find(h) == by_hash.end() && !hashed[b]) {
            by_hash[h] = b;
            hashed[b] = 1;
            block_hash[b] = h;
            block_tokens[b] = t.tail;
          }
          t.chain = h;
          t.tail.clear();
        }
      }
    }
    return npairs;
  }
};

extern "C" {

pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return nullptr;
  bm->nb = num_blocks;
  bm->bs = block_size;
  bm->ref.assign(num_blocks, 0);
  bm->hashed.assign(num_blocks, 0);
  bm->block_hash.assign(num_blocks, 0);
  bm->block_tokens.resize(num_blocks);
  bm->lru_pos.resize(num_blocks);
  bm->in_lru.assign(num_blocks, 0);
  for (int32_t b = 0; b < num_blocks; ++b) bm->free_list.push_back(b);
  return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int32_t pa_bm_num_free(const pa_block_manager* bm) { return bm ? bm->available() : 0; }

int32_t pa_bm_append(pa_block_manager* bm, int64_t seq, int32_t n, int64_t* slots_out,
                     int32_t* copy_pairs_out, int32_t copy_cap) {
  if (!bm) return PA_BM_BAD_ARG;
  return bm->append(seq, nullptr, n, slots_out, copy_pairs_out, copy_cap, nullptr);
}

int32_t pa_bm_append_tokens(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int32_t n,
                            int64_t* slots_out, int32_t* copy_pairs_out, int32_t copy_cap,
                            int32_t* cached_tokens_out) {
  if (!bm || (n > 0 && !tokens)) return PA_BM_BAD_ARG;
  return bm->append(seq, tokens, n, slots_out, copy_pairs_out, copy_cap, cached_tokens_out);
}

int32_t pa_bm_cached_prefix(const pa_block_manager* bm, const int32_t* tokens, int32_t n) {
  if (!bm || n < 0 || (n > 0 && !tokens)) return PA_BM_BAD_ARG;
  uint64_t parent = kRootHash;
  int32_t hit = 0;
  for (int32_t off = 0; off + bm->bs <= n; off += bm->bs) {
    uint64_t h;
    if (bm->lookup(parent, tokens + off, &h) < 0) break;
    parent = h;
    hit += bm->bs;
  }
  return hit;
}

int32_t pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return PA_BM_BAD_ARG;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end() || bm->seqs.count(child)) return PA_BM_BAD_ARG;
  Seq copy = it->second;
  for (int32_t b : copy.blocks) ++bm->ref[b];
  bm->seqs.emplace(child, std::move(copy));
  return 0;
}

int32_t pa_bm_free(pa_block_manager* bm, int64_t seq) {
  if (!bm) return PA_BM_BAD_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_BM_BAD_ARG;
  for (int32_t b : it->second.blocks) bm->drop(b);
  bm->seqs.erase(it);
  return 0;
}

int32_t pa_bm_block_table(const pa_block_manager* bm, int64_t seq, int32_t* table_out,
                          int32_t cap) {
  if (!bm) return PA_BM_BAD_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_BM_BAD_ARG;
  const auto& blocks = it->second.blocks;
  const int32_t n = static_cast<int32_t>(blocks.size());
  for (int32_t i = 0; i < n && i < cap; ++i) table_out[i] = blocks[i];
  return n;
}

int64_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq) {
  if (!bm) return PA_BM_BAD_ARG;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? PA_BM_BAD_ARG : it->second.ntok;
}

int32_t pa_bm_refcount(const pa_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->nb) return PA_BM_BAD_ARG;
  return bm->ref[block];
}

}  // extern "C"
