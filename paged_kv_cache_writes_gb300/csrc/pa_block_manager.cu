// pa_block_manager.cu -- host-side block manager behind the C ABI: the block
// table bookkeeping that feeds the kernels (no device code).
//
// What it keeps ("Inside vLLM Architecture", section "The Block Table Mapping
// Subsystem"; "Inside vLLM v0.7 ...", section "Architectural Blueprint 2: How
// PagedAttention Actually Works"; "High-Throughput LLM Serving with vLLM &
// PagedAttention", section "2. Virtual Memory Paging Applied to GPUs"):
//  * a pool of num_blocks physical blocks of block_size token slots, a free
//    list, and a reference count per block;
//  * per sequence, its length and block table (logical block i -> physical
//    block); a token at position p lives in slot table[p / bs] * bs + p % bs;
//  * blocks are taken on demand, one when a sequence crosses into a new
//    logical block, so a sequence wastes at most block_size - 1 slots;
//  * fork: a child shares every block of its parent (reference counts rise);
//  * copy-on-write: appending into a last block that is shared first copies
//    it into a fresh block (the caller runs pa_copy_blocks on the returned
//    (src, dst) pairs before writing);
//  * prefix reuse: a full block can be identified by a chained hash of its
//    token ids (hash of the previous full block, then the block's ids).  When
//    an append fills a whole logical block whose ids match a block already in
//    the pool, that block is shared instead of allocated and its tokens get
//    slot -1 (pa_reshape_and_cache skips them: their K/V are already there).
// Not thread-safe: one manager per thread, or external locking.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Seq {
  std::vector<int32_t> blocks;
  int64_t len = 0;
  uint64_t chain = 0;       // hash of the last full block (0: the empty prefix)
  bool chain_known = true;  // every full block so far had its ids given: the prefix can be matched
  bool live = false;
};

uint64_t mix64(uint64_t x) {  // splitmix64 finaliser
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

uint64_t block_hash(uint64_t prev, const int32_t *ids, int32_t n) {
  uint64_t h = mix64(prev ^ 0x5ee5c0deull);
  for (int32_t i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint32_t>(ids[i]));
  return h | 1;  // never 0 (0 marks "no hash")
}

}  // namespace

struct pa_block_manager {
  int32_t num_blocks = 0, block_size = 0;
  std::vector<int32_t> ref;                   // per physical block
  std::vector<int32_t> free_list;             // blocks with ref 0; taken from the back
  std::vector<Seq> seqs;
  // prefix cache: hash -> block; per cached block: its hash and token ids
  std::unordered_map<uint64_t, int32_t> cache;
  std::vector<uint64_t> hash_of;              // 0: block not in the cache
  std::vector<uint64_t> prev_of;              // chain hash of the prefix before a cached block
  std::vector<int32_t> ids_of;                // [num_blocks][block_size] token ids of cached blocks

  int32_t take() {
    const int32_t b = free_list.back();
    free_list.pop_back();
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) {
      if (hash_of[b]) {
        auto it = cache.find(hash_of[b]);
        if (it != cache.end() && it->second == b) cache.erase(it);
        hash_of[b] = 0;
      }
      free_list.push_back(b);
    }
  }
  bool valid_seq(int32_t s) const { return s >= 0 && s < (int32_t)seqs.size() && seqs[s].live; }
};

extern "C" {

pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, uint64_t shuffle_seed, pa_block_manager **bm) {
  if (!bm) return PA_ERR_INVALID_ARG;
  *bm = nullptr;
  if (num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  pa_block_manager *m = new (std::nothrow) pa_block_manager;
  if (!m) return PA_ERR_UNSUPPORTED;
  try {
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->ref.assign(num_blocks, 0);
    m->hash_of.assign(num_blocks, 0);
    m->prev_of.assign(num_blocks, 0);
    m->ids_of.assign((size_t)num_blocks * block_size, 0);
    // taken from the back: lowest ids first, or a seeded shuffle (Fisher-Yates)
    m->free_list.resize(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) m->free_list[i] = num_blocks - 1 - i;
    if (shuffle_seed) {
      uint64_t st = shuffle_seed;
      for (int32_t i = num_blocks - 1; i > 0; --i) {
        st = mix64(st);
        const int32_t j = (int32_t)(st % (uint64_t)(i + 1));
        std::swap(m->free_list[i], m->free_list[j]);
      }
    }
  } catch (...) {
    delete m;
    return PA_ERR_UNSUPPORTED;
  }
  *bm = m;
  return PA_OK;
}

void pa_bm_destroy(pa_block_manager *bm) { delete bm; }

pa_status pa_bm_new_sequence(pa_block_manager *bm, int32_t *seq) {
  if (!bm || !seq) return PA_ERR_INVALID_ARG;
  try {
    bm->seqs.emplace_back();
  } catch (...) {
    return PA_ERR_UNSUPPORTED;
  }
  bm->seqs.back().live = true;
  *seq = (int32_t)bm->seqs.size() - 1;
  return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager *bm, int32_t parent, int32_t *child) {
  if (!bm || !child || !bm->valid_seq(parent)) return PA_ERR_INVALID_ARG;
  try {
    Seq c = bm->seqs[parent];
    for (int32_t b : c.blocks) ++bm->ref[b];
    bm->seqs.push_back(std::move(c));
  } catch (...) {
    return PA_ERR_UNSUPPORTED;
  }
  *child = (int32_t)bm->seqs.size() - 1;
  return PA_OK;
}

pa_status pa_bm_append(pa_block_manager *bm, int32_t seq, int32_t num_tokens, const int32_t *token_ids,
                       int64_t *slots, int32_t *cow_pairs, int32_t cow_capacity, int32_t *num_cow) {
  if (!bm || !num_cow || !bm->valid_seq(seq) || num_tokens < 0 || cow_capacity < 0) return PA_ERR_INVALID_ARG;
  if (num_tokens > 0 && !slots) return PA_ERR_INVALID_ARG;
  *num_cow = 0;
  Seq &s = bm->seqs[seq];
  const int32_t bs = bm->block_size;
  const int32_t off = (int32_t)(s.len % bs);
  // worst case (no prefix reuse): the new logical blocks, plus one copy of a shared last block
  const bool cow = off != 0 && num_tokens > 0 && bm->ref[s.blocks.back()] > 1;
  const int64_t need = (off + (int64_t)num_tokens + bs - 1) / bs - (off ? 1 : 0) + (cow ? 1 : 0);
  if (need > (int64_t)bm->free_list.size()) return PA_ERR_NO_BLOCKS;
  if (cow && (cow_capacity < 1 || !cow_pairs)) {
    *num_cow = 1;
    return PA_ERR_INVALID_ARG;
  }
  if ((int64_t)s.blocks.size() + need > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (cow) {
    const int32_t src = s.blocks.back(), dst = bm->take();
    bm->release(src);
    s.blocks.back() = dst;
    cow_pairs[0] = src;
    cow_pairs[1] = dst;
    *num_cow = 1;
  }
  int32_t t = 0;
  while (t < num_tokens) {
    const int64_t p = s.len;
    const int32_t o = (int32_t)(p % bs);
    if (o == 0) {
      // a new logical block: share an identical full block if the ids are known and cached
      if (token_ids && s.chain_known && num_tokens - t >= bs) {
        const uint64_t h = block_hash(s.chain, token_ids + t, bs);
        auto it = bm->cache.find(h);
        if (it != bm->cache.end() && bm->prev_of[it->second] == s.chain &&
            std::memcmp(&bm->ids_of[(size_t)it->second * bs], token_ids + t, sizeof(int32_t) * bs) == 0) {
          const int32_t b = it->second;
          ++bm->ref[b];
          s.blocks.push_back(b);
          for (int32_t i = 0; i < bs; ++i) slots[t + i] = -1;  // already in the cache
          s.len += bs;
          s.chain = h;
          t += bs;
          continue;
        }
      }
      s.blocks.push_back(bm->take());
    }
    const int32_t b = s.blocks.back();
    slots[t] = (int64_t)b * bs + o;
    ++s.len;
    ++t;
    if (s.len % bs == 0 && token_ids) {
      // the block is full: publish it for prefix reuse (its ids: the last bs of this append,
      // available only when the whole block was written by this call)
      const int32_t first = t - bs;
      if (s.chain_known && first >= 0 && bm->ref[b] == 1) {
        const uint64_t h = block_hash(s.chain, token_ids + first, bs);
        if (!bm->cache.count(h) && !bm->hash_of[b]) {
          bm->cache.emplace(h, b);
          bm->hash_of[b] = h;
          bm->prev_of[b] = s.chain;
          std::memcpy(&bm->ids_of[(size_t)b * bs], token_ids + first, sizeof(int32_t) * bs);
        }
        s.chain = h;
      } else {
        s.chain_known = false;  // ids of this block unknown: later blocks cannot be matched either
      }
    } else if (s.len % bs == 0) {
      s.chain_known = false;
    }
  }
  return PA_OK;
}

pa_status pa_bm_free(pa_block_manager *bm, int32_t seq) {
  if (!bm || !bm->valid_seq(seq)) return PA_ERR_INVALID_ARG;
  Seq &s = bm->seqs[seq];
  for (int32_t b : s.blocks) bm->release(b);
  s.blocks.clear();
  s.blocks.shrink_to_fit();
  s.len = 0;
  s.chain = 0;
  s.chain_known = true;
  s.live = false;
  return PA_OK;
}

pa_status pa_bm_block_table(const pa_block_manager *bm, int32_t seq, int32_t *table, int32_t capacity,
                            int32_t *num_blocks, int32_t *seq_len) {
  if (!bm || !num_blocks || !seq_len || !bm->valid_seq(seq) || capacity < 0) return PA_ERR_INVALID_ARG;
  const Seq &s = bm->seqs[seq];
  *num_blocks = (int32_t)s.blocks.size();
  *seq_len = (int32_t)std::min<int64_t>(s.len, INT32_MAX);
  if ((int32_t)s.blocks.size() > capacity) return PA_ERR_INVALID_ARG;
  if (!s.blocks.empty()) {
    if (!table) return PA_ERR_INVALID_ARG;
    std::memcpy(table, s.blocks.data(), sizeof(int32_t) * s.blocks.size());
  }
  return PA_OK;
}

pa_status pa_bm_get_stats(const pa_block_manager *bm, pa_bm_stats *st) {
  if (!bm || !st) return PA_ERR_INVALID_ARG;
  pa_bm_stats r{};
  r.free_blocks = (int32_t)bm->free_list.size();
  for (int32_t v : bm->ref) {
    r.used_blocks += v > 0;
    r.shared_blocks += v > 1;
  }
  for (const Seq &s : bm->seqs)
    if (s.live) {
      r.live_sequences += 1;
      r.logical_tokens += s.len;
      r.logical_blocks += (int64_t)s.blocks.size();
    }
  r.cached_blocks = (int32_t)bm->cache.size();
  *st = r;
  return PA_OK;
}

}  // extern "C"
