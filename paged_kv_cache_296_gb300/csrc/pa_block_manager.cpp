// The KV block manager (host) behind the pa_bm_* entry points of include/pa.h.
//
// What it follows ("vLLM 部署深度指南", section 代码层面理解, the
// PagedAttentionKVCache sketch; "vLLM GitHub 项目…", section 二 items 1 and 4,
// section 三 item 1): a free list that starts as every block id in increasing
// order and hands out blocks from its front; a sequence of n tokens holds
// ceil(n / block_size) blocks and takes a new one when a token falls past its
// last block; running out of blocks is an out-of-memory error; sequences may
// share physical blocks (parallel sampling, beam search) and release them as
// soon as they finish.  Where the pages are silent: a request that does not
// fit changes nothing; blocks are reference counted and go to the back of the
// free list (in table order) when the last table lets go; a write into a block
// another table also holds first moves the writer to a private copy (the
// (src, dst) pair is returned for pa_copy_blocks).
//
// Prefix caching ("vLLM 部署深度指南", Prefix Caching 加速 table, 前缀共享 row;
// "vLLM高性能推理引擎实战解密", section 3.1, cross-request sharing of a common
// prefix): a full block serves any request whose tokens, from the first up to
// that block's last, are the same.  It is found by the exact key (parent
// block, the parent's generation, the block's tokens); the generation counts
// how often a block id was handed out, so keys naming a since-reused block
// never match.  Released cached blocks stay on the free list, findable, until
// the allocator hands them out (which drops their key); at least one prompt
// token is always left to compute.
//
// Every call takes the manager's mutex, so one manager may be driven from
// several host threads.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

// Key of a cached block: parent block (-1 at a sequence's start), the
// parent's generation, and the block's token ids.
struct CacheKey {
  int32_t parent = -1;
  uint32_t parent_gen = 0;
  std::vector<int32_t> tokens;
  bool operator==(const CacheKey& o) const {
    return parent == o.parent && parent_gen == o.parent_gen && tokens == o.tokens;
  }
};

struct CacheKeyHash {
  size_t operator()(const CacheKey& k) const {
    uint64_t h = 1469598103934665603ull;  // FNV-1a over the fields
    auto mix = [&h](uint64_t v) {
      for (int i = 0; i < 8; ++i) {
        h ^= (v >> (8 * i)) & 0xFFu;
        h *= 1099511628211ull;
      }
    };
    mix((uint64_t)(uint32_t)k.parent);
    mix(k.parent_gen);
    for (int32_t t : k.tokens) mix((uint64_t)(uint32_t)t);
    return (size_t)h;
  }
};

}  // namespace

struct pa_block_manager {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
    uint64_t batch = 0;  // the last append batch that named this sequence
  };
  int32_t num_blocks = 0;
  int32_t block_size = 16;
  // The free list, in order: a doubly linked list over block ids (-1 ends),
  // so a cached block can leave it from the middle.
  std::vector<int32_t> prev, next;
  std::vector<uint8_t> on_free;
  int32_t head = -1, tail = -1, nfree = 0;
  std::vector<int32_t> ref;
  std::vector<uint32_t> gen;                       // times each id was handed out
  std::unordered_map<CacheKey, int32_t, CacheKeyHash> cache;
  std::vector<CacheKey> key_of;                    // a cached block's key
  std::vector<uint8_t> cached;
  std::unordered_map<int64_t, Seq> seqs;
  uint64_t batch_no = 0;       // append batches so far
  std::vector<Seq*> scratch;   // the sequences of the call in progress
  std::mutex mu;

  int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }

  void push_back_free(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    on_free[b] = 1;
    ++nfree;
  }

  void unlink_free(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    on_free[b] = 0;
    --nfree;
  }

  void uncache(int32_t b) {
    if (cached[b]) {
      cache.erase(key_of[b]);
      key_of[b].tokens.clear();
      cached[b] = 0;
    }
  }

  int32_t take() {
    const int32_t b = head;
    unlink_free(b);
    uncache(b);  // handing out a cached block evicts it
    ++gen[b];
    ref[b] = 1;
    return b;
  }

  void drop(int32_t b) {
    if (--ref[b] == 0) push_back_free(b);
  }

  CacheKey key(int32_t parent, const int32_t* toks) const {
    CacheKey k;
    k.parent = parent;
    k.parent_gen = parent >= 0 ? gen[parent] : 0;
    k.tokens.assign(toks, toks + block_size);
    return k;
  }

  // Make the full blocks of s findable (tokens: its ids from the first).
  void register_blocks(const Seq& s, const int32_t* tokens, int64_t n) {
    int32_t parent = -1;
    const int64_t full = std::min<int64_t>(n, s.len) / block_size;
    for (int64_t j = 0; j < full; ++j) {
      const int32_t b = s.blocks[(size_t)j];
      CacheKey k = key(parent, tokens + j * block_size);
      if (!cached[b] && cache.find(k) == cache.end()) {
        key_of[b] = k;
        cache.emplace(std::move(k), b);
        cached[b] = 1;
      }
      parent = b;
    }
  }

  // New blocks (and whether a copy-on-write is needed) for appending n tokens.
  void append_need(const Seq& s, int64_t n, int64_t* new_blocks, bool* cow) const {
    const int64_t L = s.len;
    *cow = n > 0 && L % block_size != 0 && ref[s.blocks[L / block_size]] > 1;
    *new_blocks = blocks_for(L + n) - (int64_t)s.blocks.size();
  }

  // Apply an append whose blocks are known to be available.
  void append_apply(Seq& s, int64_t n, int64_t* slots, int64_t* copies, int32_t* n_copies) {
    int64_t nb;
    bool cow;
    append_need(s, n, &nb, &cow);
    const int64_t L = s.len;
    if (cow) {
      const int32_t old = s.blocks[L / block_size];
      const int32_t fresh = take();
      copies[2 * *n_copies] = old;
      copies[2 * *n_copies + 1] = fresh;
      ++*n_copies;
      --ref[old];  // another table still holds it
      s.blocks[L / block_size] = fresh;
    }
    for (int64_t k = 0; k < nb; ++k) s.blocks.push_back(take());
    for (int64_t pos = L; pos < L + n; ++pos)
      slots[pos - L] = (int64_t)s.blocks[pos / block_size] * block_size + pos % block_size;
    s.len = L + n;
  }
};

namespace {
pa_status bm_fail(pa_status st, const char* msg) {
  return (pa_status)pa::record_error_code((int)st, msg);
}
pa_status bm_ok() { return (pa_status)pa::record_error_code((int)PA_OK, ""); }
}  // namespace

extern "C" {

pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size) {
  if (num_blocks <= 0 || block_size <= 0) {
    pa::record_error_code((int)PA_ERR_INVALID_ARG, "num_blocks and block_size must be > 0");
    return nullptr;
  }
  auto* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  const size_t nb = (size_t)num_blocks;
  bm->prev.assign(nb, -1);
  bm->next.assign(nb, -1);
  bm->on_free.assign(nb, 0);
  bm->ref.assign(nb, 0);
  bm->gen.assign(nb, 0);
  bm->key_of.resize(nb);
  bm->cached.assign(nb, 0);
  for (int32_t b = 0; b < num_blocks; ++b) bm->push_back_free(b);
  return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int32_t pa_bm_num_free(pa_block_manager* bm) {
  if (!bm) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  return bm->nfree;
}

int32_t pa_bm_ref_count(pa_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  return bm->ref[(size_t)block];
}

pa_status pa_bm_allocate(pa_block_manager* bm, int64_t seq_id, int64_t num_tokens) {
  if (!bm || num_tokens < 0) return bm_fail(PA_ERR_INVALID_ARG, "bad manager or token count");
  std::lock_guard<std::mutex> g(bm->mu);
  if (bm->seqs.count(seq_id)) return bm_fail(PA_ERR_INVALID_ARG, "sequence id already present");
  const int64_t need = bm->blocks_for(num_tokens);
  if (need > (int64_t)bm->nfree)
    return bm_fail(PA_ERR_OUT_OF_BLOCKS, "KV cache exhausted: not enough free blocks");
  pa_block_manager::Seq s;
  s.blocks.reserve((size_t)need);
  for (int64_t k = 0; k < need; ++k) s.blocks.push_back(bm->take());
  s.len = num_tokens;
  bm->seqs.emplace(seq_id, std::move(s));
  return bm_ok();
}

pa_status pa_bm_append(pa_block_manager* bm, int64_t seq_id, int64_t n, int64_t* slots_out,
                       int64_t* copies_out, int32_t* n_copies_out) {
  return pa_bm_append_batch(bm, &seq_id, &n, 1, slots_out, copies_out, n_copies_out);
}

pa_status pa_bm_append_batch(pa_block_manager* bm, const int64_t* seq_ids, const int64_t* counts,
                             int32_t n_seqs, int64_t* slots_out, int64_t* copies_out,
                             int32_t* n_copies_out) {
  if (!bm || n_seqs < 0 || (n_seqs > 0 && (!seq_ids || !counts || !n_copies_out)))
    return bm_fail(PA_ERR_INVALID_ARG, "bad manager or null pointer");
  std::lock_guard<std::mutex> g(bm->mu);
  // Check everything first: a batch that does not fit changes nothing.  The
  // appends apply in batch order, so an earlier copy-on-write that leaves a
  // shared block with one holder spares a later one: replay the reference
  // drops while counting.
  int64_t total_blocks = 0, total_slots = 0;
  bool any_cow = false;
  std::unordered_map<int32_t, int32_t> dropped;  // block -> copies-on-write so far
  // Each sequence is looked up once; a stamp per batch finds an id named twice.
  const uint64_t stamp = ++bm->batch_no;
  bm->scratch.clear();
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence id");
    if (it->second.batch == stamp)
      return bm_fail(PA_ERR_INVALID_ARG, "a sequence id appears twice in one batch");
    it->second.batch = stamp;
    bm->scratch.push_back(&it->second);
    if (counts[i] < 0) return bm_fail(PA_ERR_INVALID_ARG, "negative token count");
    const auto& sq = it->second;
    const int64_t L = sq.len;
    bool cow = false;
    if (counts[i] > 0 && L % bm->block_size != 0) {
      const int32_t b = sq.blocks[(size_t)(L / bm->block_size)];
      const auto d = dropped.find(b);
      cow = bm->ref[(size_t)b] - (d == dropped.end() ? 0 : d->second) > 1;
      if (cow) ++dropped[b];
    }
    total_blocks += bm->blocks_for(L + counts[i]) - (int64_t)sq.blocks.size() + (cow ? 1 : 0);
    total_slots += counts[i];
    any_cow = any_cow || cow;
  }
  if (total_slots > 0 && !slots_out) return bm_fail(PA_ERR_INVALID_ARG, "null slots_out");
  if (any_cow && !copies_out) return bm_fail(PA_ERR_INVALID_ARG, "null copies_out");
  if (total_blocks > (int64_t)bm->nfree)
    return bm_fail(PA_ERR_OUT_OF_BLOCKS, "KV cache exhausted: not enough free blocks");
  *n_copies_out = 0;
  int64_t off = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    bm->append_apply(*bm->scratch[(size_t)i], counts[i], slots_out + off, copies_out,
                     n_copies_out);
    off += counts[i];
  }
  return bm_ok();
}

pa_status pa_bm_allocate_cached(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                                int64_t n_tokens, int64_t* n_cached_out) {
  if (!bm || n_tokens < 0 || (n_tokens > 0 && !tokens) || !n_cached_out)
    return bm_fail(PA_ERR_INVALID_ARG, "bad manager, token count or null pointer");
  std::lock_guard<std::mutex> g(bm->mu);
  if (bm->seqs.count(seq_id)) return bm_fail(PA_ERR_INVALID_ARG, "sequence id already present");
  const int32_t bs = bm->block_size;
  const int64_t reusable = n_tokens > 0 ? (n_tokens - 1) / bs : 0;
  std::vector<int32_t> hits;
  int32_t parent = -1;
  for (int64_t j = 0; j < reusable; ++j) {
    auto it = bm->cache.find(bm->key(parent, tokens + j * bs));
    if (it == bm->cache.end()) break;
    hits.push_back(it->second);
    parent = it->second;
  }
  const int64_t need = bm->blocks_for(n_tokens) - (int64_t)hits.size();
  int64_t idle = 0;  // cached blocks sitting on the free list
  for (int32_t b : hits) idle += bm->ref[(size_t)b] == 0 ? 1 : 0;
  if (need > (int64_t)bm->nfree - idle)
    return bm_fail(PA_ERR_OUT_OF_BLOCKS, "KV cache exhausted: not enough free blocks");
  pa_block_manager::Seq s;
  for (int32_t b : hits) {
    if (bm->ref[(size_t)b] == 0) bm->unlink_free(b);
    ++bm->ref[(size_t)b];
    s.blocks.push_back(b);
  }
  for (int64_t k = 0; k < need; ++k) s.blocks.push_back(bm->take());
  s.len = n_tokens;
  bm->register_blocks(s, tokens, n_tokens);
  bm->seqs.emplace(seq_id, std::move(s));
  *n_cached_out = (int64_t)hits.size() * bs;
  return bm_ok();
}

pa_status pa_bm_register(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                         int64_t n_tokens) {
  if (!bm || n_tokens < 0 || (n_tokens > 0 && !tokens))
    return bm_fail(PA_ERR_INVALID_ARG, "bad manager, token count or null pointer");
  std::lock_guard<std::mutex> g(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence id");
  bm->register_blocks(it->second, tokens, n_tokens);
  return bm_ok();
}

pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return bm_fail(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> g(bm->mu);
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return bm_fail(PA_ERR_INVALID_ARG, "unknown parent sequence id");
  if (bm->seqs.count(child)) return bm_fail(PA_ERR_INVALID_ARG, "child sequence id already present");
  pa_block_manager::Seq s = it->second;
  for (int32_t b : s.blocks) ++bm->ref[(size_t)b];
  bm->seqs.emplace(child, std::move(s));
  return bm_ok();
}

pa_status pa_bm_free(pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return bm_fail(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> g(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence id");
  for (int32_t b : it->second.blocks) bm->drop(b);
  bm->seqs.erase(it);
  return bm_ok();
}

pa_status pa_bm_block_tables(pa_block_manager* bm, const int64_t* seq_ids, int32_t n_seqs,
                             int32_t width, int32_t* tables_out, int32_t* lens_out) {
  if (!bm || n_seqs < 0 || width < 0 || (n_seqs > 0 && (!seq_ids || !tables_out || !lens_out)))
    return bm_fail(PA_ERR_INVALID_ARG, "bad manager, size or null pointer");
  std::lock_guard<std::mutex> g(bm->mu);
  bm->scratch.clear();
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence id");
    if ((int64_t)it->second.blocks.size() > width)
      return bm_fail(PA_ERR_INVALID_ARG, "a block table is wider than width");
    if (it->second.len > 0x7FFFFFFFll) return bm_fail(PA_ERR_UNSUPPORTED, "sequence too long");
    bm->scratch.push_back(&it->second);
  }
  for (int32_t i = 0; i < n_seqs; ++i) {
    const auto& s = *bm->scratch[(size_t)i];
    int32_t* row = tables_out + (size_t)i * (size_t)width;
    std::copy(s.blocks.begin(), s.blocks.end(), row);
    std::fill(row + s.blocks.size(), row + width, -1);
    lens_out[i] = (int32_t)s.len;
  }
  return bm_ok();
}

}  // extern "C"
