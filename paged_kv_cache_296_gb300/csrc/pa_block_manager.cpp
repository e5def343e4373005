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
// Every call takes the manager's mutex, so one manager may be driven from
// several host threads.
#include <cstdint>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

struct pa_block_manager {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
  };
  int32_t num_blocks = 0;
  int32_t block_size = 16;
  std::deque<int32_t> free_list;
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Seq> seqs;
  std::mutex mu;

  int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }

  int32_t take() {
    const int32_t b = free_list.front();
    free_list.pop_front();
    ref[b] = 1;
    return b;
  }

  void drop(int32_t b) {
    if (--ref[b] == 0) free_list.push_back(b);
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
  bm->ref.assign((size_t)num_blocks, 0);
  for (int32_t b = 0; b < num_blocks; ++b) bm->free_list.push_back(b);
  return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int32_t pa_bm_num_free(pa_block_manager* bm) {
  if (!bm) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  return (int32_t)bm->free_list.size();
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
  if (need > (int64_t)bm->free_list.size())
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
  std::unordered_set<int64_t> seen;
  std::unordered_map<int32_t, int32_t> dropped;  // block -> copies-on-write so far
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence id");
    if (!seen.insert(seq_ids[i]).second)
      return bm_fail(PA_ERR_INVALID_ARG, "a sequence id appears twice in one batch");
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
  if (total_blocks > (int64_t)bm->free_list.size())
    return bm_fail(PA_ERR_OUT_OF_BLOCKS, "KV cache exhausted: not enough free blocks");
  *n_copies_out = 0;
  int64_t off = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto& s = bm->seqs[seq_ids[i]];
    bm->append_apply(s, counts[i], slots_out + off, copies_out, n_copies_out);
    off += counts[i];
  }
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
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence id");
    if ((int64_t)it->second.blocks.size() > width)
      return bm_fail(PA_ERR_INVALID_ARG, "a block table is wider than width");
    if (it->second.len > 0x7FFFFFFFll) return bm_fail(PA_ERR_UNSUPPORTED, "sequence too long");
  }
  for (int32_t i = 0; i < n_seqs; ++i) {
    const auto& s = bm->seqs[seq_ids[i]];
    int32_t* row = tables_out + (size_t)i * (size_t)width;
    for (int32_t j = 0; j < width; ++j)
      row[j] = j < (int32_t)s.blocks.size() ? s.blocks[(size_t)j] : -1;
    lens_out[i] = (int32_t)s.len;
  }
  return bm_ok();
}

}  // extern "C"
