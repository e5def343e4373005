// pa_find_shared_prefixes: the shared-prefix groups pa_decode_shared reads,
// found from block tables in host memory.
//
// Sequences forked from one prompt (parallel sampling, beam search) hold the
// prompt's physical blocks at the start of their tables ("vLLM GitHub 项目：
// 探索高效 LLM 推理服务", section 二 item 4).  Grouping: by the first table
// entry, in sequence order, at most 32 / G sequences per group (G query heads
// per KV head; the group's members x G query heads are one 32-column MMA
// tile of the decode kernel).  A group's shared length is the number of
// leading entries, within every member's ceil(L / block_size) blocks, that are
// equal in all members' tables.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {
// Records `msg` for pa_last_error() ("" clears it) and returns `st`.
pa_status fail_msg(pa_status st, const char* msg) {
  return static_cast<pa_status>(pa::record_error_code(static_cast<int>(st), msg));
}
}  // namespace

extern "C" pa_status pa_find_shared_prefixes(const int32_t* block_tables,
                                             const int32_t* context_lens, int num_seqs,
                                             int max_blocks_per_seq, int block_size,
                                             int num_q_heads, int num_kv_heads, int min_blocks,
                                             int32_t* group_offsets, int32_t* group_seqs,
                                             int32_t* group_blocks, int32_t* num_groups_out) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
      num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || min_blocks < 0)
    return fail_msg(PA_ERR_INVALID_ARG, "pa_find_shared_prefixes: invalid sizes");
  const int g = num_q_heads / num_kv_heads;
  if (g > pa::kPrefixCols)
    return fail_msg(PA_ERR_UNSUPPORTED, "pa_find_shared_prefixes: too many query heads per KV head");
  if (!num_groups_out || !group_offsets || (num_seqs > 0 && (!block_tables || !context_lens ||
                                                             !group_seqs || !group_blocks)))
    return fail_msg(PA_ERR_INVALID_ARG, "pa_find_shared_prefixes: null pointer argument");
  const int max_members = pa::kPrefixCols / g;
  auto nblk = [&](int i) {
    const long long cap = (long long)max_blocks_per_seq * block_size;
    const long long L = std::min<long long>(std::max(context_lens[i], 0), cap);
    return (int)((L + block_size - 1) / block_size);
  };
  auto row = [&](int i) { return block_tables + (size_t)i * max_blocks_per_seq; };

  // candidates: sequences with at least one block, ordered by first block then index
  std::vector<int> order;
  order.reserve(num_seqs);
  for (int i = 0; i < num_seqs; ++i)
    if (nblk(i) > 0) order.push_back(i);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return row(a)[0] < row(b)[0]; });

  int ng = 0, nm = 0;
  group_offsets[0] = 0;
  for (size_t r0 = 0; r0 < order.size();) {
    size_t r1 = r0 + 1;
    while (r1 < order.size() && row(order[r1])[0] == row(order[r0])[0]) ++r1;
    // the run [r0, r1) starts with the same block; split it into groups
    for (size_t c0 = r0; c0 < r1; c0 += max_members) {
      const size_t c1 = std::min(r1, c0 + max_members);
      if (c1 - c0 < 2) continue;
      const int lead = order[c0];
      int shared = nblk(lead);
      for (size_t k = c0 + 1; k < c1 && shared > 0; ++k) {
        const int s = order[k];
        const int lim = std::min(shared, nblk(s));
        int j = 0;
        while (j < lim && row(s)[j] == row(lead)[j]) ++j;
        shared = j;
      }
      if (shared < std::max(min_blocks, 1)) continue;
      for (size_t k = c0; k < c1; ++k) group_seqs[nm++] = order[k];
      group_blocks[ng] = shared;
      group_offsets[++ng] = nm;
    }
    r0 = r1;
  }
  *num_groups_out = ng;
  return fail_msg(PA_OK, "");
}
