// extern "C" entry points of libpagedattn.so (declared in include/pa.h).
//
// Each entry point validates its arguments on the host, records a message for
// pa_last_error() on failure, and otherwise enqueues kernels on the caller's
// stream.  Nothing here allocates device memory.
#include <cstdarg>
#include <cstdio>
#include <cstdint>
#include <algorithm>
#include <string>

#include <cuda_runtime.h>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

thread_local std::string g_last_error;

constexpr int kBlockSize = 16;
constexpr int kMinPartitionTokens = 512;
constexpr int kMaxPartitionTokens = 8192;
constexpr long long kTargetPairs = 512;
constexpr int kMaxGroup = 8;

pa_status fail(pa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

pa_status ok() {
  g_last_error.clear();
  return PA_OK;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elt_bytes(pa_dtype d) {
  switch (d) {
    case PA_F16:
    case PA_BF16:
      return 2;
    case PA_E4M3:
      return 1;
    case PA_F32:
      return 4;
  }
  return 0;
}

// Whether the stream-K kernel can plan this batch: its per-CTA plan holds
// every sequence and group, and unit counts stay below 2^31.
bool split_fits(int num_seqs, int num_kv_heads, int max_blocks_per_seq, int num_groups) {
  return num_seqs <= pa::kMaxPlanSeqs && num_groups <= pa::kMaxPlanGroups &&
         2 * num_kv_heads <= pa::kMaxSplitCtas &&  // two CTAs per KV head group at least
         ((long long)num_seqs + num_groups) * max_blocks_per_seq * std::max(1, num_kv_heads) <
             (1LL << 31);
}

// Split-KV partition size (tokens), 0 for a balanced split, or -1 when the
// request is invalid.  A request of 0 decides from the batch shape alone (no
// device query, so the host-side sizing calls agree with pa_decode everywhere):
//   * with >= kTargetPairs (sequence, KV head) pairs there are enough CTAs
//     already: no split, except that no partition exceeds kMaxPartitionTokens
//     (bounds the slowest CTA);
//   * otherwise a balanced split (returned as 0): the decode kernel reads the
//     actual context lengths and picks the smallest partition size, at least
//     kMinPartitionTokens, whose partitions over all sequences and KV heads
//     fit in one wave of resident CTAs, so every SM streams from the start to
//     the end and the longest CTA is as short as that allows.
// Measured on GB300: a CTA streams about its ring (64 KB) per loaded memory
// latency (~3.5 us), so a batch of a few long sequences must be split, and a
// split that spills into a second wave leaves a long tail.
int partition_tokens(int num_seqs, int num_kv_heads, int max_blocks_per_seq, int requested) {
  if (requested < 0 || requested % kBlockSize != 0) return -1;
  if (requested > 0) return requested;
  const long long max_tokens = (long long)max_blocks_per_seq * kBlockSize;
  const long long pairs = std::max(1LL, (long long)num_seqs * std::max(1, num_kv_heads));
  if (pairs >= kTargetPairs) {
    return (int)std::max<long long>(kBlockSize, std::min<long long>(max_tokens, kMaxPartitionTokens));
  }
  if (max_tokens <= kMinPartitionTokens) return (int)std::max<long long>(kBlockSize, max_tokens);
  return 0;
}

// Partitions of the grid (per sequence and KV head) for a partition size from
// partition_tokens(); for a balanced split, enough for its smallest size.
int num_partitions(int max_blocks_per_seq, int part_tokens) {
  const long long max_tokens = (long long)max_blocks_per_seq * kBlockSize;
  const long long unit = part_tokens > 0 ? part_tokens : kMinPartitionTokens;
  const long long p = (max_tokens + unit - 1) / unit;
  return (int)(p < 1 ? 1 : p);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Split-KV workspace.  Partitions (given or balanced): partial m, l, O per
// (sequence, query head, partition), then 256 bytes where a balanced split
// records its partition size.  Shared prefixes (the stream-K kernel): "cut"
// partials per (CTA, slot, column) for at most kMaxSplitCtas CTAs of up to
// kMaxSplitHeads KV heads (kPrefixCols columns per head), "whole" partials per
// (sequence, query head) for the prefix and the suffix of group members, and
// the kernel's plan for the merge kernel.
struct WorkspaceLayout {
  size_t m_off, l_off, o_off;              // fixed partitions or cut partials
  size_t wm_off, wl_off, wo_off;           // whole partials (groups only)
  size_t plan_off, total;
  int cut_cols;
};

WorkspaceLayout workspace_layout(int num_seqs, int num_q_heads, int head_size, int nparts,
                                 bool split, int num_groups) {
  WorkspaceLayout w{0, 0, 0, 0, 0, 0, 0, 0, 0};
  size_t rows = 0;
  if (split) {
    w.cut_cols = pa::kMaxSplitHeads * pa::kPrefixCols;
    rows = (size_t)pa::kMaxSplitCtas * 2 * w.cut_cols;
  } else {
    if (nparts <= 1) return w;
    rows = (size_t)num_seqs * num_q_heads * nparts;
  }
  w.m_off = 0;
  w.l_off = align256(rows * sizeof(float));
  w.o_off = w.l_off + align256(rows * sizeof(float));
  size_t end = w.o_off + align256(rows * head_size * sizeof(float));
  if (split) {
    const size_t wrows = 2 * (size_t)num_seqs * num_q_heads;
    w.wm_off = end;
    w.wl_off = w.wm_off + align256(wrows * sizeof(float));
    w.wo_off = w.wl_off + align256(wrows * sizeof(float));
    end = w.wo_off + align256(wrows * head_size * sizeof(float));
  }
  w.plan_off = end;
  const size_t plan_ints =
      split ? (size_t)pa::kPlanHeader + pa::kPlanSeqInts * (size_t)num_seqs : 64;
  w.total = w.plan_off + align256(plan_ints * sizeof(int));
  return w;
}

pa_status check_head_size(int head_size) {
  if (head_size != 64 && head_size != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_size %d is not supported (64 or 128)", head_size);
  return PA_OK;
}

pa_status check_block_size(int block_size) {
  if (block_size != kBlockSize)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d is not supported (16 tokens per block)",
                block_size);
  return PA_OK;
}

pa_status check_pool(int num_blocks, int num_kv_heads) {
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be > 0 (got %d)", num_blocks);
  if ((long long)num_blocks * kBlockSize > 0x7FFFFFFFll)
    return fail(PA_ERR_UNSUPPORTED, "num_blocks %d exceeds 2^31 token rows", num_blocks);
  if (num_kv_heads <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads must be > 0 (got %d)", num_kv_heads);
  return PA_OK;
}

// Shared-prefix groups of one call (device arrays; see pa_decode_shared).
struct Groups {
  const int32_t* offsets;   // [num_groups + 1]
  const int32_t* seqs;      // [offsets[num_groups]]
  const int32_t* blocks;    // [num_groups]
  int num_groups;
};

// Shared by pa_decode, pa_decode_append and their shared-prefix forms (`fn`
// names the caller in messages; `k_new` == NULL means no fused write; `grp` ==
// NULL means no shared-prefix groups).
pa_status decode_impl(const char* fn, void* out, const void* q, const void* k_cache,
                      const void* v_cache, const int32_t* block_tables,
                      const int32_t* context_lens, int num_seqs, int max_blocks_per_seq,
                      int num_blocks, int num_q_heads, int num_kv_heads, int head_size,
                      int block_size, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                      float kv_scale, int partition_size, void* workspace,
                      size_t workspace_bytes, void* stream, const void* k_new,
                      const void* v_new, const int64_t* slot_mapping, int64_t src_token_stride,
                      const Groups* grp) {
  pa_status st;
  if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs must be >= 0 (got %d)", num_seqs);
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "num_seqs %d exceeds 65535", num_seqs);
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be > 0 (got %d)", max_blocks_per_seq);
  if (max_blocks_per_seq > (1 << 26))
    return fail(PA_ERR_UNSUPPORTED, "max_blocks_per_seq %d exceeds 2^26", max_blocks_per_seq);
  if ((st = check_block_size(block_size)) != PA_OK) return st;
  if ((st = check_head_size(head_size)) != PA_OK) return st;
  if ((st = check_pool(num_blocks, num_kv_heads)) != PA_OK) return st;
  if (num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                num_q_heads, num_kv_heads);
  if (num_q_heads / num_kv_heads > kMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "query heads per KV head %d exceeds %d",
                num_q_heads / num_kv_heads, kMaxGroup);
  if (num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads exceeds 65535");
  if (q_dtype != PA_F16 && q_dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "q dtype must be PA_F16 or PA_BF16");
  if (kv_dtype != q_dtype && kv_dtype != PA_E4M3)
    return fail(PA_ERR_UNSUPPORTED, "cache dtype must equal the q dtype or be PA_E4M3");
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(PA_ERR_INVALID_ARG, "scale must be finite");
  if (kv_dtype == PA_E4M3 && (!(kv_scale > 0.f) || kv_scale == INFINITY))
    return fail(PA_ERR_INVALID_ARG, "kv_scale must be finite and > 0 for an E4M3 cache");
  int part;
  int num_groups = 0;
  if (grp && grp->num_groups < 0)
    return fail(PA_ERR_INVALID_ARG, "num_groups must be >= 0 (got %d)", grp->num_groups);
  if (grp && grp->num_groups > 0) {
    num_groups = grp->num_groups;
    if (!split_fits(num_seqs, num_kv_heads, max_blocks_per_seq, num_groups))
      return fail(PA_ERR_UNSUPPORTED,
                  "%s: at most %d sequences and %d groups, and fewer than 2^31 blocks over all "
                  "sequences and KV heads",
                  fn, pa::kMaxPlanSeqs, pa::kMaxPlanGroups);
    if (num_groups > 0 && (!grp->offsets || !grp->seqs || !grp->blocks))
      return fail(PA_ERR_INVALID_ARG, "null group array");
    if ((reinterpret_cast<uintptr_t>(grp->offsets) | reinterpret_cast<uintptr_t>(grp->seqs) |
         reinterpret_cast<uintptr_t>(grp->blocks)) & 3u)
      return fail(PA_ERR_INVALID_ARG, "group arrays must be 4-byte aligned");
    part = 0;  // the shared-prefix (stream-K) kernel serves the groups
  } else {
    part = partition_tokens(num_seqs, num_kv_heads, max_blocks_per_seq, partition_size);
    if (part < 0)
      return fail(PA_ERR_INVALID_ARG,
                  "partition_size must be 0 or a positive multiple of 16 (got %d)", partition_size);
  }
  const int np = num_partitions(max_blocks_per_seq, part);
  if (np > 65535) return fail(PA_ERR_UNSUPPORTED, "too many partitions (%d)", np);
  const bool split = num_groups > 0;  // the shared-prefix kernel
  const WorkspaceLayout ws = workspace_layout(num_seqs, num_q_heads, head_size, np, split, num_groups);
  if (num_seqs == 0) return ok();
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PA_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  const int64_t hkv_d = (int64_t)num_kv_heads * head_size;
  const int64_t src_stride = src_token_stride == 0 ? hkv_d : src_token_stride;
  if (k_new) {
    if (!v_new || !slot_mapping) return fail(PA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(k_new) || !aligned16(v_new))
      return fail(PA_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)
      return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
    if (src_stride < hkv_d || (src_stride * 2) % 16 != 0)
      return fail(PA_ERR_INVALID_ARG,
                  "src_token_stride must be >= num_kv_heads*head_size and a multiple of 16 bytes");
  }
  if (ws.total > 0) {
    if (!workspace || workspace_bytes < ws.total)
      return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", ws.total,
                  workspace ? workspace_bytes : (size_t)0);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(PA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }

  pa::DecodeArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_size = head_size;
  a.q_dtype = (int)q_dtype;
  a.kv_dtype = (int)kv_dtype;
  a.scale = scale;
  a.kv_scale = kv_dtype == PA_E4M3 ? kv_scale : 1.0f;
  a.partition_tokens = part;
  a.min_partition_tokens = (int)kMinPartitionTokens;
  a.num_partitions = np;
  auto* wsb = static_cast<uint8_t*>(workspace);
  auto at = [&](size_t off) { return ws.total ? reinterpret_cast<float*>(wsb + off) : nullptr; };
  a.part_m = split ? nullptr : at(ws.m_off);
  a.part_l = split ? nullptr : at(ws.l_off);
  a.part_o = split ? nullptr : at(ws.o_off);
  a.cut_m = split ? at(ws.m_off) : nullptr;
  a.cut_l = split ? at(ws.l_off) : nullptr;
  a.cut_o = split ? at(ws.o_off) : nullptr;
  a.cut_cols = ws.cut_cols;
  a.whole_m = split ? at(ws.wm_off) : nullptr;
  a.whole_l = split ? at(ws.wl_off) : nullptr;
  a.whole_o = split ? at(ws.wo_off) : nullptr;
  a.plan = ws.total ? reinterpret_cast<int*>(wsb + ws.plan_off) : nullptr;
  a.grp_off = grp && num_groups ? grp->offsets : nullptr;
  a.grp_seq = grp && num_groups ? grp->seqs : nullptr;
  a.grp_blocks = grp && num_groups ? grp->blocks : nullptr;
  a.num_groups = num_groups;
  a.append = k_new != nullptr;
  a.k_new = k_new;
  a.v_new = v_new;
  a.slot_mapping = slot_mapping;
  a.src_stride_bytes = src_stride * 2;
  cudaError_t e = pa::device_status_ptr(&a.status);
  if (e != cudaSuccess) return cuda_fail(e, "status word");

  const char* why = "launch failed";
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kv_dtype == PA_E4M3) {
    e = pa::launch_decode_e4m3(a, s, &why);
  } else if (kv_dtype == PA_BF16) {
    e = pa::launch_decode_bf16(a, s, &why);
  } else {
    e = pa::launch_decode_f16(a, s, &why);
  }
  if (e == cudaErrorInvalidValue) return fail(PA_ERR_CUDA, "%s: %s", fn, why);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

}  // namespace

namespace pa {
int record_error_code(int status, const char* msg) {
  g_last_error = msg;
  return status;
}
}  // namespace pa

extern "C" {

const char* pa_last_error(void) { return g_last_error.c_str(); }

int pa_version(void) { return 120; }

uint32_t pa_device_status(int clear) {
  unsigned* p = nullptr;
  if (pa::device_status_ptr(&p) != cudaSuccess) return 0xFFFFFFFFu;
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return 0xFFFFFFFFu;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return 0xFFFFFFFFu;
  if (clear && cudaMemset(p, 0, sizeof(unsigned)) != cudaSuccess) return 0xFFFFFFFFu;
  return v;
}

pa_status pa_copy_blocks(void* pool, const int64_t* pairs, int64_t n_pairs, int32_t num_blocks,
                         int64_t block_bytes, void* stream) {
  if (n_pairs < 0) return fail(PA_ERR_INVALID_ARG, "n_pairs must be >= 0");
  if (n_pairs == 0) return ok();
  if (n_pairs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 pairs per call");
  if (!pool || !pairs) return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(pool)) return fail(PA_ERR_INVALID_ARG, "pool must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(pairs) & 7u)
    return fail(PA_ERR_INVALID_ARG, "pairs must be 8-byte aligned");
  if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be > 0");
  if (block_bytes <= 0 || block_bytes % 16 != 0)
    return fail(PA_ERR_INVALID_ARG, "block_bytes must be a positive multiple of 16");
  unsigned* status = nullptr;
  cudaError_t e = pa::device_status_ptr(&status);
  if (e != cudaSuccess) return cuda_fail(e, "status word");
  e = pa::launch_copy_blocks(pool, pairs, n_pairs, num_blocks, block_bytes, status,
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pa_copy_blocks");
  return ok();
}

pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens,
                     const int32_t* query_start_loc, int num_seqs, int max_query_len,
                     int max_blocks_per_seq, int num_blocks, int num_q_heads, int num_kv_heads,
                     int head_size, int block_size, float scale, pa_dtype q_dtype,
                     pa_dtype kv_dtype, float kv_scale, void* stream) {
  pa_status st;
  if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs must be >= 0 (got %d)", num_seqs);
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "num_seqs %d exceeds 65535", num_seqs);
  if (max_query_len < 0)
    return fail(PA_ERR_INVALID_ARG, "max_query_len must be >= 0 (got %d)", max_query_len);
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be > 0 (got %d)", max_blocks_per_seq);
  if (max_blocks_per_seq > (1 << 26))
    return fail(PA_ERR_UNSUPPORTED, "max_blocks_per_seq %d exceeds 2^26", max_blocks_per_seq);
  if ((st = check_block_size(block_size)) != PA_OK) return st;
  if ((st = check_head_size(head_size)) != PA_OK) return st;
  if ((st = check_pool(num_blocks, num_kv_heads)) != PA_OK) return st;
  if (num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                num_q_heads, num_kv_heads);
  if (num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads exceeds 65535");
  if (q_dtype != PA_F16 && q_dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "q_dtype must be PA_F16 or PA_BF16");
  if (kv_dtype != q_dtype && kv_dtype != PA_E4M3)
    return fail(PA_ERR_UNSUPPORTED, "kv_dtype must be q_dtype or PA_E4M3");
  if (kv_dtype == PA_E4M3 && (!(kv_scale > 0.f) || kv_scale == INFINITY))
    return fail(PA_ERR_INVALID_ARG, "kv_scale must be finite and > 0 for an E4M3 cache");
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(PA_ERR_INVALID_ARG, "scale must be finite");
  if (num_seqs == 0 || max_query_len == 0) return ok();
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start_loc)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "out, q, k_cache and v_cache must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_start_loc) & 3u))
    return fail(PA_ERR_INVALID_ARG,
                "block_tables, context_lens and query_start_loc must be 4-byte aligned");
  if ((long long)max_query_len * (num_q_heads / num_kv_heads) > 0x7FFFFFFFll)
    return fail(PA_ERR_UNSUPPORTED, "max_query_len too large");
  pa::PrefillArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.query_start_loc = query_start_loc;
  a.num_seqs = num_seqs;
  a.max_query_len = max_query_len;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_size = head_size;
  a.dtype = q_dtype == PA_BF16 ? 1 : 0;
  a.kv_dtype = kv_dtype == PA_E4M3 ? 2 : a.dtype;
  a.kv_scale = kv_dtype == PA_E4M3 ? kv_scale : 1.0f;
  a.scale = scale;
  cudaError_t e = pa::device_status_ptr(&a.status);
  if (e != cudaSuccess) return cuda_fail(e, "status word");
  const char* why = "launch failed";
  e = pa::launch_prefill(a, static_cast<cudaStream_t>(stream), &why);
  if (e == cudaErrorInvalidValue) return fail(PA_ERR_CUDA, "pa_prefill: %s", why);
  if (e != cudaSuccess) return cuda_fail(e, "pa_prefill");
  return ok();
}

pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int64_t n_tokens,
                               int64_t src_token_stride, int num_blocks, int num_kv_heads,
                               int head_size, int block_size, pa_dtype src_dtype,
                               pa_dtype kv_dtype, float kv_scale, void* stream) {
  pa_status st;
  if (n_tokens < 0) return fail(PA_ERR_INVALID_ARG, "n_tokens must be >= 0 (got %lld)", (long long)n_tokens);
  if (n_tokens > 0x7FFFFFFFll) return fail(PA_ERR_UNSUPPORTED, "n_tokens exceeds 2^31-1");
  if ((st = check_block_size(block_size)) != PA_OK) return st;
  if ((st = check_head_size(head_size)) != PA_OK) return st;
  if ((st = check_pool(num_blocks, num_kv_heads)) != PA_OK) return st;
  const int se = elt_bytes(src_dtype), ke = elt_bytes(kv_dtype);
  if (se == 0 || ke == 0) return fail(PA_ERR_INVALID_ARG, "unknown dtype code");
  if (kv_dtype == PA_E4M3) {
    if (src_dtype == PA_E4M3)
      return fail(PA_ERR_UNSUPPORTED, "an E4M3 cache takes f16, bf16 or f32 sources");
    if (!(kv_scale > 0.f) || kv_scale == INFINITY)
      return fail(PA_ERR_INVALID_ARG, "kv_scale must be finite and > 0 for an E4M3 cache");
  } else if (kv_dtype == PA_F32) {
    return fail(PA_ERR_UNSUPPORTED, "an f32 cache is not supported");
  } else if (src_dtype != kv_dtype) {
    return fail(PA_ERR_UNSUPPORTED, "a 16-bit cache takes sources of its own dtype");
  }
  const int64_t hkv_d = (int64_t)num_kv_heads * head_size;
  if (hkv_d > (1 << 24)) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads*head_size too large");
  const int64_t stride = src_token_stride == 0 ? hkv_d : src_token_stride;
  if (stride < hkv_d)
    return fail(PA_ERR_INVALID_ARG, "src_token_stride %lld is smaller than num_kv_heads*head_size",
                (long long)src_token_stride);
  if ((stride * se) % 16 != 0)
    return fail(PA_ERR_INVALID_ARG, "src_token_stride must be a multiple of 16 bytes");
  if (n_tokens == 0) return ok();
  if (!k || !v || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "k, v, k_cache and v_cache must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
    return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  cudaError_t e = pa::launch_reshape_and_cache(
      k, v, k_cache, v_cache, slot_mapping, n_tokens, stride * se,
      (int64_t)num_blocks * kBlockSize, (int)hkv_d, (int)src_dtype, (int)kv_dtype, kv_scale,
      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pa_reshape_and_cache launch");
  return ok();
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                                int max_blocks_per_seq, int block_size, int partition_size) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
      block_size != kBlockSize || (head_size != 64 && head_size != 128)) {
    fail(PA_ERR_INVALID_ARG, "invalid arguments to pa_decode_workspace_size");
    return 0;
  }
  const int part = partition_tokens(num_seqs, num_kv_heads, max_blocks_per_seq, partition_size);
  if (part < 0) {
    fail(PA_ERR_INVALID_ARG, "partition_size must be 0 or a positive multiple of 16");
    return 0;
  }
  const int np = num_partitions(max_blocks_per_seq, part);
  return workspace_layout(num_seqs, num_q_heads, head_size, np, false, 0).total;
}

size_t pa_decode_shared_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_size, int max_blocks_per_seq, int block_size,
                                       int num_groups) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
      block_size != kBlockSize || (head_size != 64 && head_size != 128) || num_groups < 0 ||
      !split_fits(num_seqs, num_kv_heads, max_blocks_per_seq, num_groups)) {
    fail(PA_ERR_INVALID_ARG, "invalid arguments to pa_decode_shared_workspace_size");
    return 0;
  }
  if (num_groups == 0)  // the call is pa_decode's library choice
    return pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                    max_blocks_per_seq, block_size, 0);
  return workspace_layout(num_seqs, num_q_heads, head_size, 0, true, num_groups).total;
}

int pa_decode_partition_size(int num_seqs, int num_kv_heads, int max_blocks_per_seq,
                             int block_size, int partition_size) {
  if (block_size != kBlockSize || max_blocks_per_seq <= 0) return -1;
  return partition_tokens(num_seqs, num_kv_heads, max_blocks_per_seq, partition_size);
}

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                    int max_blocks_per_seq, int num_blocks, int num_q_heads, int num_kv_heads,
                    int head_size, int block_size, float scale, pa_dtype q_dtype,
                    pa_dtype kv_dtype, float kv_scale, int partition_size, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return decode_impl("pa_decode", out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_blocks, num_q_heads, num_kv_heads, head_size,
                     block_size, scale, q_dtype, kv_dtype, kv_scale, partition_size, workspace,
                     workspace_bytes, stream, nullptr, nullptr, nullptr, 0, nullptr);
}

pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, int64_t src_token_stride, void* k_cache,
                           void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, int num_seqs, int max_blocks_per_seq,
                           int num_blocks, int num_q_heads, int num_kv_heads, int head_size,
                           int block_size, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                           float kv_scale, int partition_size, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping))
    return fail(PA_ERR_INVALID_ARG, "pa_decode_append: k_new, v_new and slot_mapping are required");
  return decode_impl("pa_decode_append", out, q, k_cache, v_cache, block_tables, context_lens,
                     num_seqs, max_blocks_per_seq, num_blocks, num_q_heads, num_kv_heads,
                     head_size, block_size, scale, q_dtype, kv_dtype, kv_scale, partition_size,
                     workspace, workspace_bytes, stream, k_new, v_new, slot_mapping,
                     src_token_stride, nullptr);
}

pa_status pa_decode_shared(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                           int max_blocks_per_seq, int num_blocks, int num_q_heads,
                           int num_kv_heads, int head_size, int block_size, float scale,
                           pa_dtype q_dtype, pa_dtype kv_dtype, float kv_scale,
                           const int32_t* group_offsets, const int32_t* group_seqs,
                           const int32_t* group_blocks, int num_groups, void* workspace,
                           size_t workspace_bytes, void* stream) {
  const Groups grp{group_offsets, group_seqs, group_blocks, num_groups};
  return decode_impl("pa_decode_shared", out, q, k_cache, v_cache, block_tables, context_lens,
                     num_seqs, max_blocks_per_seq, num_blocks, num_q_heads, num_kv_heads,
                     head_size, block_size, scale, q_dtype, kv_dtype, kv_scale, 0, workspace,
                     workspace_bytes, stream, nullptr, nullptr, nullptr, 0, &grp);
}

pa_status pa_decode_append_shared(void* out, const void* q, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, int64_t src_token_stride,
                                  void* k_cache, void* v_cache, const int32_t* block_tables,
                                  const int32_t* context_lens, int num_seqs,
                                  int max_blocks_per_seq, int num_blocks, int num_q_heads,
                                  int num_kv_heads, int head_size, int block_size, float scale,
                                  pa_dtype q_dtype, pa_dtype kv_dtype, float kv_scale,
                                  const int32_t* group_offsets, const int32_t* group_seqs,
                                  const int32_t* group_blocks, int num_groups, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping))
    return fail(PA_ERR_INVALID_ARG,
                "pa_decode_append_shared: k_new, v_new and slot_mapping are required");
  const Groups grp{group_offsets, group_seqs, group_blocks, num_groups};
  return decode_impl("pa_decode_append_shared", out, q, k_cache, v_cache, block_tables,
                     context_lens, num_seqs, max_blocks_per_seq, num_blocks, num_q_heads,
                     num_kv_heads, head_size, block_size, scale, q_dtype, kv_dtype, kv_scale, 0,
                     workspace, workspace_bytes, stream, k_new, v_new, slot_mapping,
                     src_token_stride, &grp);
}

pa_status pa_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens,
                       const int64_t* cu_seqlens, int num_seqs, int max_blocks_per_seq,
                       int num_blocks, int num_kv_heads, int head_size, int block_size,
                       pa_dtype kv_dtype, void* stream) {
  pa_status st;
  if (num_seqs < 0 || num_seqs > 65535)
    return fail(PA_ERR_INVALID_ARG, "num_seqs must be in [0, 65535] (got %d)", num_seqs);
  if (max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be > 0 (got %d)", max_blocks_per_seq);
  if (max_blocks_per_seq > (1 << 26))
    return fail(PA_ERR_UNSUPPORTED, "max_blocks_per_seq %d exceeds 2^26", max_blocks_per_seq);
  if ((st = check_block_size(block_size)) != PA_OK) return st;
  if ((st = check_head_size(head_size)) != PA_OK) return st;
  if ((st = check_pool(num_blocks, num_kv_heads)) != PA_OK) return st;
  const int ke = elt_bytes(kv_dtype);
  if (ke == 0 || kv_dtype == PA_F32) return fail(PA_ERR_UNSUPPORTED, "unsupported cache dtype");
  if (num_seqs == 0) return ok();
  if (!k_out || !v_out || !k_cache || !v_cache || !block_tables || !context_lens || !cu_seqlens)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(k_out) || !aligned16(v_out) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID_ARG, "k_out, v_out, k_cache and v_cache must be 16-byte aligned");
  const long long row = (long long)num_kv_heads * head_size * ke;
  if (row > 0x7FFFFFFF) return fail(PA_ERR_UNSUPPORTED, "row too large");
  cudaError_t e = pa::launch_gather_kv(k_out, v_out, k_cache, v_cache, block_tables, context_lens,
                                       cu_seqlens, num_seqs, max_blocks_per_seq, num_blocks,
                                       (int)row, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pa_gather_kv launch");
  return ok();
}

pa_status pa_check_tables(const int32_t* block_tables, const int32_t* context_lens,
                          const int64_t* slot_mapping, int64_t n_tokens, int num_seqs,
                          int max_blocks_per_seq, int num_blocks, int block_size,
                          int32_t* counts_dev, int32_t* counts_host, void* stream) {
  if (num_seqs < 0 || n_tokens < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
      block_size <= 0)
    return fail(PA_ERR_INVALID_ARG, "invalid sizes for pa_check_tables");
  if (!counts_dev) return fail(PA_ERR_INVALID_ARG, "counts_dev is required");
  if ((num_seqs > 0 && (!block_tables || !context_lens)) || (n_tokens > 0 && !slot_mapping))
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = pa::launch_check_tables(block_tables, context_lens, slot_mapping, n_tokens,
                                          num_seqs, max_blocks_per_seq, num_blocks, block_size,
                                          counts_dev, s);
  if (e != cudaSuccess) return cuda_fail(e, "pa_check_tables launch");
  if (!counts_host) return ok();
  e = cudaMemcpyAsync(counts_host, counts_dev, 3 * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "pa_check_tables readback");
  if (counts_host[0] || counts_host[1] || counts_host[2])
    return fail(PA_ERR_BAD_INDEX,
                "bad indices: %d context lengths, %d block-table entries, %d slots out of range",
                counts_host[0], counts_host[1], counts_host[2]);
  return ok();
}

}  // extern "C"
