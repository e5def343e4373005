/*
 * pa.h -- C ABI of the GB300 paged-KV-cache decode library (libpagedattn.so).
 *
 * The library implements the data-parallel hot path of a paged KV cache:
 * the per-step write of new keys/values into a pool of fixed-size blocks and
 * single-query ("decode") attention for every running sequence, reaching its
 * keys/values through a per-sequence block table.
 *
 * Sources: "vLLM 部署深度指南" (section PagedAttention 方案: 16 tokens per
 * block and the logical-view / block-table figure; section 代码层面理解: the
 * preallocated pool [num_blocks, block_size, 2, num_heads, head_size],
 * allocate() and append_kv()); "vLLM GitHub 项目：探索高效 LLM 推理服务"
 * (section 二: the block table maps logical to physical blocks, physical
 * blocks need not be contiguous, several tables may point at one block;
 * decode is memory-bandwidth bound).
 *
 * ---------------------------------------------------------------- conventions
 * Pool layout.  One tensor [num_blocks, block_size, 2, num_kv_heads, head_size]
 * of the cache dtype.  Index 2 selects K (0) or V (1).  `k_cache` is the
 * address of element (0, 0, 0, 0, 0) and `v_cache` of (0, 0, 1, 0, 0); both
 * views share token stride 2*num_kv_heads*head_size elements and block stride
 * block_size times that.  Element (blk, t, h, d) of the K view is at
 *   k_cache + ((blk*block_size + t) * 2*num_kv_heads + h) * head_size + d.
 * A flat slot s names token row s = blk*block_size + t of the pool.
 *
 * Memory.  Every pointer argument is device memory owned by the caller
 * (except where a parameter says "host"), 16-byte aligned unless stated.  The
 * library never allocates, frees or keeps a reference past the call.
 *
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 * Compute calls only enqueue work and return; results are visible once the
 * stream reaches them.  No compute call synchronises.
 *
 * Errors.  Every entry point validates its scalar arguments and pointer
 * alignment on the host before launching anything, and returns a pa_status.
 * On error nothing is enqueued and pa_last_error() describes the problem.
 * Launch failures reported by the CUDA runtime return PA_ERR_CUDA.  Index
 * values inside device arrays (block ids, slots, lengths) are not checked by
 * the compute calls: out-of-range block ids read zeros and out-of-range slots
 * are skipped, so no access leaves the pool, but the result is then
 * meaningless.  pa_check_tables() validates them on request.
 *
 * Supported values: block_size == 16; head_size in {64, 128};
 * num_q_heads % num_kv_heads == 0 with 1 <= num_q_heads/num_kv_heads <= 8;
 * q/out dtype PA_F16 or PA_BF16; cache dtype equal to the q dtype, or
 * PA_E4M3 with either q dtype.  Others return PA_ERR_UNSUPPORTED.
 *
 * Determinism: identical inputs give bit-identical outputs.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  PA_F32 is accepted only as the source of a PA_E4M3 write. */
typedef enum {
  PA_F16 = 0,  /* IEEE binary16 */
  PA_BF16 = 1, /* bfloat16 */
  PA_E4M3 = 2, /* OCP 8-bit float E4M3 (bias 7, max 448, NaN 0x7F/0xFF) */
  PA_F32 = 3   /* IEEE binary32 */
} pa_dtype;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misalignment, bad combination */
  PA_ERR_UNSUPPORTED = 2, /* a shape or dtype outside the supported set above */
  PA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than pa_decode_workspace_size() */
  PA_ERR_CUDA = 4,        /* the CUDA runtime or driver reported an error */
  PA_ERR_BAD_INDEX = 5,   /* pa_check_tables() found out-of-range indices */
  PA_ERR_OUT_OF_BLOCKS = 6 /* the block manager has too few free blocks (nothing changed) */
} pa_status;

/*
 * pa_reshape_and_cache -- write one step's new keys and values into the pool.
 *
 * Defined by append_kv() ("vLLM 部署深度指南", section 代码层面理解: write the new
 * token's K/V into its physical block) with the slot naming that block and
 * the offset inside it (section PagedAttention 方案, logical-view figure).
 *
 * For every token n with 0 <= slot_mapping[n] < num_blocks*block_size:
 *   pool[s / block_size, s % block_size, 0, :, :] = enc(k[n])
 *   pool[s / block_size, s % block_size, 1, :, :] = enc(v[n])
 * Tokens with slot_mapping[n] < 0 (padding) or past the pool are skipped.
 *
 * k, v          [n_tokens, num_kv_heads, head_size] of src_dtype; token n
 *               starts at element n*src_token_stride (0 = num_kv_heads*head_size,
 *               i.e. contiguous).  The stride in bytes must be a multiple of 16.
 * k_cache, v_cache  the pool's K and V views (see conventions), kv_dtype.
 * slot_mapping  int64 [n_tokens].
 * kv_dtype == src_dtype (PA_F16/PA_BF16): the element bits are copied.
 * kv_dtype == PA_E4M3 (src PA_F16, PA_BF16 or PA_F32): each element becomes
 *   e4m3_rn_satfinite(float32(x) / kv_scale), one IEEE float32 division and
 *   one round-to-nearest-even to E4M3 saturating at +-448 (NaN stays NaN).
 *   kv_scale must be finite and > 0; it is ignored for 16-bit caches.
 * Distinct tokens must name distinct slots (the last writer is unspecified).
 */
pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int64_t n_tokens,
                               int64_t src_token_stride, int num_blocks, int num_kv_heads,
                               int head_size, int block_size, pa_dtype src_dtype,
                               pa_dtype kv_dtype, float kv_scale, void* stream);

/*
 * pa_decode -- single-query attention for every sequence through its block table.
 *
 * Paging changes only where K/V live, so the result is standard attention
 * ("vLLM GitHub 项目…", section 二; "vLLM 部署深度指南", section PagedAttention 方案):
 * for sequence i with L = context_lens[i] and query head h (G = num_q_heads /
 * num_kv_heads, KV head h / G),
 *   K_i[j] = pool[block_tables[i, j / 16], j % 16, 0, h / G, :]   (j < L)
 *   out[i, h, :] = softmax(scale * q[i, h, :] . K_i^T) . V_i
 * with K/V dequantised as code * kv_scale for a PA_E4M3 cache.  L == 0 gives
 * zeros.  context_lens count every cached token, including one written this
 * step by pa_reshape_and_cache (which must be enqueued first).
 *
 * out, q        [num_seqs, num_q_heads, head_size] of q_dtype, contiguous.
 * block_tables  int32 [num_seqs, max_blocks_per_seq], row-major; entries past
 *               ceil(L / 16) are never read.
 * context_lens  int32 [num_seqs], 0 <= L <= max_blocks_per_seq * 16 (a larger L
 *               is cut to max_blocks_per_seq * 16, so no table entry past the
 *               row is read; pa_check_tables reports such lengths).
 * num_blocks    number of blocks in the pool (bounds the loads).
 * partition_size  tokens per split-KV partition: 0 = library choice (see
 *               pa_decode_partition_size), else a multiple of 16.  Sequences longer than one partition are
 *               processed as partitions whose fp32 partial results are merged
 *               by log-sum-exp (a second kernel on the same stream).
 * workspace     device scratch of at least pa_decode_workspace_size(...) bytes
 *               (256-byte aligned) for those partials; may be NULL when that
 *               size is 0.  Its contents need no initialisation.  Calls that
 *               share a workspace must not overlap in time.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                    int max_blocks_per_seq, int num_blocks, int num_q_heads, int num_kv_heads,
                    int head_size, int block_size, float scale, pa_dtype q_dtype,
                    pa_dtype kv_dtype, float kv_scale, int partition_size, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * pa_decode_append -- one decode step in one launch: append each sequence's
 * new token to the pool, then attend through the block table.
 *
 * The same result as pa_reshape_and_cache over the step's tokens followed by
 * pa_decode (bit for bit: the same writes and the same attention arithmetic),
 * for the decode case of "vLLM 部署深度指南", section 代码层面理解, where
 * append_kv adds one token per running sequence and attention follows.
 * Token i belongs to sequence i and is its last cached token (position
 * context_lens[i] - 1, already counted in context_lens[i]); slot_mapping[i] is
 * its slot (< 0: no write).  The CTA that attends over that position writes
 * the token (head by head) before loading it.
 *
 * k_new, v_new  [num_seqs, num_kv_heads, head_size] of q_dtype; token i starts
 *               at element i*src_token_stride (0 = contiguous); the stride in
 *               bytes must be a multiple of 16.  A PA_E4M3 cache quantises them
 *               with kv_scale exactly as pa_reshape_and_cache does.
 * Every other argument is pa_decode's.  A slot that is not the one the block
 * table gives position L - 1 leaves the result undefined (no access leaves
 * the pool).
 */
pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, int64_t src_token_stride, void* k_cache,
                           void* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, int num_seqs, int max_blocks_per_seq,
                           int num_blocks, int num_q_heads, int num_kv_heads, int head_size,
                           int block_size, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                           float kv_scale, int partition_size, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * pa_decode_shared -- pa_decode for a batch in which groups of sequences share
 * the leading blocks of their block tables: each shared block is read once
 * per call for all its sequences.
 *
 * Parallel sampling and beam search fork several sequences from one prompt;
 * their block tables point at the same physical blocks for the prompt, and
 * block-level sharing avoids storing (and, here, reading) that prefix again
 * ("vLLM GitHub 项目：探索高效 LLM 推理服务", section 二 item 4; "vLLM 部署深度指南",
 * section 代码层面理解, where several sequences' tables may name one block).
 * The result is exactly what pa_decode defines for the same tables (up to
 * fp32 rounding order): sharing changes only which CTA reads a block.
 *
 * Groups, as device int32 arrays in CSR form: group g's members are the
 * sequence indices group_seqs[group_offsets[g] .. group_offsets[g+1]), and
 * each member's table holds the same physical block at every entry j <
 * group_blocks[g].  group_offsets has num_groups + 1 non-decreasing entries,
 * group_offsets[0] = 0, and group_seqs has group_offsets[num_groups] entries.
 * A sequence belongs to at most one group.  A member shorter than its group's
 * shared blocks is handled exactly (it attends only its own tokens).  Per KV
 * head, a group's members times the query heads per KV head are served as the
 * columns of one tensor-core tile: at most 32 / (num_q_heads / num_kv_heads)
 * members share; members past that count are decoded as unshared sequences.
 * pa_find_shared_prefixes() builds the arrays from the tables.
 *
 * Limits: num_seqs <= 1024, num_groups <= 1024, and num_seqs *
 * max_blocks_per_seq * num_kv_heads < 2^31 (else PA_ERR_UNSUPPORTED).
 * The split of the work over CTAs is the library's (partition_size has no
 * counterpart).  workspace: at least pa_decode_shared_workspace_size(...)
 * bytes, 256-byte aligned, no initialisation needed.  Every other argument
 * is pa_decode's.
 */
pa_status pa_decode_shared(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                           int max_blocks_per_seq, int num_blocks, int num_q_heads,
                           int num_kv_heads, int head_size, int block_size, float scale,
                           pa_dtype q_dtype, pa_dtype kv_dtype, float kv_scale,
                           const int32_t* group_offsets, const int32_t* group_seqs,
                           const int32_t* group_blocks, int num_groups, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * pa_decode_append_shared -- pa_decode_append with shared-prefix groups: one
 * launch appends each sequence's new token and attends as pa_decode_shared.
 * A new token must land in a block that no other sequence of the batch reads
 * (copy-on-write gives a forked sequence a private block before it writes);
 * a member whose new token falls inside its group's shared blocks is not
 * written.  Arguments: pa_decode_append's plus the group arrays.
 */
pa_status pa_decode_append_shared(void* out, const void* q, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, int64_t src_token_stride,
                                  void* k_cache, void* v_cache, const int32_t* block_tables,
                                  const int32_t* context_lens, int num_seqs,
                                  int max_blocks_per_seq, int num_blocks, int num_q_heads,
                                  int num_kv_heads, int head_size, int block_size, float scale,
                                  pa_dtype q_dtype, pa_dtype kv_dtype, float kv_scale,
                                  const int32_t* group_offsets, const int32_t* group_seqs,
                                  const int32_t* group_blocks, int num_groups, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * pa_decode_shared_workspace_size -- bytes of workspace pa_decode_shared and
 * pa_decode_append_shared need (host only; 0 with pa_last_error() set for
 * invalid arguments).
 */
size_t pa_decode_shared_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_size, int max_blocks_per_seq, int block_size,
                                       int num_groups);

/*
 * pa_find_shared_prefixes -- build pa_decode_shared's group arrays from block
 * tables held in HOST memory (host only, no GPU).
 *
 * Sequences whose tables start with the same physical block are grouped (in
 * index order, at most 32 / (num_q_heads / num_kv_heads) per group); a group's
 * shared length is the number of leading entries, within every member's
 * ceil(L / block_size) blocks, on which all members' tables agree.  Groups of
 * one sequence, or sharing fewer than min_blocks blocks, are dropped.
 * block_tables int32 [num_seqs, max_blocks_per_seq] and context_lens int32
 * [num_seqs] are host arrays; the outputs are host arrays with room for
 * num_seqs + 1 (group_offsets) and num_seqs (group_seqs, group_blocks)
 * entries; *num_groups_out receives the group count.
 */
pa_status pa_find_shared_prefixes(const int32_t* block_tables, const int32_t* context_lens,
                                  int num_seqs, int max_blocks_per_seq, int block_size,
                                  int num_q_heads, int num_kv_heads, int min_blocks,
                                  int32_t* group_offsets, int32_t* group_seqs,
                                  int32_t* group_blocks, int32_t* num_groups_out);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call: it exists for callers with no
 * device allocator of their own (a plugin or extension that its host runtime
 * hands only input and output buffers), or that must not allocate while they
 * serve (cudaMalloc can synchronise the device and carves up a memory budget
 * fixed in advance).  It computes exactly what pa_decode computes, with the
 * same arguments minus the workspace.  The caller still passes every input
 * and output.
 *
 * Scratch: the split-KV partials live in one array compiled into the library,
 * PA_DECODE_NOALLOC_SCRATCH_BYTES (64 MiB) per device.  It is reserved on each
 * device whose context loads it and is held until the process exits.  The call
 * itself allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before capturing any stream on that device.
 * Limit: if these sizes need more scratch than the array holds
 * (pa_decode_workspace_size(...) > PA_DECODE_NOALLOC_SCRATCH_BYTES) the call
 * returns PA_ERR_WORKSPACE and enqueues nothing; a larger partition_size needs
 * less scratch.
 * Sharing: every call on a device uses the same array, which keeps whatever
 * the last call left there.  Nothing in it has to start at zero (each partial
 * the merge reads is written earlier in the same call), but calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race on
 * it.  Serialise them, for example by issuing them on one stream.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            int num_seqs, int max_blocks_per_seq, int num_blocks,
                            int num_q_heads, int num_kv_heads, int head_size, int block_size,
                            float scale, pa_dtype q_dtype, pa_dtype kv_dtype, float kv_scale,
                            int partition_size, void* stream);

/*
 * pa_prefill -- causal multi-query attention over the paged pool: a prefill
 * (or a chunk of one) for every sequence of the batch.
 *
 * The pages schedule prefill steps beside decode steps ("vLLM 部署深度指南",
 * section Continuous Batching, the scheduler sketch) and leave the attention
 * itself to the plainest reading, causal self-attention: sequence i has
 * L = context_lens[i] cached tokens, of which its n = query_start_loc[i+1] -
 * query_start_loc[i] query tokens are the last n (positions L-n .. L-1, their
 * K/V already written by pa_reshape_and_cache); the query at position p and
 * query head h (KV head h / G, G = num_q_heads / num_kv_heads) gives
 *   out[r, h, :] = softmax(scale * q[r, h, :] . K_i[0..p]^T) . V_i[0..p]
 * for r = query_start_loc[i] + (p - (L - n)), with K_i / V_i read through the
 * block table as in pa_decode.  A chunk of one token per sequence is a decode
 * step.
 *
 * out, q           [T, num_q_heads, head_size] of q_dtype, T = query_start_loc[num_seqs];
 *                  16-byte aligned, contiguous.
 * query_start_loc  int32 [num_seqs + 1], non-decreasing, query_start_loc[0] = 0.
 * max_query_len    >= every n (sizes the grid; the kernel checks it).
 * block_tables, context_lens, num_blocks  as for pa_decode (n <= L <= max_blocks_per_seq * 16).
 * q_dtype          PA_F16 or PA_BF16 (q and out).
 * kv_dtype         q_dtype, or PA_E4M3: the cache holds codes whose values are
 *                  code * kv_scale (kv_scale finite and > 0, else PA_ERR_INVALID_ARG;
 *                  ignored for a 16-bit cache).  Over an E4M3 cache the MMAs run in
 *                  f16: the codes are exact in f16, bf16 queries are rounded to f16
 *                  (exact for magnitudes in [2^-14, 65504], saturated above), and
 *                  kv_scale multiplies the logits and the output once each.
 * Rows of sequences whose n exceeds L or max_query_len are not written and the
 * device status bit 2 is raised (pa_device_status).  Asynchronous on `stream`;
 * no workspace.
 */
pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens,
                     const int32_t* query_start_loc, int num_seqs, int max_query_len,
                     int max_blocks_per_seq, int num_blocks, int num_q_heads, int num_kv_heads,
                     int head_size, int block_size, float scale, pa_dtype q_dtype,
                     pa_dtype kv_dtype, float kv_scale, void* stream);

/*
 * pa_decode_workspace_size -- bytes of workspace pa_decode needs for these
 * arguments (0 when no sequence can span more than one partition).  Host only;
 * returns 0 and sets pa_last_error() for invalid arguments.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                                int max_blocks_per_seq, int block_size, int partition_size);

/*
 * pa_decode_partition_size -- the partition size pa_decode uses when given
 * partition_size.  A positive request is used as given.  0 asks for the
 * library's choice, made from the batch shape: with num_seqs*num_kv_heads >=
 * 512 no split (partitions capped at 8192 tokens; a sequence no longer than
 * 512 tokens is never split either); otherwise a stream-K split, returned as
 * 0: the decode kernel reads the context lengths and gives each CTA of one
 * wave of resident CTAs on this GPU an equal range (at least 512 tokens) of
 * the batch's (sequence, KV head, block) units, a range crossing from one
 * sequence into the next where it ends.
 * Host only; -1 on invalid input.
 */
int pa_decode_partition_size(int num_seqs, int num_kv_heads, int max_blocks_per_seq,
                             int block_size, int partition_size);

/*
 * pa_gather_kv -- copy each sequence's cached K and V, in token order, into
 * contiguous buffers: the block-table gather alone, bit for bit.
 *
 * Logical token j of sequence i is pool row block_tables[i, j/16]*16 + j%16
 * ("vLLM 部署深度指南", section PagedAttention 方案, logical-view figure).
 *   k_out[cu_seqlens[i] + j, :, :] = pool[block_tables[i, j/16], j%16, 0, :, :]
 *   v_out[...]                      = pool[...,                        1, :, :]
 * k_out, v_out  [cu_seqlens[num_seqs], num_kv_heads, head_size] of kv_dtype.
 * cu_seqlens    int64 [num_seqs + 1] output row offsets (device); sequence i
 *               fills rows [cu_seqlens[i], cu_seqlens[i] + context_lens[i]).
 * Rows whose block id is out of range are left unwritten.
 */
pa_status pa_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens,
                       const int64_t* cu_seqlens, int num_seqs, int max_blocks_per_seq,
                       int num_blocks, int num_kv_heads, int head_size, int block_size,
                       pa_dtype kv_dtype, void* stream);

/*
 * pa_check_tables -- validate the index arrays of one step (not on the hot path).
 *
 * Counts into counts_dev (int32 [3], device, overwritten):
 *   [0] sequences with context_lens[i] < 0 or > max_blocks_per_seq*block_size;
 *   [1] table entries j < ceil(L_i / block_size) outside [0, num_blocks), over
 *       the sequences whose length passed check [0];
 *   [2] slot_mapping entries >= num_blocks*block_size (negative = padding, fine).
 * slot_mapping may be NULL when n_tokens == 0.  If counts_host (int32 [3],
 * host) is non-NULL the call synchronises the stream, copies the counts there
 * and returns PA_ERR_BAD_INDEX when any is non-zero; otherwise it only
 * enqueues the check.
 */
pa_status pa_check_tables(const int32_t* block_tables, const int32_t* context_lens,
                          const int64_t* slot_mapping, int64_t n_tokens, int num_seqs,
                          int max_blocks_per_seq, int num_blocks, int block_size,
                          int32_t* counts_dev, int32_t* counts_host, void* stream);

/*
 * pa_device_status -- error bits raised by kernels on the current device
 * instead of trapping (1 = a bounded wait inside a kernel timed out and the
 * kernel returned early; its outputs are then invalid; 2 = pa_prefill met a
 * sequence whose query count exceeds its length or max_query_len; 4 =
 * pa_copy_blocks skipped a pair naming a block outside the pool).  Synchronises the
 * device.  `clear` != 0 resets the bits.  Returns 0xFFFFFFFF if the status
 * word cannot be read.
 */
uint32_t pa_device_status(int clear);

/*
 * ---------------------------------------------------------------- block manager
 *
 * pa_bm_* -- the host-side allocator of the pool's physical blocks (native
 * C++; no GPU needed).  It follows the pages' KV cache sketch ("vLLM 部署深度指南",
 * section 代码层面理解; "vLLM GitHub 项目…", section 二 items 1 and 4, section 三
 * item 1): the free list starts as every block id in increasing order and
 * blocks are taken from its front; a sequence of n tokens holds ceil(n /
 * block_size) blocks and takes a new block when a token falls past its last
 * one; too few free blocks is PA_ERR_OUT_OF_BLOCKS (the pages' OOMError), and
 * the failed call changes nothing.  Sequences may share blocks (pa_bm_fork,
 * for parallel sampling / beam search); blocks are reference counted and go
 * to the back of the free list, in table order, when the last table lets go.
 * An append whose first token lands in a partially filled block that another
 * table also holds first moves the sequence to a private copy: it takes a new
 * block and returns the (src, dst) pair, which the caller copies on the GPU
 * (pa_copy_blocks) before writing the new tokens (pa_reshape_and_cache at the
 * returned slots).  Sequence ids are arbitrary int64 keys.  Every call locks
 * the manager.  Errors set pa_last_error().
 */
typedef struct pa_block_manager pa_block_manager;

/* A manager of num_blocks blocks of block_size tokens; NULL on bad arguments. */
pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size);
void pa_bm_destroy(pa_block_manager* bm);

/* Free blocks (-1 for a NULL manager); reference count of one block (-1 if out of range). */
int32_t pa_bm_num_free(pa_block_manager* bm);
int32_t pa_bm_ref_count(pa_block_manager* bm, int32_t block);

/* A new sequence already holding num_tokens tokens (a prompt): ceil(n / block_size) blocks. */
pa_status pa_bm_allocate(pa_block_manager* bm, int64_t seq_id, int64_t num_tokens);

/*
 * pa_bm_append_batch -- reserve counts[i] new tokens at the end of sequence
 * seq_ids[i] (distinct ids), all or nothing.  slots_out (int64, sum(counts)
 * entries, in batch order) receives each new token's slot block*block_size +
 * offset, the slot_mapping of pa_reshape_and_cache; copies_out (int64 pairs,
 * room for n_seqs pairs) receives the copy-on-write (src, dst) block pairs
 * and *n_copies_out their number.
 */
pa_status pa_bm_append_batch(pa_block_manager* bm, const int64_t* seq_ids, const int64_t* counts,
                             int32_t n_seqs, int64_t* slots_out, int64_t* copies_out,
                             int32_t* n_copies_out);
/* pa_bm_append_batch for one sequence (copies_out: room for one pair). */
pa_status pa_bm_append(pa_block_manager* bm, int64_t seq_id, int64_t n, int64_t* slots_out,
                       int64_t* copies_out, int32_t* n_copies_out);

/*
 * pa_bm_allocate_cached -- pa_bm_allocate for a prompt given by its token ids,
 * with prefix caching ("vLLM 部署深度指南", Prefix Caching 加速 and the 前缀共享 row;
 * "vLLM高性能推理引擎实战解密", section 3.1, cross-request sharing): the longest
 * run of cached full blocks from the prompt's start is reused (a block is
 * found by its parent block, the parent's generation and its tokens, exactly;
 * released cached blocks stay findable until handed out again), the rest is
 * allocated, and the prompt's full blocks become findable.  *n_cached_out
 * receives the number of leading tokens whose K/V are already in the pool (a
 * multiple of block_size, below n_tokens unless the prompt is empty): the
 * caller writes and prefills only the tokens after them.
 */
pa_status pa_bm_allocate_cached(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                                int64_t n_tokens, int64_t* n_cached_out);

/* Make the full blocks of seq_id findable by later prompts (tokens: its ids from the first). */
pa_status pa_bm_register(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                         int64_t n_tokens);

/* child (a new id) shares every block of parent; both hold the same tokens. */
pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child);

/* Release a finished sequence (its blocks return to the free list once unreferenced). */
pa_status pa_bm_free(pa_block_manager* bm, int64_t seq_id);

/*
 * Block tables of n_seqs sequences as pa_decode reads them: tables_out int32
 * [n_seqs, width] row-major, -1 past each sequence's blocks; lens_out int32
 * [n_seqs] (context lengths).  PA_ERR_INVALID_ARG if a table is wider than width.
 */
pa_status pa_bm_block_tables(pa_block_manager* bm, const int64_t* seq_ids, int32_t n_seqs,
                             int32_t width, int32_t* tables_out, int32_t* lens_out);

/*
 * pa_copy_blocks -- copy whole physical blocks of the pool on the GPU: for
 * each pair p, block pairs[2p + 1] becomes a byte copy of block pairs[2p]
 * (all tokens, K and V, every head: a block is block_bytes = block_size * 2 *
 * num_kv_heads * head_size * elt contiguous bytes of the pool's layout).
 * pairs: device int64 [n_pairs, 2]; no destination may also be a source in
 * the same call.  Pairs naming a block outside [0, num_blocks) are skipped
 * and raise device status bit 4.  pool 16-byte aligned, block_bytes a
 * multiple of 16.  Asynchronous on `stream`.
 */
pa_status pa_copy_blocks(void* pool, const int64_t* pairs, int64_t n_pairs, int32_t num_blocks,
                         int64_t block_bytes, void* stream);

/* Message describing the last error returned on the calling thread ("" if none). */
const char* pa_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
