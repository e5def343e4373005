// Internal host-side interface between the C entry points (pa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pa {

// The shared-prefix (stream-K) kernel (pa_decode_split.cuh): limits the host
// checks before using it.
constexpr int kMaxSplitCtas = 1024;   // grid cap; cut partials are sized for it
constexpr int kMaxPlanSeqs = 1024;    // sequences in one stream-K call
constexpr int kMaxPlanGroups = 1024;  // shared-prefix groups in one call
constexpr int kPrefixCols = 32;       // MMA columns per KV head on the prefix line
constexpr int kPlanHeader = 8;        // ints before the per-sequence plan records
constexpr int kPlanSeqInts = 8;       // ints of one sequence's plan record
constexpr int kMaxSplitHeads = 2;     // KV heads per CTA of any instantiation (E4M3)

// Everything one pa_decode launch needs, already validated by the caller.
struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs;
  int max_blocks_per_seq;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int head_size;
  int q_dtype;   // 0 f16, 1 bf16
  int kv_dtype;  // 0 f16, 1 bf16, 2 e4m3
  float scale;
  float kv_scale;
  int partition_tokens;      // > 0: given partitions; 0: balanced split chosen in the kernel
  int min_partition_tokens;  // balanced split / shared prefixes: the smallest partition or range
  int num_partitions;        // grid partitions per sequence (balanced: an upper bound)
  float* part_m;             // partitions: partials [B, Hq, P]
  float* part_l;
  float* part_o;
  unsigned* status;
  // pa_decode_append: the step's new token per sequence, written by the kernel.
  bool append;
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  int64_t src_stride_bytes;
  // shared prefixes: the groups (num_groups == 0: none, the partition kernel
  // runs) and the stream-K kernel's partials
  const int32_t* grp_off;
  const int32_t* grp_seq;
  const int32_t* grp_blocks;
  int num_groups;
  int cut_cols;
  float* cut_m;
  float* cut_l;
  float* cut_o;
  float* whole_m;
  float* whole_l;
  float* whole_o;
  int* plan;
};

// Per-dtype decode launchers (one translation unit each, compiled in parallel).
cudaError_t launch_decode_f16(const DecodeArgs& a, cudaStream_t stream, const char** why);
cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t stream, const char** why);
cudaError_t launch_decode_e4m3(const DecodeArgs& a, cudaStream_t stream, const char** why);

// Everything one pa_prefill launch needs, already validated by the caller.
struct PrefillArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int num_seqs;
  int max_query_len;
  int max_blocks_per_seq;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int head_size;
  int dtype;     // 0 f16, 1 bf16 (q and out)
  int kv_dtype;  // the cache: 0 f16, 1 bf16 (q's type), 2 E4M3 codes
  float kv_scale;
  float scale;
  unsigned* status;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream, const char** why);
cudaError_t launch_prefill_fp8(const PrefillArgs& a, cudaStream_t stream, const char** why);

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int64_t n_tokens,
                                     int64_t src_stride_bytes, int64_t max_slot, int hkv_d,
                                     int src_dtype, int kv_dtype, float kv_scale,
                                     cudaStream_t stream);

cudaError_t launch_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             const int64_t* cu_seqlens, int num_seqs, int max_blocks_per_seq,
                             int num_blocks, int row_bytes, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* pool, const int64_t* pairs, int64_t n_pairs, int num_blocks,
                               int64_t block_bytes, unsigned* status, cudaStream_t stream);

cudaError_t launch_check_tables(const int32_t* block_tables, const int32_t* context_lens,
                                const int64_t* slot_mapping, int64_t n_tokens, int num_seqs,
                                int max_blocks_per_seq, int num_blocks, int block_size,
                                int32_t* counts_dev, cudaStream_t stream);

// Records `msg` for pa_last_error() on the calling thread and returns `status`.
// (int-typed so this header needs no pa.h; the value is a pa_status.)
int record_error_code(int status, const char* msg);

// Address of this library's device status word on the current device.
cudaError_t device_status_ptr(unsigned** ptr);

// Encodes a TMA descriptor for one view (K or V) of the pool, as used by the
// decode kernel: rows of head_size elements per (token, kv head); a box is 16
// tokens x `box_heads` adjacent KV heads (heads past the last read as zeros),
// 128B (or 64B) swizzle.  `desc` points to a CUtensorMap.
bool encode_kv_tensor_map(void* desc, const void* base, int num_blocks, int num_kv_heads,
                          int head_size, int elt_bytes, int box_heads, const char** why);

// The same view for rows of a multiple of 128 bytes, with the row split into
// 128-byte pieces as its own dimension: a box of 16 tokens x `box_pieces`
// pieces x one head lands piece-major, [pieces][16 tokens][128 B], each piece
// a 16-row 128B-swizzled tile (box_pieces = 1 copies one piece, so a kernel
// can place each piece of a block where it wants).
bool encode_kv_tensor_map_planes(void* desc, const void* base, int num_blocks, int num_kv_heads,
                                 int head_size, int elt_bytes, int box_pieces, const char** why);

}  // namespace pa
