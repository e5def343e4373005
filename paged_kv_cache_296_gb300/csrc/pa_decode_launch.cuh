// Host launcher for one instantiation of the paged decode kernels and their
// split-KV merge.  Included by the per-dtype translation units.
#pragma once

#include <algorithm>
#include <atomic>

#include <cuda_runtime.h>

#include "pa_decode_kernel.cuh"
#include "pa_decode_split.cuh"
#include "pa_internal.h"

namespace pa {

// Both kernels of a call are launched with programmatic stream serialisation:
// each may start while the kernel before it drains, and waits
// (griddepcontrol.wait) before touching anything that kernel writes.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                     cudaLaunchAttribute* attr) {
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Opt `kernel` in to `bytes` of dynamic shared memory, once per device.
template <typename K>
cudaError_t smem_opt_in(K kernel, int bytes, std::atomic<unsigned long long>& done, int dev) {
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int D, int KV, int QT, bool kAppend>
cudaError_t launch_fixed(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                         const DecodeArgs& a, cudaStream_t stream, int dev) {
  using C = DecodeCfg<D, KV>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_opt_in(paged_decode_kernel<D, KV, QT, kAppend>, C::kSmemBytes, attr_done, dev);
  if (e != cudaSuccess) return e;
  // The balanced split's grid: resident CTAs of this kernel on the whole GPU
  // (its partitions fit in one such wave), once per device.
  if (p.partition_blocks == 0) {
    static std::atomic<int> slots_cache[64];
    int slots = slots_cache[dev & 63].load(std::memory_order_acquire);
    if (slots == 0) {
      int per_sm = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, paged_decode_kernel<D, KV, QT, kAppend>, C::kThreads, C::kSmemBytes);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      slots = std::max(1, per_sm * sms);
      slots_cache[dev & 63].store(slots, std::memory_order_release);
    }
    // one CTA per work item; at least one item per (sequence, KV head group)
    const_cast<DecodeParams&>(p).slots = std::max(slots, a.num_seqs * p.kv_groups);
  }
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pdl_config(
      p.partition_blocks == 0
          ? dim3((unsigned)p.slots)
          : dim3((unsigned)p.kv_groups, (unsigned)a.num_partitions, (unsigned)a.num_seqs),
      dim3(C::kThreads), C::kSmemBytes, stream, &attr);
  e = cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, KV, QT, kAppend>, tk, tv, p);
  if (e != cudaSuccess || a.num_partitions <= 1) return e;
  cudaLaunchConfig_t mcfg = pdl_config(dim3((unsigned)((long long)a.num_seqs * a.num_q_heads)),
                                       dim3(kMergeThreads), 0, stream, &attr);
  return cudaLaunchKernelEx(&mcfg, paged_decode_merge_kernel<D, QT>, p);
}

// CTAs of the stream-K kernel resident on the whole GPU for this shared-memory
// size (one wave), capped at kMaxSplitCtas; cached per device for the last few
// sizes asked.
template <int D, int KV, int QT, bool kAppend>
cudaError_t split_slots(int dev, size_t smem, int* slots) {
  using C = DecodeCfg<D, KV>;
  constexpr int kEntries = 8;
  // entry: smem bytes in the high 32 bits, slots in the low 32 (0 = empty)
  static std::atomic<unsigned long long> cache[64][kEntries];
  static std::atomic<unsigned> next[64];
  auto& row = cache[dev & 63];
  for (int k = 0; k < kEntries; ++k) {
    const unsigned long long v = row[k].load(std::memory_order_acquire);
    if (v != 0 && (v >> 32) == smem) {
      *slots = (int)(v & 0xFFFFFFFFu);
      return cudaSuccess;
    }
  }
  int per_sm = 0, sms = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, paged_decode_split_kernel<D, KV, QT, kAppend>, SplitCfg<D, KV>::kThreads, smem);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int v = std::min(kMaxSplitCtas, std::max(1, per_sm * sms));
  const unsigned k = next[dev & 63].fetch_add(1, std::memory_order_relaxed) % kEntries;
  row[k].store(((unsigned long long)smem << 32) | (unsigned)v, std::memory_order_release);
  *slots = v;
  return cudaSuccess;
}

template <int D, int KV, int QT, bool kAppend>
cudaError_t launch_split(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                         const DecodeArgs& a, cudaStream_t stream, int dev) {
  using C = DecodeCfg<D, KV>;
  using SC = SplitCfg<D, KV>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_opt_in(paged_decode_split_kernel<D, KV, QT, kAppend>,
                              (int)SC::smem_bytes(kMaxPlanSeqs, kMaxPlanGroups), attr_done, dev);
  if (e != cudaSuccess) return e;
  const size_t smem = SC::smem_bytes(a.num_seqs, a.num_groups);
  int slots = 0;
  e = split_slots<D, KV, QT, kAppend>(dev, smem, &slots);
  if (e != cudaSuccess) return e;
  // at least two CTAs per KV head group (one for each line); the host admits
  // at most kMaxSplitCtas / 2 groups
  const int grid = std::max(slots, 2 * p.kv_groups);
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)grid), dim3(SC::kThreads), smem, stream, &attr);
  e = cudaLaunchKernelEx(&cfg, paged_decode_split_kernel<D, KV, QT, kAppend>, tk, tv, p);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)a.num_seqs * a.num_q_heads;
  cudaLaunchConfig_t mcfg =
      pdl_config(dim3((unsigned)((rows + kSplitMergeWarps - 1) / kSplitMergeWarps)),
                 dim3(kSplitMergeWarps * 32), 0, stream, &attr);
  return cudaLaunchKernelEx(&mcfg, paged_decode_split_merge_kernel<D, QT, C::kHeads>, p);
}

template <int D, int KV, int QT>
cudaError_t launch_decode_instance(const DecodeArgs& a, cudaStream_t stream, const char** why) {
  using C = DecodeCfg<D, KV>;
  alignas(64) CUtensorMap tk;
  alignas(64) CUtensorMap tv;
  if (!encode_kv_tensor_map(&tk, a.k_cache, a.num_blocks, a.num_kv_heads, D, C::kElt, C::kHeads,
                            why) ||
      !encode_kv_tensor_map(&tv, a.v_cache, a.num_blocks, a.num_kv_heads, D, C::kElt, C::kHeads,
                            why)) {
    return cudaErrorInvalidValue;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  DecodeParams p = {};
  p.out = a.out;
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.part_m = a.part_m;
  p.part_l = a.part_l;
  p.part_o = a.part_o;
  p.status = a.status;
  p.num_seqs = a.num_seqs;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.kv_groups = (a.num_kv_heads + C::kHeads - 1) / C::kHeads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.partition_blocks = a.partition_tokens / 16;
  p.num_partitions = a.num_partitions;
  const double log2e = 1.4426950408889634;
  const double kvs = (KV == kKvE4m3) ? (double)a.kv_scale : 1.0;
  p.scale_log2 = (float)((double)a.scale * log2e * kvs);
  p.out_scale = (float)kvs;
  p.kv_scale = a.kv_scale;
  p.k_new = static_cast<const uint8_t*>(a.k_new);
  p.v_new = static_cast<const uint8_t*>(a.v_new);
  p.slot_mapping = a.slot_mapping;
  p.src_stride_bytes = a.src_stride_bytes;
  p.k_cache = static_cast<uint8_t*>(const_cast<void*>(a.k_cache));
  p.v_cache = static_cast<uint8_t*>(const_cast<void*>(a.v_cache));
  p.min_partition_blocks = a.min_partition_tokens / 16;
  p.plan = a.plan;
  if (a.num_groups == 0) {
    if (a.append) return launch_fixed<D, KV, QT, true>(tk, tv, p, a, stream, dev);
    return launch_fixed<D, KV, QT, false>(tk, tv, p, a, stream, dev);
  }
  p.min_units = a.min_partition_tokens / 16;
  p.grp_off = a.grp_off;
  p.grp_seq = a.grp_seq;
  p.grp_blocks = a.grp_blocks;
  p.num_groups = a.num_groups;
  p.cut_cols = a.cut_cols;
  p.cut_m = a.cut_m;
  p.cut_l = a.cut_l;
  p.cut_o = a.cut_o;
  p.whole_m = a.whole_m;
  p.whole_l = a.whole_l;
  p.whole_o = a.whole_o;
  p.plan = a.plan;
  if (a.append) return launch_split<D, KV, QT, true>(tk, tv, p, a, stream, dev);
  return launch_split<D, KV, QT, false>(tk, tv, p, a, stream, dev);
}

}  // namespace pa
