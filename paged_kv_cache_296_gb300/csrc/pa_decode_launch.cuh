// Host launcher for one instantiation of the paged decode kernel and its
// split-KV merge.  Included by the per-dtype translation units.
#pragma once

#include <algorithm>
#include <atomic>

#include <cuda_runtime.h>

#include "pa_decode_kernel.cuh"
#include "pa_internal.h"

namespace pa {

template <int D, int KV, int QT, bool kAppend>
cudaError_t launch_decode_kernel(const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeParams& p, const DecodeArgs& a, cudaStream_t stream) {
  using C = DecodeCfg<D, KV>;
  // Opt in to more than 48 KB of dynamic shared memory, once per device.
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(paged_decode_kernel<D, KV, QT, kAppend>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  // Resident CTAs of this kernel on the whole GPU (the balanced split fits its
  // partitions into one such wave), once per device.
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
    // One CTA per work item; at least one item per (sequence, KV head group).
    const_cast<DecodeParams&>(p).slots = std::max(slots, a.num_seqs * p.kv_groups);
  }
  // Both kernels are launched with programmatic stream serialisation: each may
  // start while the kernel before it drains, and waits (griddepcontrol.wait)
  // before touching anything that kernel writes.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.partition_blocks == 0
                    ? dim3((unsigned)p.slots)
                    : dim3((unsigned)p.kv_groups, (unsigned)a.num_partitions, (unsigned)a.num_seqs);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, KV, QT, kAppend>, tk, tv, p);
  if (e != cudaSuccess) return e;
  if (a.num_partitions > 1) {
    cudaLaunchConfig_t mcfg = cfg;
    mcfg.gridDim = dim3((unsigned)((long long)a.num_seqs * a.num_q_heads));
    mcfg.blockDim = dim3(kMergeThreads);
    mcfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&mcfg, paged_decode_merge_kernel<D, QT>, p);
  }
  return e;
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
  DecodeParams p;
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
  p.min_partition_blocks = a.min_partition_tokens / 16;
  p.slots = 0;
  p.plan = a.plan;
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
  if (a.append) return launch_decode_kernel<D, KV, QT, true>(tk, tv, p, a, stream);
  return launch_decode_kernel<D, KV, QT, false>(tk, tv, p, a, stream);
}

}  // namespace pa
