// Host launcher for one instantiation of the paged decode kernel and its
// split-KV merge.  Included by the per-dtype translation units.
#pragma once

#include <atomic>

#include <cuda_runtime.h>

#include "pa_decode_kernel.cuh"
#include "pa_internal.h"

namespace pa {

template <int D, int KV, int QT>
cudaError_t launch_decode_instance(const DecodeArgs& a, cudaStream_t stream, const char** why) {
  using C = DecodeCfg<D, KV>;
  alignas(64) CUtensorMap tk;
  alignas(64) CUtensorMap tv;
  if (!encode_kv_tensor_map(&tk, a.k_cache, a.num_blocks, a.num_kv_heads, D, C::kElt, why) ||
      !encode_kv_tensor_map(&tv, a.v_cache, a.num_blocks, a.num_kv_heads, D, C::kElt, why)) {
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
  p.group = a.num_q_heads / a.num_kv_heads;
  p.partition_blocks = a.partition_tokens / 16;
  p.num_partitions = a.num_partitions;
  const double log2e = 1.4426950408889634;
  const double kvs = (KV == kKvE4m3) ? (double)a.kv_scale : 1.0;
  p.scale_log2 = (float)((double)a.scale * log2e * kvs);
  p.out_scale = (float)kvs;

  // Opt in to more than 48 KB of dynamic shared memory, once per device.
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(paged_decode_kernel<D, KV, QT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }

  const dim3 grid((unsigned)a.num_kv_heads, (unsigned)a.num_partitions, (unsigned)a.num_seqs);
  paged_decode_kernel<D, KV, QT><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.num_partitions > 1) {
    const long long warps = (long long)a.num_seqs * a.num_q_heads;
    paged_decode_merge_kernel<D, QT><<<(unsigned)((warps + 3) / 4), 128, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace pa
