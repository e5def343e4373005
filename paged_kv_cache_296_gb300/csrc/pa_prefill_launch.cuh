// Launch of the paged prefill kernel: tensor maps, grid and parameters for one
// (head size, query type, cache type) instance.
#pragma once

#include <algorithm>
#include <atomic>

#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_prefill_params.cuh"
#include "pa_prefill_tc.cuh"

namespace pa {

template <int D, int QT, bool KV8>
cudaError_t launch_prefill_instance(const PrefillArgs& a, cudaStream_t stream, const char** why) {
  using C = PrefillTcCfg<D, KV8>;
  const int G = a.num_q_heads / a.num_kv_heads;
  const long long tiles =
      ((long long)a.max_query_len * G + C::kTiles * C::kRows - 1) / (C::kTiles * C::kRows);
  if (tiles == 0 || a.num_seqs == 0) return cudaSuccess;
  if (tiles * a.num_kv_heads * a.num_seqs > 0x7FFFFFFFll) {
    *why = "too many CTAs: max_query_len * heads per KV head * sequences";
    return cudaErrorInvalidValue;
  }
  alignas(64) CUtensorMap tk;
  alignas(64) CUtensorMap tv;
  if constexpr (KV8) {
    // fp8 rows: one block of one head per box, [16 tokens][D bytes], swizzled
    if (!encode_kv_tensor_map(&tk, a.k_cache, a.num_blocks, a.num_kv_heads, D, 1, 1, why) ||
        !encode_kv_tensor_map(&tv, a.v_cache, a.num_blocks, a.num_kv_heads, D, 1, 1, why)) {
      return cudaErrorInvalidValue;
    }
  } else {
    if (!encode_kv_tensor_map_planes(&tk, a.k_cache, a.num_blocks, a.num_kv_heads, D, 2, 1,
                                     why) ||
        !encode_kv_tensor_map_planes(&tv, a.v_cache, a.num_blocks, a.num_kv_heads, D, 2, 1,
                                     why)) {
      return cudaErrorInvalidValue;
    }
  }
  // Opt in to more than 48 KB of dynamic shared memory, once per device.
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(paged_prefill_tc_kernel<D, QT, KV8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  PrefillParams p;
  p.out = a.out;
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.query_start_loc = a.query_start_loc;
  p.status = a.status;
  p.num_seqs = a.num_seqs;
  p.max_query_len = a.max_query_len;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = G;
  p.tiles = (int)tiles;
  // Tiles of one (sequence, KV head) read the same K/V: when the pool is larger
  // than half of L2 they run in adjacent bands of 8 so those reads hit in L2;
  // a smaller pool stays in L2 anyway and the heaviest tiles simply go first.
  const double pool_bytes = 2.0 * a.num_blocks * 16.0 * a.num_kv_heads * D * (KV8 ? 1.0 : 2.0);
  p.band = pool_bytes > 64.0 * 1024 * 1024 ? 8 : 1;
  // an E4M3 cache holds codes: the logits and the output take kv_scale once each
  p.scale_log2 = (float)((double)a.scale * (KV8 ? (double)a.kv_scale : 1.0) * 1.4426950408889634);
  p.out_scale = KV8 ? a.kv_scale : 1.f;
  // Programmatic stream serialisation: the grid may start while the kernel
  // before it drains (every thread waits for it before reading inputs).
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * a.num_kv_heads * a.num_seqs));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_prefill_tc_kernel<D, QT, KV8>, tk, tv, p);
}

}  // namespace pa
