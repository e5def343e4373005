// KV-cache write, block-table gather and index validation kernels, plus the
// host helpers shared by the decode launchers (device status word, TMA
// descriptors).
//
// reshape_and_cache is the "write to physical block" step of append_kv
// ("vLLM 部署深度指南", section 代码层面理解): a slot s names token row s of the
// pool [num_blocks, 16, 2, Hkv, D], i.e. physical block s / 16, offset s % 16
// (section PagedAttention 方案, logical-view figure).  The gather follows the
// same figure in the other direction: logical token j of a sequence lives in
// the block its table names at position j / 16.
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

// ---------------------------------------------------------------- status word

// Error bits raised by kernels instead of trapping (see pa_device_status()).
__device__ unsigned g_pa_status;

cudaError_t device_status_ptr(unsigned** ptr) {
  constexpr int kMaxDev = 64;
  static std::atomic<unsigned*> cache[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev) {
    unsigned* p = cache[dev].load(std::memory_order_acquire);
    if (p) {
      *ptr = p;
      return cudaSuccess;
    }
  }
  void* addr = nullptr;
  e = cudaGetSymbolAddress(&addr, g_pa_status);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev) cache[dev].store(static_cast<unsigned*>(addr), std::memory_order_release);
  *ptr = static_cast<unsigned*>(addr);
  return cudaSuccess;
}

// ---------------------------------------------------------------- TMA descriptors

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}
}  // namespace

bool encode_kv_tensor_map_planes(void* desc, const void* base, int num_blocks, int num_kv_heads,
                                 int head_size, int elt_bytes, int box_pieces, const char** why) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  const cuuint64_t row = (cuuint64_t)head_size * elt_bytes;
  if (row % 128 != 0) {
    *why = "128-byte planes need rows of a multiple of 128 bytes";
    return false;
  }
  const cuuint64_t token_stride = 2ull * num_kv_heads * row;
  const cuuint64_t ntok = (cuuint64_t)num_blocks * 16;
  const CUtensorMapDataType dt =
      elt_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  // dims (elements of a 128-byte piece, token rows, pieces of a row, kv heads):
  // a box lands as [piece][token][128 B], each piece a 16-row swizzled tile.
  const cuuint64_t dims[4] = {128ull / elt_bytes, ntok, row / 128, (cuuint64_t)num_kv_heads};
  const cuuint64_t strides[3] = {token_stride, 128ull, row};
  const cuuint32_t box[4] = {128u / elt_bytes, 16u, (cuuint32_t)box_pieces, 1u};
  const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
  const CUresult r = fn(static_cast<CUtensorMap*>(desc), dt, 4, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled rejected the plane view of the KV pool";
    return false;
  }
  return true;
}

bool encode_kv_tensor_map(void* desc, const void* base, int num_blocks, int num_kv_heads,
                          int head_size, int elt_bytes, int box_heads, const char** why) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  const cuuint64_t row = (cuuint64_t)head_size * elt_bytes;
  const cuuint64_t token_stride = 2ull * num_kv_heads * row;
  const cuuint64_t ntok = (cuuint64_t)num_blocks * 16;
  const CUtensorMapDataType dt =
      elt_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUresult r;
  if (row > 128) {
    // Split each row into 128-byte halves so the box's inner extent fits the
    // 128B swizzle span: dims (elements of a half, halves, kv heads, token rows).
    const cuuint64_t dims[4] = {128ull / elt_bytes, row / 128, (cuuint64_t)num_kv_heads, ntok};
    const cuuint64_t strides[3] = {128ull, row, token_stride};
    const cuuint32_t box[4] = {128u / elt_bytes, (cuuint32_t)(row / 128), (cuuint32_t)box_heads,
                               16u};
    const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
    r = fn(static_cast<CUtensorMap*>(desc), dt, 4, const_cast<void*>(base), dims, strides, box,
           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[3] = {(cuuint64_t)head_size, (cuuint64_t)num_kv_heads, ntok};
    const cuuint64_t strides[2] = {row, token_stride};
    const cuuint32_t box[3] = {(cuuint32_t)head_size, (cuuint32_t)box_heads, 16u};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    r = fn(static_cast<CUtensorMap*>(desc), dt, 3, const_cast<void*>(base), dims, strides, box,
           es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           row == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled rejected the KV pool view";
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- reshape_and_cache

namespace {

constexpr int kSrcF16 = 0, kSrcBf16 = 1, kSrcF32 = 3;


template <int SRC>
__device__ __forceinline__ void load8(const uint8_t* p, float (&x)[8]) {
  if constexpr (SRC == kSrcF32) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (SRC == kSrcF16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      } else {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }
}

// Grid (token, chunk): each thread moves one 16-byte vector of K or V (16-bit
// caches) or quantises 8 elements into 8 bytes (E4M3 cache), so every load of
// a token is in flight at once.
constexpr int kWriteThreads = 256;

template <int SRC, bool FP8>
__global__ void __launch_bounds__(kWriteThreads)
    reshape_and_cache_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                             uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                             const int64_t* __restrict__ slots, int64_t src_stride_bytes,
                             int64_t max_slot, int hkv_d, float kv_scale) {
  // The decode kernel that follows may begin launching now; it waits for this
  // grid to complete before it reads the pool.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t n = blockIdx.x;
  const int64_t s = slots[n];
  if (s < 0 || s >= max_slot) return;  // padding, or a slot past the pool
  const uint8_t* ks = k + n * src_stride_bytes;
  const uint8_t* vs = v + n * src_stride_bytes;
  const int i = blockIdx.y * kWriteThreads + threadIdx.x;
  if constexpr (!FP8) {
    const int64_t tok_stride = 2ll * hkv_d * 2;
    const int nvec = hkv_d * 2 / 16;
    if (i >= 2 * nvec) return;
    const bool isv = i >= nvec;
    const int j = isv ? i - nvec : i;
    const uint4 x = reinterpret_cast<const uint4*>(isv ? vs : ks)[j];
    reinterpret_cast<uint4*>((isv ? vc : kc) + s * tok_stride)[j] = x;
  } else {
    constexpr int kSrcElt = (SRC == kSrcF32) ? 4 : 2;
    const int64_t tok_stride = 2ll * hkv_d;
    const int ngrp = hkv_d / 8;
    if (i >= 2 * ngrp) return;
    const bool isv = i >= ngrp;
    const int j = isv ? i - ngrp : i;
    float x[8];
    load8<SRC>((isv ? vs : ks) + (size_t)j * 8 * kSrcElt, x);
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint16_t a = f32x2_to_e4m3x2(__fdiv_rn(x[4 * h], kv_scale),
                                         __fdiv_rn(x[4 * h + 1], kv_scale));
      const uint16_t b = f32x2_to_e4m3x2(__fdiv_rn(x[4 * h + 2], kv_scale),
                                         __fdiv_rn(x[4 * h + 3], kv_scale));
      w[h] = (uint32_t)a | ((uint32_t)b << 16);
    }
    reinterpret_cast<uint2*>((isv ? vc : kc) + s * tok_stride)[j] = make_uint2(w[0], w[1]);
  }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int64_t n_tokens,
                                     int64_t src_stride_bytes, int64_t max_slot, int hkv_d,
                                     int src_dtype, int kv_dtype, float kv_scale,
                                     cudaStream_t stream) {
  if (n_tokens == 0) return cudaSuccess;
  const int units = (kv_dtype != 2) ? 2 * (hkv_d * 2 / 16) : 2 * (hkv_d / 8);
  const dim3 grid((unsigned)n_tokens, (unsigned)((units + kWriteThreads - 1) / kWriteThreads));
  const auto* kk = static_cast<const uint8_t*>(k);
  const auto* vv = static_cast<const uint8_t*>(v);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  if (kv_dtype != 2) {
    reshape_and_cache_kernel<kSrcF16, false><<<grid, kWriteThreads, 0, stream>>>(
        kk, vv, kc, vc, slot_mapping, src_stride_bytes, max_slot, hkv_d, kv_scale);
  } else if (src_dtype == 0) {
    reshape_and_cache_kernel<kSrcF16, true><<<grid, kWriteThreads, 0, stream>>>(
        kk, vv, kc, vc, slot_mapping, src_stride_bytes, max_slot, hkv_d, kv_scale);
  } else if (src_dtype == 1) {
    reshape_and_cache_kernel<kSrcBf16, true><<<grid, kWriteThreads, 0, stream>>>(
        kk, vv, kc, vc, slot_mapping, src_stride_bytes, max_slot, hkv_d, kv_scale);
  } else {
    reshape_and_cache_kernel<kSrcF32, true><<<grid, kWriteThreads, 0, stream>>>(
        kk, vv, kc, vc, slot_mapping, src_stride_bytes, max_slot, hkv_d, kv_scale);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- gather

namespace {

// One CTA per (logical block, sequence): copies the block's valid token rows
// of K and then V, 16 bytes per thread step.
__global__ void __launch_bounds__(128)
    gather_kv_kernel(uint8_t* __restrict__ k_out, uint8_t* __restrict__ v_out,
                     const uint8_t* __restrict__ kc, const uint8_t* __restrict__ vc,
                     const int32_t* __restrict__ tables, const int32_t* __restrict__ lens,
                     const int64_t* __restrict__ cu, int max_blocks, int num_blocks,
                     int row_bytes) {
  const int b = blockIdx.x;
  const int seq = blockIdx.y;
  const int L = lens[seq];
  const int tok0 = b * 16;
  if (tok0 >= L) return;
  const int valid = min(16, L - tok0);
  const int phys = tables[(size_t)seq * max_blocks + b];
  if (phys < 0 || phys >= num_blocks) return;
  const int64_t out_row0 = cu[seq] + tok0;
  const int nvec = row_bytes / 16;
  const int per = valid * nvec;
  for (int i = threadIdx.x; i < 2 * per; i += blockDim.x) {
    const bool isv = i >= per;
    const int r = isv ? i - per : i;
    const int t = r / nvec;
    const int c = r - t * nvec;
    const uint8_t* src = (isv ? vc : kc) + ((int64_t)phys * 16 + t) * (2ll * row_bytes) + c * 16;
    uint8_t* dst = (isv ? v_out : k_out) + (out_row0 + t) * row_bytes + c * 16;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

}  // namespace

cudaError_t launch_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             const int64_t* cu_seqlens, int num_seqs, int max_blocks_per_seq,
                             int num_blocks, int row_bytes, cudaStream_t stream) {
  if (num_seqs == 0) return cudaSuccess;
  const dim3 grid((unsigned)max_blocks_per_seq, (unsigned)num_seqs);
  gather_kv_kernel<<<grid, 128, 0, stream>>>(
      static_cast<uint8_t*>(k_out), static_cast<uint8_t*>(v_out),
      static_cast<const uint8_t*>(k_cache), static_cast<const uint8_t*>(v_cache), block_tables,
      context_lens, cu_seqlens, max_blocks_per_seq, num_blocks, row_bytes);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- block copies

namespace {

// Copy-on-write copies: pair p copies block pairs[2p] onto block pairs[2p+1]
// (a block is one contiguous run of block_bytes bytes of the pool).  A grid of
// (chunks, pairs) CTAs; each thread moves kCopyUnroll 16-byte vectors per
// step, all loads issued before the stores, coalesced on both sides.
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint8_t* __restrict__ pool, const int64_t* __restrict__ pairs,
                       int num_blocks, int64_t block_bytes, unsigned* status) {
  const int64_t p = blockIdx.y;
  const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, 4u);
    return;
  }
  const uint4* s = reinterpret_cast<const uint4*>(pool + src * block_bytes);
  uint4* d = reinterpret_cast<uint4*>(pool + dst * block_bytes);
  const int64_t n = block_bytes / 16;
  constexpr int64_t kSpan = (int64_t)kCopyThreads * kCopyUnroll;
  for (int64_t base = (int64_t)blockIdx.x * kSpan + threadIdx.x; base < n;
       base += (int64_t)gridDim.x * kSpan) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kCopyThreads;
      if (i < n) v[u] = s[i];
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kCopyThreads;
      if (i < n) d[i] = v[u];
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(void* pool, const int64_t* pairs, int64_t n_pairs, int num_blocks,
                               int64_t block_bytes, unsigned* status, cudaStream_t stream) {
  if (n_pairs == 0) return cudaSuccess;
  const int64_t vec = block_bytes / 16;
  const int64_t span = (int64_t)kCopyThreads * kCopyUnroll;
  const int64_t chunks = std::min<int64_t>((vec + span - 1) / span, 64);
  const dim3 grid((unsigned)std::max<int64_t>(chunks, 1), (unsigned)n_pairs);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(static_cast<uint8_t*>(pool), pairs,
                                                        num_blocks, block_bytes, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- index validation

namespace {

__global__ void check_tables_kernel(const int32_t* __restrict__ tables,
                                    const int32_t* __restrict__ lens,
                                    const int64_t* __restrict__ slots, int64_t n_tokens,
                                    int num_seqs, int max_blocks, int num_blocks, int block_size,
                                    int32_t* counts) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t max_len = (int64_t)max_blocks * block_size;
  const int64_t entries = (int64_t)num_seqs * max_blocks;
  for (int64_t idx = first; idx < entries; idx += stride) {
    const int seq = (int)(idx / max_blocks);
    const int j = (int)(idx - (int64_t)seq * max_blocks);
    const int64_t L = lens[seq];
    if (L < 0 || L > max_len) {  // counted once; its table is not judged
      if (j == 0) atomicAdd(&counts[0], 1);
      continue;
    }
    const int64_t nb = (L + block_size - 1) / block_size;
    if (j < nb) {
      const int32_t e = tables[idx];
      if (e < 0 || e >= num_blocks) atomicAdd(&counts[1], 1);
    }
  }
  const int64_t max_slot = (int64_t)num_blocks * block_size;
  for (int64_t i = first; i < n_tokens; i += stride) {
    if (slots[i] >= max_slot) atomicAdd(&counts[2], 1);
  }
}

}  // namespace

cudaError_t launch_check_tables(const int32_t* block_tables, const int32_t* context_lens,
                                const int64_t* slot_mapping, int64_t n_tokens, int num_seqs,
                                int max_blocks_per_seq, int num_blocks, int block_size,
                                int32_t* counts_dev, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(counts_dev, 0, 3 * sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  check_tables_kernel<<<1024, 256, 0, stream>>>(block_tables, context_lens, slot_mapping,
                                                n_tokens, num_seqs, max_blocks_per_seq,
                                                num_blocks, block_size, counts_dev);
  return cudaGetLastError();
}

}  // namespace pa
