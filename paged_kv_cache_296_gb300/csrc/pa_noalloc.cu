// pa_decode_noalloc: paged decode whose split-KV scratch is a fixed array
// compiled into this library, for callers that cannot allocate device memory.
//
// Some callers of a decode kernel have no device allocator of their own: a
// plugin or extension that a host runtime hands only its input and output
// buffers, or a serving loop that must not call cudaMalloc while requests are
// in flight (it can synchronise the device and fragments a memory budget that
// was fixed up front).  pa_decode needs scratch for its split-KV partials; this
// entry point takes it from g_noalloc_scratch instead of from the caller.
#include <cstddef>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

pa_status record_error(pa_status st, const char* msg) {
  return static_cast<pa_status>(pa::record_error_code(static_cast<int>(st), msg));
}

constexpr size_t kScratchBytes = PA_DECODE_NOALLOC_SCRATCH_BYTES;

// Lives on every device that loads this module, from then until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch per device.  In host code the array's
// name is only a host-side stand-in, so the address must come from the runtime.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // with `dev` current
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, int num_seqs,
                                       int max_blocks_per_seq, int num_blocks, int num_q_heads,
                                       int num_kv_heads, int head_size, int block_size,
                                       float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                                       float kv_scale, int partition_size, void* stream) {
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                               max_blocks_per_seq, block_size, partition_size);
  if (need > kScratchBytes) {
    return record_error(PA_ERR_WORKSPACE,
                            "pa_decode_noalloc: these sizes need more split-KV scratch than the "
                            "library's fixed buffer holds (see PA_DECODE_NOALLOC_SCRATCH_BYTES); "
                            "use pa_decode with a caller workspace or a larger partition_size");
  }
  void* scratch = nullptr;
  if (need > 0) {
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
      return record_error(PA_ERR_CUDA, "pa_decode_noalloc: cudaGetSymbolAddress of the "
                                           "scratch buffer failed");
    }
  }
  // Everything else (validation, launch) is pa_decode's, with the fixed buffer
  // as its workspace.  The partials need no zeroing: every one the merge reads
  // is written earlier in the same call.
  return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                   max_blocks_per_seq, num_blocks, num_q_heads, num_kv_heads, head_size,
                   block_size, scale, q_dtype, kv_dtype, kv_scale, partition_size, scratch,
                   scratch ? kScratchBytes : 0, stream);
}
