// Host launchers for the paged prefill kernel over 16-bit caches (fp16 / bf16,
// head_size 64 / 128); the E4M3-cache instances are in pa_prefill_fp8.cu.
#include "pa_prefill_launch.cuh"

namespace pa {

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream, const char** why) {
  if (a.kv_dtype == 2) return launch_prefill_fp8(a, stream, why);
  if (a.dtype == 0) {
    if (a.head_size == 64) return launch_prefill_instance<64, 0, false>(a, stream, why);
    return launch_prefill_instance<128, 0, false>(a, stream, why);
  }
  if (a.head_size == 64) return launch_prefill_instance<64, 1, false>(a, stream, why);
  return launch_prefill_instance<128, 1, false>(a, stream, why);
}

}  // namespace pa
