// Host launchers for the paged prefill kernel over an E4M3 cache (fp16 / bf16
// queries, head_size 64 / 128).
#include "pa_prefill_launch.cuh"

namespace pa {

cudaError_t launch_prefill_fp8(const PrefillArgs& a, cudaStream_t stream, const char** why) {
  if (a.dtype == 0) {
    if (a.head_size == 64) return launch_prefill_instance<64, 0, true>(a, stream, why);
    return launch_prefill_instance<128, 0, true>(a, stream, why);
  }
  if (a.head_size == 64) return launch_prefill_instance<64, 1, true>(a, stream, why);
  return launch_prefill_instance<128, 1, true>(a, stream, why);
}

}  // namespace pa
