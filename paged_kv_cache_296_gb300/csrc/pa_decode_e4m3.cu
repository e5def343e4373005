// fp16 or bf16 q / fp8-E4M3 KV-cache instantiations of the paged decode kernel.
#include "pa_decode_launch.cuh"

namespace pa {
cudaError_t launch_decode_e4m3(const DecodeArgs& a, cudaStream_t stream, const char** why) {
  if (a.q_dtype == kKvF16) {
    if (a.head_size == 64) return launch_decode_instance<64, kKvE4m3, kKvF16>(a, stream, why);
    return launch_decode_instance<128, kKvE4m3, kKvF16>(a, stream, why);
  }
  if (a.head_size == 64) return launch_decode_instance<64, kKvE4m3, kKvBf16>(a, stream, why);
  return launch_decode_instance<128, kKvE4m3, kKvBf16>(a, stream, why);
}
}  // namespace pa
