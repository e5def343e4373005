// bf16 q / bf16 KV-cache instantiations of the paged decode kernel.
#include "pa_decode_launch.cuh"

namespace pa {
cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t stream, const char** why) {
  if (a.head_size == 64) return launch_decode_instance<64, kKvBf16, kKvBf16>(a, stream, why);
  return launch_decode_instance<128, kKvBf16, kKvBf16>(a, stream, why);
}
}  // namespace pa
