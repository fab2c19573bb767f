// decode_d64_bf16.cu — instantiation of the decode, head_dim 64, bf16 elements
// (decode_kernel.cuh), in its own translation unit so the variants compile in parallel.
#include "decode_kernel.cuh"

namespace pa {

int launch_decode_d64_bf16(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  return dispatch_slab<false, 64, false>(a, info, stream);
}

}  // namespace pa
