// decode_step_d128_f16.cu — instantiation of the decode step with the fused store, head_dim 128, IEEE fp16 elements
// (decode_kernel.cuh), in its own translation unit so the variants compile in parallel.
#include "decode_kernel.cuh"

namespace pa {

int launch_decode_step_d128_f16(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  return dispatch_slab<true, 128, true>(a, info, stream);
}

}  // namespace pa
