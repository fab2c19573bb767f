// decode_step_tc.cu — instantiations of the decode step with the fused store on the
// tensor-core path (decode_tc.cuh): every shape the CUDA-core kernel does not take
// (decode_uses_tc), head_dim 64 or 128, bf16 or IEEE fp16 elements.
#include "decode_tc.cuh"

namespace pa {

int launch_decode_step_tc(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  if (a.head_dim == 128) return a.f16 ? dispatch_slab_tc<true, 128, true>(a, info, stream)
                                      : dispatch_slab_tc<true, 128, false>(a, info, stream);
  if (a.head_dim == 64) return a.f16 ? dispatch_slab_tc<true, 64, true>(a, info, stream)
                                     : dispatch_slab_tc<true, 64, false>(a, info, stream);
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
