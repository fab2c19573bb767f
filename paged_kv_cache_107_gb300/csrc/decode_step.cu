// decode_step.cu — host side of pa_decode_step: the decode kernel (decode_kernel.cuh)
// instantiated with the store of each sequence's new token fused into it.
#include "decode_kernel.cuh"

namespace pa {

int launch_decode_step(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  if (decode_uses_tc(a.num_heads, a.num_kv_heads)) return launch_decode_step_tc(a, info, stream);
  if (a.head_dim == 128 && !a.f16) return dispatch_slab<true, 128, false>(a, info, stream);
  if (a.head_dim == 64) return a.f16 ? launch_decode_step_d64_f16(a, info, stream)
                                     : launch_decode_step_d64_bf16(a, info, stream);
  if (a.head_dim == 128) return launch_decode_step_d128_f16(a, info, stream);
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
