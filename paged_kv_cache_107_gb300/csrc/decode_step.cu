// decode_step.cu — host side of pa_decode_step: the decode with the store of each
// sequence's new token fused into it, on the CUDA-core kernel (decode_kernel.cuh) or the
// tensor-core kernel (decode_step_tc.cu) as for pa_decode.
#include "decode_kernel.cuh"

namespace pa {

int launch_decode_step(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  if (decode_uses_tc(a.num_heads, a.num_kv_heads, a.head_dim))
    return launch_decode_step_tc(a, info, stream);
  if (a.head_dim == 128 && !a.f16) return dispatch_slab<true, 128, false>(a, info, stream);
  if (a.head_dim == 128) return launch_decode_step_d128_f16(a, info, stream);
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
