// decode_step.cu — host side of pa_decode_step: the decode kernel (decode_kernel.cuh)
// instantiated with the store of each sequence's new token fused into it.
#include "decode_kernel.cuh"

namespace pa {

int launch_decode_step(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  switch (decode_head_slab(a.num_kv_heads)) {
    case 8: return dispatch_group<8, true>(a, info, stream);
    case 4: return dispatch_group<4, true>(a, info, stream);
    case 2: return dispatch_group<2, true>(a, info, stream);
    default: return dispatch_group<1, true>(a, info, stream);
  }
}

}  // namespace pa
