// prefill_d128_f16.cu — instantiation of the prefill kernel (prefill_kernel.cuh) for head_dim 128
// with IEEE fp16 elements, in its own translation unit so the variants compile in parallel.
#include "prefill_kernel.cuh"

namespace pa {

int launch_prefill_d128_f16(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                   const CUtensorMap& mk, const CUtensorMap& mv) {
  return dispatch_prefill<128, true>(a, info, stream, mk, mv);
}

}  // namespace pa
