// prefill_d64_bf16.cu — instantiation of the prefill kernel (prefill_kernel.cuh) for head_dim 64
// with bf16 elements, in its own translation unit so the variants compile in parallel.
#include "prefill_kernel.cuh"

namespace pa {

int launch_prefill_d64_bf16(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                   const CUtensorMap& mk, const CUtensorMap& mv) {
  return dispatch_prefill<64, false>(a, info, stream, mk, mv);
}

}  // namespace pa
