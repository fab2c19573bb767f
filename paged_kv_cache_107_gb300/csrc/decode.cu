// decode.cu — host side of pa_decode: workspace layout, head-slab choice and the
// launch of the decode without the fused store: the CUDA-core kernel (decode_kernel.cuh)
// for one or two query heads per KV head at head_dim 128 (bf16 here, fp16 in
// decode_d128_f16.cu), the tensor-core kernel (decode_tc.cu) for every other shape.
#include "decode_kernel.cuh"

namespace pa {

int decode_head_slab(int num_kv_heads) {
  if (num_kv_heads % 8 == 0) return 8;
  if (num_kv_heads % 4 == 0) return 4;
  if (num_kv_heads % 2 == 0) return 2;
  return 1;
}

bool decode_supported(int num_heads, int num_kv_heads) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return false;
  const int g = num_heads / num_kv_heads;
  return g >= 1 && g <= 8;
}

int decode_max_ctas(const DeviceInfo& info) { return 4 * info.num_sms; }

void decode_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int max_ctas,
                             size_t* off_counters, size_t* off_lse, size_t* off_o,
                             size_t* total) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t counters = up((size_t)num_seqs * num_kv_heads * sizeof(int));
  const size_t lse = up((size_t)max_ctas * 2 * num_heads * sizeof(float));
  const size_t o = up((size_t)max_ctas * 2 * num_heads * kHeadDim * sizeof(float));
  // partials first, counters last: the counters' offset depends on the SM count and
  // num_heads only, so a workspace sized for B sequences serves every call with fewer
  // (same heads) and always finds its counters zero
  *off_lse = 0;
  *off_o = lse;
  *off_counters = lse + o;
  *total = lse + o + counters;
}

int launch_decode(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  if (decode_uses_tc(a.num_heads, a.num_kv_heads, a.head_dim)) return launch_decode_tc(a, info, stream);
  if (a.head_dim == 128 && !a.f16) return dispatch_slab<false, 128, false>(a, info, stream);
  if (a.head_dim == 128) return launch_decode_d128_f16(a, info, stream);
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
