// prefill.cu — host side of pa_prefill_varlen: the 4-D tensor maps over the paged cache,
// the supported shapes, and the launch of the prefill kernel (prefill_kernel.cuh); head_dim
// 128 with bf16 is instantiated here, the other combinations in prefill_d*_*.cu.
#include "prefill_kernel.cuh"
#include "tensor_map.h"

namespace pa {
namespace {

// ---------------------------------------------------------------- host side
bool make_cache_map(CUtensorMap* map, const void* base, int num_kv_heads, int head_dim,
                    bool f16, int block_size, int64_t num_blocks) {
  auto encode = tmap_encode_fn();
  if (!encode) return false;
  const int box_rows = block_size < kKeys ? block_size : kKeys;
  cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size,
                        (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_kv_heads * head_dim * 2,
                           (cuuint64_t)block_size * num_kv_heads * head_dim * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult rc = encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                       4, const_cast<void*>(base), dims,
                       strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int num_heads, int num_kv_heads, int block_size) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return false;
  const int g = num_heads / num_kv_heads;
  if (!(g == 1 || g == 2 || g == 4 || g == 8)) return false;
  if (block_size % kKeys == 0) return true;
  return block_size >= 8 && block_size % 8 == 0 && kKeys % block_size == 0;
}

int launch_prefill(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  if (a.num_seqs > 65535 || a.max_seqlen_q <= 0) return PA_ERR_UNSUPPORTED;
  CUtensorMap mk, mv;
  if (!make_cache_map(&mk, a.k_cache, a.num_kv_heads, a.head_dim, a.f16, a.block_size,
                      a.num_blocks) ||
      !make_cache_map(&mv, a.v_cache, a.num_kv_heads, a.head_dim, a.f16, a.block_size,
                      a.num_blocks))
    return PA_ERR_CUDA;
  if (a.head_dim == 128 && !a.f16) return dispatch_prefill<128, false>(a, info, stream, mk, mv);
  if (a.head_dim == 64) return a.f16 ? launch_prefill_d64_f16(a, info, stream, mk, mv)
                                     : launch_prefill_d64_bf16(a, info, stream, mk, mv);
  if (a.head_dim == 128) return launch_prefill_d128_f16(a, info, stream, mk, mv);
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
