// tensor_map.cu — host-side tensor maps over the paged caches (tensor_map.h).
#include "tensor_map.h"

#include <cuda_runtime.h>

#include <mutex>

namespace pa {

PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_slab_map(CUtensorMap* map, const void* base, int num_kv_heads, int head_dim, bool f16,
                   int block_size, int64_t num_blocks, int box_tokens, int box_heads) {
  auto encode = tmap_encode_fn();
  if (!encode) return false;
  const cuuint64_t row = (cuuint64_t)num_kv_heads * head_dim * 2;  // bytes of one token row
  cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)block_size, (cuuint64_t)num_kv_heads,
                        (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {row, (cuuint64_t)head_dim * 2, row * (cuuint64_t)block_size};
  cuuint32_t box[4] = {64, (cuuint32_t)box_tokens, (cuuint32_t)box_heads, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult rc =
      encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

bool make_rows_map(CUtensorMap* map, const void* base, int64_t rows, int num_heads,
                   int head_dim, bool f16, int box_heads, int box_rows) {
  auto encode = tmap_encode_fn();
  if (!encode || rows <= 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_heads * head_dim * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult rc =
      encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

}  // namespace pa
