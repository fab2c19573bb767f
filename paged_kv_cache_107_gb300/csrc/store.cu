// store.cu — scatter of new tokens' K/V rows into the paged cache.
//
// "nano-vllm解读", section "KVCache的写入": one kernel writes every new token's K and V
// row to its slot, the row index of the cache viewed as [num_blocks*block_size,
// H_kv*head_dim]; "3.6 ModelRunner、CUDA Graph 与性能基准", sections 2 and 5: the slot is
// computed on the host and -1 marks a padding row that writes nothing.
//
// Design: a flat grid over 16-byte vectors. Thread i moves vector i of the (token, K|V,
// vector) space, so a warp copies 512 contiguous bytes of one row and every load and
// store is a full 16-byte access. The slot is validated once per vector (the load hits
// L1 for the 2*rows/32 warps of a token).
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

template <typename Vec>
__global__ void __launch_bounds__(256) store_kvcache_kernel(
    const Vec* __restrict__ k, const Vec* __restrict__ v, int64_t k_stride_vec,
    int64_t v_stride_vec, Vec* __restrict__ k_cache, Vec* __restrict__ v_cache,
    const int32_t* __restrict__ slot_mapping, int64_t num_tokens, int row_vec,
    int64_t num_slots, int* dev_err) {
  const int64_t per_token = 2 * (int64_t)row_vec;
  const int64_t total = num_tokens * per_token;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = idx / per_token;
    const int rem = (int)(idx - tok * per_token);
    const int is_v = rem >= row_vec;
    const int e = is_v ? rem - row_vec : rem;
    const int64_t slot = __ldg(slot_mapping + tok);
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      if (e == 0 && !is_v) set_dev_err(dev_err, PA_DEV_ERR_SLOT);
      continue;
    }
    if (is_v) {
      v_cache[slot * row_vec + e] = __ldg(v + tok * v_stride_vec + e);
    } else {
      k_cache[slot * row_vec + e] = __ldg(k + tok * k_stride_vec + e);
    }
  }
}

int launch_store_kvcache(const void* k, const void* v, int64_t k_tok_stride,
                         int64_t v_tok_stride, void* k_cache, void* v_cache,
                         const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int64_t num_slots, int* dev_err, cudaStream_t stream,
                         int num_sms) {
  const int64_t row = (int64_t)num_kv_heads * head_dim;  // elements
  const bool aligned16 =
      ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
        reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) &
       15) == 0 &&
      (k_tok_stride % 8) == 0 && (v_tok_stride % 8) == 0 && (row % 8) == 0;
  const int threads = 256;
  if (aligned16) {
    const int row_vec = (int)(row / 8);
    const int64_t total = (int64_t)num_tokens * 2 * row_vec;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    store_kvcache_kernel<uint4><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), k_tok_stride / 8,
        v_tok_stride / 8, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
        slot_mapping, num_tokens, row_vec, num_slots, dev_err);
  } else {
    const int row_vec = (int)row;
    const int64_t total = (int64_t)num_tokens * 2 * row_vec;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    store_kvcache_kernel<uint16_t><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), k_tok_stride,
        v_tok_stride, static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
        slot_mapping, num_tokens, row_vec, num_slots, dev_err);
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
