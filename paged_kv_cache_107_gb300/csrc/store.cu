// store.cu — scatter of new tokens' K/V rows into the paged cache.
//
// "nano-vllm解读", section "KVCache的写入": one kernel writes every new token's K and V
// row to its slot, the row index of the cache viewed as [num_blocks*block_size,
// H_kv*head_dim]; "3.6 ModelRunner、CUDA Graph 与性能基准", sections 2 and 5: the slot is
// computed on the host and -1 marks a padding row that writes nothing.
//
// Design: one warp per (token, K|V) row, rows dealt to the warps of the grid in turn. A
// lane moves vectors lane, lane+32, ... of the row (16 bytes each when the rows allow,
// else one element), up to kStoreUnroll of them loaded before any is stored, so a lane
// keeps that many loads in flight. The first chunk's loads are issued beside the slot's
// load, before the slot is tested: the source row exists for every token, padding
// included, and the two memory round trips overlap instead of following each other.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kStoreUnroll = 4;     // vectors per lane loaded before the stores
constexpr int kStoreBlocksPerSM = 6;  // resident 256-thread blocks per SM (register budget)

template <typename Vec>
__global__ void __launch_bounds__(256, kStoreBlocksPerSM) store_kvcache_kernel(
    const Vec* __restrict__ k, const Vec* __restrict__ v, int64_t k_stride_vec,
    int64_t v_stride_vec, Vec* __restrict__ k_cache, Vec* __restrict__ v_cache,
    const int32_t* __restrict__ slot_mapping, int64_t num_tokens, int row_vec,
    int64_t num_slots, int* dev_err) {
  constexpr int U = kStoreUnroll;
  const int lane = threadIdx.x & 31;
  const int64_t rows = 2 * num_tokens;  // row 2t: K of token t, row 2t+1: its V
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const int64_t tok = r >> 1;
    const bool is_v = (r & 1) != 0;
    const Vec* src = is_v ? v + tok * v_stride_vec : k + tok * k_stride_vec;
    const int64_t slot = __ldg(slot_mapping + tok);
    Vec buf[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (lane + 32 * u < row_vec) buf[u] = __ldg(src + lane + 32 * u);
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      if (lane == 0 && !is_v) set_dev_err(dev_err, PA_DEV_ERR_SLOT);
      continue;
    }
    Vec* dst = (is_v ? v_cache : k_cache) + slot * row_vec;
    for (int e0 = lane;; ) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (e0 + 32 * u < row_vec) dst[e0 + 32 * u] = buf[u];
      e0 += 32 * U;
      if (e0 >= row_vec) break;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (e0 + 32 * u < row_vec) buf[u] = __ldg(src + e0 + 32 * u);
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
    int64_t blocks = ((int64_t)num_tokens * 2 + threads / 32 - 1) / (threads / 32);
    const int64_t cap = (int64_t)num_sms * kStoreBlocksPerSM;  // one resident wave
    if (blocks > cap) blocks = cap;
    store_kvcache_kernel<uint4><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), k_tok_stride / 8,
        v_tok_stride / 8, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
        slot_mapping, num_tokens, row_vec, num_slots, dev_err);
  } else {
    const int row_vec = (int)row;
    int64_t blocks = ((int64_t)num_tokens * 2 + threads / 32 - 1) / (threads / 32);
    const int64_t cap = (int64_t)num_sms * kStoreBlocksPerSM;  // one resident wave
    if (blocks > cap) blocks = cap;
    store_kvcache_kernel<uint16_t><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), k_tok_stride,
        v_tok_stride, static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
        slot_mapping, num_tokens, row_vec, num_slots, dev_err);
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
