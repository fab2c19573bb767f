// pa_launch.h — internal host-side launchers behind the C ABI (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// The head dims the kernels are built for.
constexpr int kHeadDimApi = 128;
inline bool head_dim_supported(int d) { return d == 64 || d == 128; }

struct DeviceInfo {
  int device;
  int num_sms;
  int max_smem_optin;
  int cc_major;
  int cc_minor;
};

// Cached per-device properties of the current device; returns false on a CUDA error.
bool current_device_info(DeviceInfo* info);

int launch_store_kvcache(const void* k, const void* v, int64_t k_tok_stride,
                         int64_t v_tok_stride, void* k_cache, void* v_cache,
                         const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int64_t num_slots, int* dev_err, cudaStream_t stream,
                         int num_sms);

int launch_staged_write(void* base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
                        int elem_bytes, const int32_t* rows, const int32_t* starts,
                        const int32_t* offsets, const void* values, int num_writes,
                        int64_t num_values, int* dev_err, cudaStream_t stream, int num_sms);

int launch_staged_upload_apply(void* base, int64_t num_rows, int64_t num_cols,
                               int64_t row_stride, int elem_bytes, const void* packed_host,
                               void* packed_dev, const pa_staged_layout* lay, int* dev_err,
                               cudaStream_t stream, int num_sms);

size_t sample_workspace_bytes(int num_rows);
int launch_gumbel_sample(int64_t* out, const void* logits, int64_t row_stride, int is_bf16,
                         int num_rows, int vocab, const float* temperatures,
                         const uint64_t* seeds, const uint64_t* offsets, void* workspace,
                         int* dev_err, cudaStream_t stream, int num_sms);

struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int max_blocks;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int block_size;
  int64_t num_blocks;
  float scale_log2;  // softmax scale * log2(e)
  int grid_ctas;     // CTAs along the key stream (per head slab)
  int min_tiles;     // fewest key tiles per CTA (1: every CTA of grid_ctas may take work)
  int head_dim;      // 64 or 128
  int f16;           // element type of q, caches, out: 0 = bf16, 1 = IEEE fp16
  int* counters;     // [num_seqs * num_kv_heads]
  // fused store (pa_decode_step only; null / 0 otherwise): token b's rows, its slot
  const void* k_new;
  const void* v_new;
  int64_t k_new_stride;  // elements between tokens
  int64_t v_new_stride;
  const int32_t* slot_mapping;
  float* part_o;     // [max_ctas * 2 * num_heads * head_dim]
  float* part_lse;   // [max_ctas * 2 * num_heads]
  int* dev_err;
};

// The new tokens of pa_decode_step (null for pa_decode and pa_decode_noalloc).
struct DecodeStepInput {
  const void* k_new;
  const void* v_new;
  int64_t k_new_stride;
  int64_t v_new_stride;
  const int32_t* slot_mapping;
};

// Argument validation and packing shared by pa_decode, pa_decode_step and
// pa_decode_noalloc (every check that does not concern the workspace). On PA_OK, *a holds
// every field but the workspace pointers, *info describes the current device and the grid
// is resolved (0 = one CTA per SM); *nothing is set when there is no sequence to launch.
int decode_prepare(void* out, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                   int head_dim, int dtype, int block_size, int64_t num_blocks, float scale,
                   int grid_ctas, int* dev_err, const DecodeStepInput* step, DecodeArgs* a,
                   DeviceInfo* info, bool* nothing);
// Points a's counters and partial-result slots into `ws`, laid out for layout_ctas CTAs
// (decode_workspace_layout); returns the bytes that layout needs. ws may be null (only
// the size is wanted then).
size_t decode_bind_workspace(DecodeArgs* a, unsigned char* ws, int layout_ctas);

// With the automatic grid, a CTA takes at least this many key tiles (64 KB of K and V
// each at H_kv = 8): a short stream is then cut into fewer, longer CTA ranges, so that a
// small batch's sequences are split into fewer segments to combine.
constexpr int kDecodeMinTilesPerCta = 4;

// Maximum CTAs along the key stream that a decode workspace is sized for.
int decode_max_ctas(const DeviceInfo& info);
// Workspace layout: byte offsets of the counters, partial LSEs and partial outputs.
void decode_workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int max_ctas,
                             size_t* off_counters, size_t* off_lse, size_t* off_o,
                             size_t* total);
// Head slab (KV heads handled by one CTA) for a given num_kv_heads: 8, 4, 2 or 1.
int decode_head_slab(int num_kv_heads);
bool decode_supported(int num_heads, int num_kv_heads);
int launch_decode(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream);
// The CUDA-core decode (and fused-step) instantiations with fp16 elements, in their own
// translation units.
int launch_decode_d128_f16(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream);
int launch_decode_step_d128_f16(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream);
// The tensor-core path (decode_tc.cuh).
int launch_decode_tc(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream);
int launch_decode_step_tc(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream);
// Shapes that take the tensor-core path: every group of 3..8 query heads per KV head, and
// groups of 1 or 2 unless the head dimension is 128 and one slab holds all KV heads
// (num_kv_heads 1, 2, 4 or 8), the case where a CUDA-core tile is one contiguous run of
// cache rows. Elsewhere the tensor-core kernel's TMA boxes stream faster.
inline bool decode_uses_tc(int num_heads, int num_kv_heads, int head_dim) {
  const int g = num_heads / num_kv_heads;
  if (g >= 3) return true;
  const bool one_slab = num_kv_heads == 1 || num_kv_heads == 2 || num_kv_heads == 4 ||
                        num_kv_heads == 8;
  return !(head_dim == 128 && one_slab);
}
// The same kernel with the store of token b (k_new/v_new row b) at slot_mapping[b] fused in;
// the caches are written, so a.k_cache / a.v_cache must point to writable memory.
int launch_decode_step(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream);

struct PrefillArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int max_blocks;
  int num_seqs;
  int max_seqlen_q;
  int max_seqlen_k;
  int num_heads;
  int num_kv_heads;
  int block_size;
  int64_t num_blocks;
  int causal;
  float scale_log2;
  int head_dim;  // 64 or 128
  int f16;       // element type of q, caches, out: 0 = bf16, 1 = IEEE fp16
  int* dev_err;
  int persistent;  // set by the launcher: 1 = one CTA per SM walking a sorted unit list
};

bool prefill_supported(int num_heads, int num_kv_heads, int block_size);
int launch_prefill(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream);
// The prefill instantiations other than head_dim 128 with bf16, one translation unit each.
int launch_prefill_d64_bf16(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                            const CUtensorMap& mk, const CUtensorMap& mv);
int launch_prefill_d64_f16(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                           const CUtensorMap& mk, const CUtensorMap& mv);
int launch_prefill_d128_f16(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                            const CUtensorMap& mk, const CUtensorMap& mv);

}  // namespace pa
