// pa_api.cu — the exported C ABI (include/pa.h): argument validation, then launch.
// Nothing here allocates device memory or synchronises the host.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_launch.h"

namespace pa {

bool current_device_info(DeviceInfo* info) {
  static DeviceInfo cache[64];
  static bool valid[64] = {false};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!valid[dev]) {
    DeviceInfo d{};
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    cache[dev] = d;
    valid[dev] = true;
  }
  *info = cache[dev];
  return true;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static float resolve_scale(float scale, int head_dim) {
  if (!(scale > 0.f) || isnan(scale)) scale = 1.0f / sqrtf((float)head_dim);
  return scale * 1.4426950408889634f;  // exp(x) = exp2(x * log2(e))
}

}  // namespace pa

extern "C" {

const char* pa_status_str(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: inconsistent sizes";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: head_dim, group size or block size not supported";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: decode workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime error";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: pointer or stride not 16-byte aligned";
    default: return "unknown pa status";
  }
}

int pa_version(void) { return (1 << 16) | 0; }

int pa_store_kvcache(const void* k, const void* v, int64_t k_tok_stride, int64_t v_tok_stride,
                     void* k_cache, void* v_cache, const int32_t* slot_mapping, int num_tokens,
                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                     int* dev_err, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_SHAPE;
  if (!pa::head_dim_supported(head_dim)) return PA_ERR_UNSUPPORTED;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (k_tok_stride < row || v_tok_stride < row) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_NULL;
  pa::DeviceInfo info;
  if (!pa::current_device_info(&info)) return PA_ERR_CUDA;
  return pa::launch_store_kvcache(k, v, k_tok_stride, v_tok_stride, k_cache, v_cache,
                                  slot_mapping, num_tokens, num_kv_heads, head_dim,
                                  num_blocks * (int64_t)block_size, dev_err,
                                  static_cast<cudaStream_t>(stream), info.num_sms);
}

int pa_staged_write_apply(void* base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
                          int elem_bytes, const int32_t* rows, const int32_t* starts,
                          const int32_t* offsets, const void* values, int num_writes,
                          int64_t num_values, int* dev_err, void* stream) {
  if (num_rows < 0 || num_cols < 0 || row_stride < num_cols || num_writes < 0 || num_values < 0)
    return PA_ERR_SHAPE;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return PA_ERR_UNSUPPORTED;
  if (num_values > INT32_MAX) return PA_ERR_UNSUPPORTED;  // offsets are int32
  if (num_values == 0) return PA_OK;
  if (num_writes == 0) return PA_ERR_SHAPE;  // values without a run to hold them
  if (!base || !rows || !starts || !offsets || !values) return PA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(base) | reinterpret_cast<uintptr_t>(values)) %
          (uintptr_t)elem_bytes !=
      0)
    return PA_ERR_ALIGN;
  pa::DeviceInfo info;
  if (!pa::current_device_info(&info)) return PA_ERR_CUDA;
  return pa::launch_staged_write(base, num_rows, num_cols, row_stride, elem_bytes, rows, starts,
                                 offsets, values, num_writes, num_values, dev_err,
                                 static_cast<cudaStream_t>(stream), info.num_sms);
}

int pa_staged_upload_apply(void* base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
                           int elem_bytes, const void* packed_host, void* packed_dev,
                           const pa_staged_layout* layout, int* dev_err, void* stream) {
  if (!layout) return PA_ERR_NULL;
  if (num_rows < 0 || num_cols < 0 || row_stride < num_cols || layout->bytes < 0 ||
      layout->num_writes < 0 || layout->num_values < 0)
    return PA_ERR_SHAPE;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return PA_ERR_UNSUPPORTED;
  if (layout->bytes == 0) return PA_OK;
  if (!packed_host || !packed_dev || (layout->num_values > 0 && !base)) return PA_ERR_NULL;
  if (layout->num_values > 0 && layout->num_writes == 0) return PA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(packed_dev) & 15) ||
      (reinterpret_cast<uintptr_t>(base) % (uintptr_t)elem_bytes) ||
      (layout->values_offset % 16) || (layout->rows_offset % 4) || (layout->starts_offset % 4) ||
      (layout->offsets_offset % 4))
    return PA_ERR_ALIGN;
  pa::DeviceInfo info;
  if (!pa::current_device_info(&info)) return PA_ERR_CUDA;
  return pa::launch_staged_upload_apply(base, num_rows, num_cols, row_stride, elem_bytes,
                                        packed_host, packed_dev, layout, dev_err,
                                        static_cast<cudaStream_t>(stream), info.num_sms);
}

size_t pa_sample_workspace_size(int num_seqs) {
  if (num_seqs < 0) return 0;
  return pa::sample_workspace_bytes(num_seqs > 0 ? num_seqs : 1);
}

int pa_gumbel_sample(int64_t* out, const void* logits, int64_t row_stride, int logits_dtype,
                     int num_seqs, int vocab_size, const float* temperatures,
                     const uint64_t* seeds, const uint64_t* offsets, void* workspace,
                     size_t workspace_bytes, int* dev_err, void* stream) {
  if (num_seqs < 0 || vocab_size <= 0 || row_stride < vocab_size) return PA_ERR_SHAPE;
  if (logits_dtype != PA_DTYPE_F32 && logits_dtype != PA_DTYPE_BF16) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!out || !logits || !temperatures || !seeds || !offsets) return PA_ERR_NULL;
  if (!workspace || workspace_bytes < pa::sample_workspace_bytes(num_seqs))
    return PA_ERR_WORKSPACE;
  const uintptr_t esz = logits_dtype == PA_DTYPE_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(logits) % esz) || (reinterpret_cast<uintptr_t>(out) & 7) ||
      (reinterpret_cast<uintptr_t>(seeds) & 7) || (reinterpret_cast<uintptr_t>(offsets) & 7) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return PA_ERR_ALIGN;
  pa::DeviceInfo info;
  if (!pa::current_device_info(&info)) return PA_ERR_CUDA;
  return pa::launch_gumbel_sample(out, logits, row_stride, logits_dtype == PA_DTYPE_BF16,
                                  num_seqs, vocab_size, temperatures, seeds, offsets, workspace,
                                  dev_err, static_cast<cudaStream_t>(stream), info.num_sms);
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || !pa::head_dim_supported(head_dim))
    return 0;
  pa::DeviceInfo info;
  if (!pa::current_device_info(&info)) return 0;
  size_t a, b, c, total;
  pa::decode_workspace_layout(num_seqs, num_heads, num_kv_heads, pa::decode_max_ctas(info), &a,
                              &b, &c, &total);
  return total;
}

}  // extern "C"

namespace pa {

int decode_prepare(void* out, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                   int head_dim, int dtype, int block_size, int64_t num_blocks, float scale,
                   int grid_ctas, int* dev_err, const DecodeStepInput* step, DecodeArgs* a,
                   DeviceInfo* info, bool* nothing) {
  *nothing = false;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq < 0 || grid_ctas < 0)
    return PA_ERR_SHAPE;
  if (num_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  if (!head_dim_supported(head_dim) || !decode_supported(num_heads, num_kv_heads) ||
      (dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_F16))
    return PA_ERR_UNSUPPORTED;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (step) {
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (step->k_new_stride < row || step->v_new_stride < row) return PA_ERR_SHAPE;
  }
  if (num_seqs == 0) {
    *nothing = true;
    return PA_OK;
  }
  if (step) {
    if (!step->k_new || !step->v_new || !step->slot_mapping) return PA_ERR_NULL;
    // rows move with bulk copies: 16-byte aligned starts
    if (!aligned16(step->k_new) || !aligned16(step->v_new) || (step->k_new_stride & 7) ||
        (step->v_new_stride & 7))
      return PA_ERR_ALIGN;
  }
  if (!out || !q || !k_cache || !v_cache || !context_lens) return PA_ERR_NULL;
  if (max_blocks_per_seq > 0 && !block_tables) return PA_ERR_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGN;
  if (!current_device_info(info)) return PA_ERR_CUDA;
  const bool auto_grid = grid_ctas == 0;
  if (auto_grid) grid_ctas = info->num_sms;
  if (grid_ctas > decode_max_ctas(*info)) return PA_ERR_SHAPE;
  *a = DecodeArgs{};
  a->out = out;
  a->q = q;
  a->k_cache = k_cache;
  a->v_cache = v_cache;
  a->block_tables = block_tables;
  a->context_lens = context_lens;
  a->max_blocks = max_blocks_per_seq;
  a->num_seqs = num_seqs;
  a->num_heads = num_heads;
  a->num_kv_heads = num_kv_heads;
  a->block_size = block_size;
  a->num_blocks = num_blocks;
  a->scale_log2 = resolve_scale(scale, head_dim);
  a->head_dim = head_dim;
  a->f16 = dtype == PA_DTYPE_F16;
  a->grid_ctas = grid_ctas;
  a->min_tiles = auto_grid ? kDecodeMinTilesPerCta : 1;
  a->dev_err = dev_err;
  if (step) {
    a->k_new = step->k_new;
    a->v_new = step->v_new;
    a->k_new_stride = step->k_new_stride;
    a->v_new_stride = step->v_new_stride;
    a->slot_mapping = step->slot_mapping;
  }
  return PA_OK;
}

size_t decode_bind_workspace(DecodeArgs* a, unsigned char* ws, int layout_ctas) {
  size_t off_c, off_l, off_o, total;
  decode_workspace_layout(a->num_seqs, a->num_heads, a->num_kv_heads, layout_ctas, &off_c,
                          &off_l, &off_o, &total);
  a->counters = ws ? reinterpret_cast<int*>(ws + off_c) : nullptr;
  a->part_lse = ws ? reinterpret_cast<float*>(ws + off_l) : nullptr;
  a->part_o = ws ? reinterpret_cast<float*>(ws + off_o) : nullptr;
  return total;
}

// pa_decode and pa_decode_step: the caller's workspace, laid out for the largest grid the
// device allows (so one workspace serves every grid_ctas); `step` is null for the plain
// call.
static int decode_entry(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int num_seqs, int num_heads,
                        int num_kv_heads, int head_dim, int dtype, int block_size,
                        int64_t num_blocks, float scale, int grid_ctas, void* workspace,
                        size_t workspace_bytes, int* dev_err, void* stream,
                        const DecodeStepInput* step) {
  DecodeArgs a;
  DeviceInfo info;
  bool nothing = false;
  const int rc = decode_prepare(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_heads, num_kv_heads, head_dim,
                                dtype, block_size, num_blocks, scale, grid_ctas, dev_err, step,
                                &a, &info, &nothing);
  if (rc != PA_OK || nothing) return rc;
  const size_t need =
      decode_bind_workspace(&a, static_cast<unsigned char*>(workspace), decode_max_ctas(info));
  if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return PA_ERR_ALIGN;
  if (step) return launch_decode_step(a, info, static_cast<cudaStream_t>(stream));
  return launch_decode(a, info, static_cast<cudaStream_t>(stream));
}

}  // namespace pa

extern "C" {

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int dtype,
              int block_size, int64_t num_blocks, float scale, int grid_ctas, void* workspace,
              size_t workspace_bytes, int* dev_err, void* stream) {
  return pa::decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                          context_lens, num_seqs, num_heads, num_kv_heads, head_dim, dtype,
                          block_size, num_blocks, scale, grid_ctas, workspace, workspace_bytes,
                          dev_err, stream, nullptr);
}

int pa_decode_step(void* out, const void* q, const void* k_new, const void* v_new,
                   int64_t k_new_stride, int64_t v_new_stride, void* k_cache, void* v_cache,
                   const int32_t* slot_mapping, const int32_t* block_tables,
                   int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                   int num_heads, int num_kv_heads, int head_dim, int dtype, int block_size,
                   int64_t num_blocks, float scale, int grid_ctas, void* workspace,
                   size_t workspace_bytes, int* dev_err, void* stream) {
  const pa::DecodeStepInput step{k_new, v_new, k_new_stride, v_new_stride, slot_mapping};
  return pa::decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                          context_lens, num_seqs, num_heads, num_kv_heads, head_dim, dtype,
                          block_size, num_blocks, scale, grid_ctas, workspace, workspace_bytes,
                          dev_err, stream, &step);
}

int pa_prefill_varlen(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
                      int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                      int head_dim, int dtype, int block_size, int64_t num_blocks, int causal,
                      float scale, int* dev_err, void* stream) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return PA_ERR_SHAPE;
  if (num_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  if (!pa::head_dim_supported(head_dim) ||
      !pa::prefill_supported(num_heads, num_kv_heads, block_size) ||
      (dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_F16))
    return PA_ERR_UNSUPPORTED;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (max_seqlen_k > (int64_t)max_blocks_per_seq * block_size) return PA_ERR_SHAPE;
  if (num_seqs == 0 || max_seqlen_q == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k) return PA_ERR_NULL;
  if (max_blocks_per_seq > 0 && !block_tables) return PA_ERR_NULL;
  if (!pa::aligned16(out) || !pa::aligned16(q) || !pa::aligned16(k_cache) ||
      !pa::aligned16(v_cache))
    return PA_ERR_ALIGN;
  pa::DeviceInfo info;
  if (!pa::current_device_info(&info)) return PA_ERR_CUDA;
  pa::PrefillArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.max_blocks = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = pa::resolve_scale(scale, head_dim);
  a.head_dim = head_dim;
  a.f16 = dtype == PA_DTYPE_F16;
  a.dev_err = dev_err;
  return pa::launch_prefill(a, info, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
