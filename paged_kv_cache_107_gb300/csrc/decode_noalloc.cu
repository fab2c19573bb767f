// decode_noalloc.cu — pa_decode_noalloc: paged decode for callers that cannot allocate
// device memory.
//
// pa_decode needs a caller-provided scratch workspace (arrival counters and the partial
// results of sequences that are split across CTAs). Some callers cannot create one: code
// that runs where no allocator is available or allowed (a plugin inside a host program
// that owns all device memory, a runtime that forbids allocation after start-up, or a
// caller with a fixed memory budget). This entry point gives them the same computation
// with the scratch held in a fixed-size array in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds
// it (kScratchBytes) until the process exits. On the host its name is only a stand-in, so
// the device address is looked up with cudaGetSymbolAddress once per device, with that
// device current, the first time pa_decode_noalloc runs on it; that first call should
// therefore come before any stream capture. Nothing here calls cudaMalloc, cudaFree or an
// allocating library routine.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB, shared by every call

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch on the current device (looked up once per device).
void* scratch_address(int device) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  if (device < 0 || device >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    addr[device] = p;
  }
  return addr[device];
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_noalloc(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* context_lens,
                                 int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                 int block_size, int64_t num_blocks, float scale, int grid_ctas,
                                 int* dev_err, void* stream) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq < 0 || grid_ctas < 0)
    return PA_ERR_SHAPE;
  if (num_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  if (!pa::head_dim_supported(head_dim) || !pa::decode_supported(num_heads, num_kv_heads))
    return PA_ERR_UNSUPPORTED;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !context_lens) return PA_ERR_NULL;
  if (max_blocks_per_seq > 0 && !block_tables) return PA_ERR_NULL;
  if (((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) |
        reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) &
       15) != 0)
    return PA_ERR_ALIGN;
  pa::DeviceInfo info;
  if (!pa::current_device_info(&info)) return PA_ERR_CUDA;
  const bool auto_grid = grid_ctas == 0;
  if (auto_grid) grid_ctas = info.num_sms;
  if (grid_ctas > pa::decode_max_ctas(info)) return PA_ERR_SHAPE;
  // the partial-result slots are indexed by CTA, so size them for this grid only
  size_t off_c, off_l, off_o, total;
  pa::decode_workspace_layout(num_seqs, num_heads, num_kv_heads, grid_ctas, &off_c, &off_l,
                              &off_o, &total);
  if (total > pa::kScratchBytes) return PA_ERR_WORKSPACE;  // beyond the fixed scratch
  unsigned char* ws = static_cast<unsigned char*>(pa::scratch_address(info.device));
  if (ws == nullptr) return PA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The arrival counters must start at zero; the array keeps whatever the last call left.
  if (cudaMemsetAsync(ws + off_c, 0, (size_t)num_seqs * num_kv_heads * sizeof(int), st) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  pa::DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  float s = scale;
  if (!(s > 0.f) || isnan(s)) s = 1.0f / sqrtf((float)head_dim);
  a.scale_log2 = s * 1.4426950408889634f;
  a.grid_ctas = grid_ctas;
  a.min_tiles = auto_grid ? pa::kDecodeMinTilesPerCta : 1;
  a.counters = reinterpret_cast<int*>(ws + off_c);
  a.part_lse = reinterpret_cast<float*>(ws + off_l);
  a.part_o = reinterpret_cast<float*>(ws + off_o);
  a.dev_err = dev_err;
  a.head_dim = head_dim;
  a.f16 = 0;  // bf16
  return pa::launch_decode(a, info, st);
}
