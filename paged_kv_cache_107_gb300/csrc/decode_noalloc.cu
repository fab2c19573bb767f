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
// the device address is looked up with cudaGetSymbolAddress, with the device current, the
// first time pa_decode_noalloc runs in a CUDA context (once per device, unless the context
// is destroyed and recreated, e.g. by cudaDeviceReset, which reloads the module and may move
// the array; the next call then looks it up again). That first call should therefore come
// before any stream capture. Nothing here calls cudaMalloc, cudaFree or an allocating
// library routine. Validation and argument packing are pa_decode's (decode_prepare).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB, shared by every call

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent (null if the driver does not export it).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_decode_scratch in the current context of `device`, looked up again
// whenever that device's current context is not the one the cached address came from.
void* scratch_address(int device) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static CUcontext owner[64] = {nullptr};
  if (device < 0 || device >= 64) return nullptr;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr || owner[device] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    addr[device] = p;
    owner[device] = ctx;
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
  pa::DecodeArgs a;
  pa::DeviceInfo info;
  bool nothing = false;
  const int rc = pa::decode_prepare(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    context_lens, num_seqs, num_heads, num_kv_heads, head_dim,
                                    PA_DTYPE_BF16, block_size, num_blocks, scale, grid_ctas,
                                    dev_err, nullptr, &a, &info, &nothing);
  if (rc != PA_OK || nothing) return rc;
  // the partial-result slots are indexed by CTA, so size them for this grid only
  if (pa::decode_bind_workspace(&a, nullptr, a.grid_ctas) > pa::kScratchBytes)
    return PA_ERR_WORKSPACE;  // beyond the fixed scratch
  unsigned char* ws = static_cast<unsigned char*>(pa::scratch_address(info.device));
  if (ws == nullptr) return PA_ERR_CUDA;
  pa::decode_bind_workspace(&a, ws, a.grid_ctas);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The arrival counters must start at zero; the array keeps whatever the last call left.
  if (cudaMemsetAsync(a.counters, 0, (size_t)num_seqs * num_kv_heads * sizeof(int), st) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return pa::launch_decode(a, info, st);
}
