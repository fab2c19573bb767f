// staged_write.cu — apply a packed batch of row-run writes to a device-resident 2-D tensor.
//
// "Model Runner V2 设计文档", section "4. StagedWriteTensor": a large tensor such as the
// block tables stays on the GPU; the host stages only the changed runs (row, start column,
// values), packs them into one contiguous buffer, copies that buffer once, and one kernel
// applies the runs. No full host-to-device copy of the tensor and no synchronisation.
//
// Design: one thread per staged value (flat grid, capped at 8 CTAs per SM, grid-stride).
// The run holding value v is the last w with offsets[w] <= v (binary search over the run
// offsets, which stay in L1/L2), so runs of any length mix balance over the grid. Each
// run is checked against the tensor once per value; a run that leaves the tensor, or
// offsets that decrease, is skipped and flagged, never written out of bounds.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

template <typename T>
__global__ void __launch_bounds__(256) staged_write_kernel(
    T* __restrict__ base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
    const int32_t* __restrict__ rows, const int32_t* __restrict__ starts,
    const int32_t* __restrict__ offsets, const T* __restrict__ values, int num_writes,
    int64_t num_values, int* dev_err) {
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < num_values;
       v += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = num_writes - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)__ldg(offsets + mid) <= v) lo = mid;
      else hi = mid - 1;
    }
    const int64_t o0 = __ldg(offsets + lo);
    const int64_t o1 = __ldg(offsets + lo + 1);
    if (v < o0 || v >= o1) {  // only when the offsets are not non-decreasing
      set_dev_err(dev_err, PA_DEV_ERR_STAGED);
      continue;
    }
    const int64_t r = __ldg(rows + lo);
    const int64_t s = __ldg(starts + lo);
    if (r < 0 || r >= num_rows || s < 0 || s + (o1 - o0) > num_cols) {
      if (v == o0) set_dev_err(dev_err, PA_DEV_ERR_STAGED);
      continue;
    }
    base[r * row_stride + s + (v - o0)] = __ldg(values + v);
  }
}

int launch_staged_write(void* base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
                        int elem_bytes, const int32_t* rows, const int32_t* starts,
                        const int32_t* offsets, const void* values, int num_writes,
                        int64_t num_values, int* dev_err, cudaStream_t stream, int num_sms) {
  const int threads = 256;
  int64_t blocks = (num_values + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  const unsigned g = (unsigned)blocks;
  switch (elem_bytes) {
    case 1:
      staged_write_kernel<uint8_t><<<g, threads, 0, stream>>>(
          static_cast<uint8_t*>(base), num_rows, num_cols, row_stride, rows, starts, offsets,
          static_cast<const uint8_t*>(values), num_writes, num_values, dev_err);
      break;
    case 2:
      staged_write_kernel<uint16_t><<<g, threads, 0, stream>>>(
          static_cast<uint16_t*>(base), num_rows, num_cols, row_stride, rows, starts, offsets,
          static_cast<const uint16_t*>(values), num_writes, num_values, dev_err);
      break;
    case 4:
      staged_write_kernel<uint32_t><<<g, threads, 0, stream>>>(
          static_cast<uint32_t*>(base), num_rows, num_cols, row_stride, rows, starts, offsets,
          static_cast<const uint32_t*>(values), num_writes, num_values, dev_err);
      break;
    case 8:
      staged_write_kernel<uint64_t><<<g, threads, 0, stream>>>(
          static_cast<uint64_t*>(base), num_rows, num_cols, row_stride, rows, starts, offsets,
          static_cast<const uint64_t*>(values), num_writes, num_values, dev_err);
      break;
    default:
      return PA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
