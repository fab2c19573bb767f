// staged_write.cu — apply a packed batch of row-run writes to a device-resident 2-D tensor.
//
// "Model Runner V2 设计文档", section "4. StagedWriteTensor": a large tensor such as the
// block tables stays on the GPU; the host stages only the changed runs (row, start column,
// values), packs them into one contiguous buffer, copies that buffer once, and one kernel
// applies the runs. No full host-to-device copy of the tensor and no synchronisation.
//
// Design: one thread per staged value (flat grid, capped at 8 CTAs per SM, grid-stride).
// The run holding value v is the last w with offsets[w] <= v: a binary search over the run
// offsets, staged in shared memory when there are at most 8192 runs (32 KB), so runs of
// any length mix balance over the grid. Each
// run is checked against the tensor once per value; a run that leaves the tensor, or
// offsets that decrease, is skipped and flagged, never written out of bounds.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <numeric>
#include <vector>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

// Run offsets up to this many entries are staged in shared memory first (one coalesced
// pass), so the binary search costs shared-memory reads instead of dependent global loads.
constexpr int kSmemOffsets = 8192;

template <typename T, bool SMEM>
__global__ void __launch_bounds__(256) staged_write_kernel(
    T* __restrict__ base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
    const int32_t* __restrict__ rows, const int32_t* __restrict__ starts,
    const int32_t* __restrict__ offsets, const T* __restrict__ values, int num_writes,
    int64_t num_values, int* dev_err) {
  extern __shared__ int32_t s_off[];
  if constexpr (SMEM) {
    for (int i = threadIdx.x; i <= num_writes; i += blockDim.x) s_off[i] = __ldg(offsets + i);
    __syncthreads();
  }
  const int32_t* off = SMEM ? s_off : offsets;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < num_values;
       v += (int64_t)gridDim.x * blockDim.x) {
    // the run holding value v: the last w with offsets[w] <= v
    int lo = 0, hi = num_writes - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)off[mid] <= v) lo = mid;
      else hi = mid - 1;
    }
    const int64_t o0 = off[lo];
    const int64_t o1 = off[lo + 1];
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

template <typename T>
void launch_staged_t(unsigned g, size_t smem, cudaStream_t stream, void* base, int64_t num_rows,
                     int64_t num_cols, int64_t row_stride, const int32_t* rows,
                     const int32_t* starts, const int32_t* offsets, const void* values,
                     int num_writes, int64_t num_values, int* dev_err) {
  if (smem)
    staged_write_kernel<T, true><<<g, 256, smem, stream>>>(
        static_cast<T*>(base), num_rows, num_cols, row_stride, rows, starts, offsets,
        static_cast<const T*>(values), num_writes, num_values, dev_err);
  else
    staged_write_kernel<T, false><<<g, 256, 0, stream>>>(
        static_cast<T*>(base), num_rows, num_cols, row_stride, rows, starts, offsets,
        static_cast<const T*>(values), num_writes, num_values, dev_err);
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
  const size_t smem = num_writes + 1 <= kSmemOffsets ? (size_t)(num_writes + 1) * 4 : 0;
  switch (elem_bytes) {
    case 1: launch_staged_t<uint8_t>(g, smem, stream, base, num_rows, num_cols, row_stride, rows,
                                     starts, offsets, values, num_writes, num_values, dev_err);
      break;
    case 2: launch_staged_t<uint16_t>(g, smem, stream, base, num_rows, num_cols, row_stride, rows,
                                      starts, offsets, values, num_writes, num_values, dev_err);
      break;
    case 4: launch_staged_t<uint32_t>(g, smem, stream, base, num_rows, num_cols, row_stride, rows,
                                      starts, offsets, values, num_writes, num_values, dev_err);
      break;
    case 8: launch_staged_t<uint64_t>(g, smem, stream, base, num_rows, num_cols, row_stride, rows,
                                      starts, offsets, values, num_writes, num_values, dev_err);
      break;
    default:
      return PA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_staged_upload_apply(void* base, int64_t num_rows, int64_t num_cols,
                               int64_t row_stride, int elem_bytes, const void* packed_host,
                               void* packed_dev, const pa_staged_layout* lay, int* dev_err,
                               cudaStream_t stream, int num_sms) {
  if (cudaMemcpyAsync(packed_dev, packed_host, (size_t)lay->bytes, cudaMemcpyHostToDevice,
                      stream) != cudaSuccess)
    return PA_ERR_CUDA;
  if (lay->num_values == 0) return PA_OK;
  unsigned char* d = static_cast<unsigned char*>(packed_dev);
  return launch_staged_write(base, num_rows, num_cols, row_stride, elem_bytes,
                             reinterpret_cast<const int32_t*>(d + lay->rows_offset),
                             reinterpret_cast<const int32_t*>(d + lay->starts_offset),
                             reinterpret_cast<const int32_t*>(d + lay->offsets_offset),
                             d + lay->values_offset, lay->num_writes, lay->num_values, dev_err,
                             stream, num_sms);
}

// ---------------------------------------------------------------- host staging
// Packed buffer: int32 rows[W], starts[W], offsets[W+1], then (16-byte aligned) the values.
static int64_t staged_values_offset(int64_t num_writes) {
  return (4 * (3 * num_writes + 1) + 15) / 16 * 16;
}

}  // namespace pa

extern "C" size_t pa_staged_pack_bound(int num_writes, int64_t num_values, int elem_bytes) {
  if (num_writes < 0 || num_values < 0 || elem_bytes <= 0) return 0;
  return (size_t)(pa::staged_values_offset(num_writes) + num_values * elem_bytes);
}

// Merge the staged writes of each row into disjoint runs (later writes win where they
// overlap; overlapping or touching writes join into one run) and pack the runs.
extern "C" int pa_staged_pack(const int32_t* rows, const int32_t* starts, const int32_t* lens,
                              const void* values, int num_writes, int elem_bytes, void* packed,
                              size_t packed_bytes, pa_staged_layout* layout) {
  if (!layout) return PA_ERR_NULL;
  if (num_writes < 0) return PA_ERR_SHAPE;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return PA_ERR_UNSUPPORTED;
  if (num_writes > 0 && (!rows || !starts || !lens)) return PA_ERR_NULL;
  std::vector<int64_t> src(num_writes + 1, 0);  // first value of each staged write
  for (int w = 0; w < num_writes; ++w) {
    if (lens[w] < 0 || starts[w] < 0) return PA_ERR_SHAPE;
    src[w + 1] = src[w] + lens[w];
  }
  if (src[num_writes] > 0 && !values) return PA_ERR_NULL;
  // the writes of each row in order of start column, staging order among equal starts
  std::vector<int> order;
  order.reserve(num_writes);
  for (int w = 0; w < num_writes; ++w)
    if (lens[w] > 0) order.push_back(w);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    return rows[a] != rows[b] ? rows[a] < rows[b] : starts[a] < starts[b];
  });
  // components: maximal groups of overlapping or touching writes of one row
  struct Run { int32_t row, start; int64_t len; int first, last; };
  std::vector<Run> runs;
  for (size_t i = 0; i < order.size();) {
    const int w0 = order[i];
    Run r{rows[w0], starts[w0], (int64_t)lens[w0], (int)i, (int)i};
    int64_t hi = (int64_t)starts[w0] + lens[w0];
    size_t j = i + 1;
    while (j < order.size() && rows[order[j]] == r.row && starts[order[j]] <= hi) {
      hi = std::max(hi, (int64_t)starts[order[j]] + lens[order[j]]);
      ++j;
    }
    r.len = hi - r.start;
    r.last = (int)j - 1;
    if (r.len > INT32_MAX) return PA_ERR_UNSUPPORTED;
    runs.push_back(r);
    i = j;
  }
  const int64_t W = (int64_t)runs.size();
  int64_t total = 0;
  for (const Run& r : runs) total += r.len;
  if (total > INT32_MAX || W > INT32_MAX) return PA_ERR_UNSUPPORTED;
  const int64_t voff = pa::staged_values_offset(W);
  const int64_t need = voff + total * elem_bytes;
  layout->rows_offset = 0;
  layout->starts_offset = 4 * W;
  layout->offsets_offset = 8 * W;
  layout->values_offset = voff;
  layout->num_writes = (int32_t)W;
  layout->num_values = total;
  layout->bytes = need;
  if (!packed || packed_bytes < (size_t)need) return PA_ERR_WORKSPACE;
  unsigned char* out = static_cast<unsigned char*>(packed);
  int32_t* o_rows = reinterpret_cast<int32_t*>(out);
  int32_t* o_starts = o_rows + W;
  int32_t* o_offs = o_starts + W;
  unsigned char* o_vals = out + voff;
  const unsigned char* in = static_cast<const unsigned char*>(values);
  int64_t at = 0;
  std::vector<int> members;
  for (int64_t k = 0; k < W; ++k) {
    const Run& r = runs[k];
    o_rows[k] = r.row;
    o_starts[k] = r.start;
    o_offs[k] = (int32_t)at;
    if (r.first == r.last) {
      const int w = order[r.first];
      memcpy(o_vals + at * elem_bytes, in + src[w] * elem_bytes, (size_t)lens[w] * elem_bytes);
    } else {
      // every column of the run is covered; apply its writes in staging order
      members.assign(order.begin() + r.first, order.begin() + r.last + 1);
      std::sort(members.begin(), members.end());
      for (int w : members)
        memcpy(o_vals + (at + (starts[w] - r.start)) * elem_bytes, in + src[w] * elem_bytes,
               (size_t)lens[w] * elem_bytes);
    }
    at += r.len;
  }
  o_offs[W] = (int32_t)at;
  return PA_OK;
}
