// tensor_map.h — host-side construction of the TMA tensor maps: over the paged K/V caches,
// and over the prefill's q.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace pa {

// cuTensorMapEncodeTiled from the driver (null if the driver does not export it).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn();

// A 4-D map over one cache [num_blocks, block_size, num_kv_heads, head_dim] of 16-bit
// elements, walked as (dim, token in block, KV head, block): a box of 64 dims x box_tokens
// tokens x box_heads heads lands in shared memory as [head][token][64 dims], 128-byte rows
// with the 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)). Returns false
// if the driver rejects the map.
bool make_slab_map(CUtensorMap* map, const void* base, int num_kv_heads, int head_dim, bool f16,
                   int block_size, int64_t num_blocks, int box_tokens, int box_heads);

// A 3-D map over a [rows, num_heads, head_dim] tensor of 16-bit elements (q or out of the
// prefill), walked as (dim, head, row): a box of 64 dims x box_heads heads x box_rows rows
// lands in shared memory as [row][head][64 dims], 128-byte rows with the 128-byte swizzle.
// Boxes reaching past `rows` read zeros there. Returns false if the driver rejects the map.
bool make_rows_map(CUtensorMap* map, const void* base, int64_t rows, int num_heads,
                   int head_dim, bool f16, int box_heads, int box_rows);

}  // namespace pa
