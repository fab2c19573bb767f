// tensor_map.h — host-side construction of the TMA tensor maps over the paged K/V caches.
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

}  // namespace pa
