// prefill.cu — chunked (varlen, causal) prefill attention over the paged cache on the
// tcgen05 tensor cores.
//
// What it computes ("nano-vllm解读", section "如何适配不同请求不同序列长度"; "3.6 ModelRunner、
// CUDA Graph 与性能基准", section 2): for sequence s with n_s new tokens (rows
// cu_seqlens_q[s]..) and k_s = cu_seqlens_k[s+1]-cu_seqlens_k[s] keys (c_s = k_s - n_s cached
// ones first), new token i sits at absolute position c_s + i and attends, per query head
// h, over keys t <= c_s + i (causal) or all k_s keys, read through block_tables[s]:
// o = softmax(scale * q K^T) V.
//
// GB300 design (one CTA per (KV head j, sequence s, 128-row query tile)):
//  * The 128 rows of a query tile are 128/G positions x the G query heads of KV group j
//    (G = H/H_kv), so every K/V tile fetched for the group serves all of its heads.
//  * TMA: K and V are described by 4-D tensor maps over [num_blocks, block_size, H_kv, D];
//    a box of (64 dims x 1 head x R rows x 1 block), 128-byte swizzled, takes the
//    physical block id straight from the block table as a coordinate, so a 128-key tile is
//    2 boxes (R = 128 when block_size >= 128) or 2*(128/block_size) boxes.
//  * tcgen05.mma (kind::f16, bf16 operands, fp32 accumulators in tensor memory):
//    S = Q K^T (A = Q, B = K, both K-major) into one of two S buffers (256 columns), then
//    O += P V (A = P in shared memory, B = V MN-major) into O (128 columns). One elected
//    thread issues all MMAs; completion reaches the other warps through tcgen05.commit
//    on mbarriers. While the softmax warps work on S(i), the tensor core already runs
//    S(i+1).
//  * Softmax: 4 warps, thread r owns row r (TMEM lane r): scores are masked by key index
//    (causal and length), the running max is only moved when it grows by more than 2^8
//    (then O is rescaled in tensor memory), P is written to shared memory as bf16 in the
//    128-byte-swizzled K-major layout the MMA reads. Rows past the sequence length of the
//    last V tile are zeroed so stale or poisoned rows never meet a zero probability.
//  * Every wait is bounded; on a timeout the kernel records PA_DEV_ERR_TIMEOUT, runs to
//    the end of its protocol and frees its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "umma.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;          // query rows per CTA (TMEM lanes)
constexpr int kKeys = 128;          // keys per K/V tile
constexpr int kHalfBytes = 128 * 128;  // one 64-dim (or 64-key) column block: 128 rows x 128 B
constexpr int kTileBytes = 2 * kHalfBytes;  // 32 KB: a 128 x 128 bf16 tile
constexpr int kThreads = 192;       // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows 256x

struct PrefillSmem {
  // 1024-byte aligned tiles (128-byte swizzle atoms are 1024 bytes)
  unsigned char q[kTileBytes];
  unsigned char k[2][kTileBytes];
  unsigned char v[2][kTileBytes];
  unsigned char p[kTileBytes];
  uint64_t q_full;
  uint64_t k_full[2];
  uint64_t v_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_done;
  uint32_t tmem_base;
  int abort;
};

// Byte offset of 16-byte chunk `chunk` (0..15) of row `row` in a 128 x 128 bf16 tile stored
// as two 128-byte-swizzled column blocks (chunks 0..7 and 8..15).
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * kHalfBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void note_timeout(PrefillSmem& sm, int* dev_err) {
  sm.abort = 1;
  set_dev_err(dev_err, PA_DEV_ERR_TIMEOUT);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  constexpr int P = kRows / G;  // query positions per CTA
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int j = blockIdx.x;  // KV head
  const int s = blockIdx.y;  // sequence
  const int qt = (int)gridDim.z - 1 - (int)blockIdx.z;  // heaviest (latest) tiles first
  const int H = a.num_heads;

  // ---- sequence shape (uniform over the CTA) ------------------------------------------
  const int q0 = __ldg(a.cu_seqlens_q + s);
  const int n = __ldg(a.cu_seqlens_q + s + 1) - q0;
  const int kv_len = __ldg(a.cu_seqlens_k + s + 1) - __ldg(a.cu_seqlens_k + s);
  const int c_len = kv_len - n;
  const int cap = a.max_blocks * a.block_size;
  if (n < 0 || c_len < 0 || kv_len > cap) {
    if (tid == 0 && qt == 0 && j == 0) set_dev_err(a.dev_err, PA_DEV_ERR_SEQLENS);
    return;
  }
  if (n > a.max_seqlen_q && tid == 0 && qt == 0 && j == 0) set_dev_err(a.dev_err, PA_DEV_ERR_SEQLENS);
  const int i0 = qt * P;
  if (i0 >= n) return;  // nothing to do (before any barrier or tensor memory)
  const int rows_valid = min(P, n - i0);
  const int n_keys = a.causal ? (c_len + i0 + rows_valid) : kv_len;
  const int n_tiles = (n_keys + kKeys - 1) / kKeys;

  if (tid == 0) {
    mbar_init(&sm.q_full, 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.k_full[b], 1);
      mbar_init(&sm.v_full[b], 1);
      mbar_init(&sm.kv_empty[b], 1);
      mbar_init(&sm.s_full[b], 1);
    }
    mbar_init(&sm.p_full, 128);
    mbar_init(&sm.o_done, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    umma::tmem_alloc(&sm.tmem_base, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      umma::prefetch_tmap(&tm_k);
      umma::prefetch_tmap(&tm_v);
      const int bs = a.block_size;
      const int box_rows = bs < kKeys ? bs : kKeys;
      const int boxes = kKeys / box_rows;
      const int32_t* table = a.block_tables + (int64_t)s * a.max_blocks;
      for (int it = 0; it < n_tiles; ++it) {
        const int st = it & 1;
        if (it >= 2 && !mbar_wait(&sm.kv_empty[st], (uint32_t)(((it >> 1) - 1) & 1), abort_flag))
          note_timeout(sm, a.dev_err);
        const int t0 = it * kKeys;
        int blk[kKeys / 8];  // at most 16 boxes (block_size 8)
        uint32_t bytes = 0;
        for (int bx = 0; bx < boxes; ++bx) {
          const int key0 = t0 + bx * box_rows;
          blk[bx] = -1;
          if (key0 < kv_len) {
            const int id = __ldg(table + key0 / bs);
            if (id >= 0 && (int64_t)id < a.num_blocks) {
              blk[bx] = id;
              bytes += 2u * box_rows * 128u;
            } else {
              set_dev_err(a.dev_err, PA_DEV_ERR_BLOCK_ID);
            }
          }
        }
        const int row0 = (bs > kKeys) ? (t0 % bs) : 0;
        mbar_arrive_expect_tx(&sm.k_full[st], bytes);
        for (int bx = 0; bx < boxes; ++bx) {
          if (blk[bx] < 0) continue;
          for (int h2 = 0; h2 < 2; ++h2)
            umma::tma_load_4d(sm.k[st] + h2 * kHalfBytes + bx * box_rows * 128, &tm_k, h2 * 64, j,
                              row0, blk[bx], &sm.k_full[st]);
        }
        mbar_arrive_expect_tx(&sm.v_full[st], bytes);
        for (int bx = 0; bx < boxes; ++bx) {
          if (blk[bx] < 0) continue;
          for (int h2 = 0; h2 < 2; ++h2)
            umma::tma_load_4d(sm.v[st] + h2 * kHalfBytes + bx * box_rows * 128, &tm_v, h2 * 64, j,
                              row0, blk[bx], &sm.v_full[st]);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma::idesc_bf16_f32(kRows, kKeys, false);
      constexpr uint32_t idesc_o = umma::idesc_bf16_f32(kRows, 128, true);
      const uint32_t q_addr = smem_u32(sm.q);
      const uint32_t p_addr = smem_u32(sm.p);
      if (!mbar_wait(&sm.q_full, 0, abort_flag)) note_timeout(sm, a.dev_err);
      umma::fence_after_sync();
      auto issue_pv = [&](int it) {
        const int st = it & 1;
        if (!mbar_wait(&sm.p_full, (uint32_t)(it & 1), abort_flag)) note_timeout(sm, a.dev_err);
        if (!mbar_wait(&sm.v_full[st], (uint32_t)((it >> 1) & 1), abort_flag))
          note_timeout(sm, a.dev_err);
        umma::fence_after_sync();
        const uint32_t v_addr = smem_u32(sm.v[st]);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t ad = umma::smem_desc(p_addr + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = umma::smem_desc(v_addr + kk * 16 * 128, kHalfBytes, 1024);
          umma::mma_bf16(tmem + kColO, ad, bd, idesc_o, (it > 0) || (kk > 0));
        }
        umma::commit(&sm.kv_empty[st]);
        umma::commit(&sm.o_done);
      };
      for (int it = 0; it < n_tiles; ++it) {
        const int st = it & 1;
        if (!mbar_wait(&sm.k_full[st], (uint32_t)((it >> 1) & 1), abort_flag))
          note_timeout(sm, a.dev_err);
        umma::fence_after_sync();
        const uint32_t k_addr = smem_u32(sm.k[st]);
        const uint32_t s_col = (it & 1) ? kColS1 : kColS0;
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          const uint64_t ad = umma::smem_desc(q_addr + off, 16, 1024);
          const uint64_t bd = umma::smem_desc(k_addr + off, 16, 1024);
          umma::mma_bf16(tmem + s_col, ad, bd, idesc_s, kk > 0);
        }
        umma::commit(&sm.s_full[it & 1]);
        if (it > 0) issue_pv(it - 1);
      }
      issue_pv(n_tiles - 1);
      // the last commit must land before tensor memory is released
      if (!mbar_wait(&sm.o_done, (uint32_t)((n_tiles - 1) & 1), abort_flag))
        note_timeout(sm, a.dev_err);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int r = tid;  // row == TMEM lane
    const int pos = r / G, hh = r % G;
    const int qi = i0 + pos;             // new-token index within the sequence
    const bool row_ok = qi < n;
    const int qpos = c_len + qi;         // absolute position of this query row
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);

    // Q row -> shared memory (128-byte swizzled, K-major)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(a.q) + ((int64_t)(q0 + qi) * H + j * G + hh) * kHeadDim);
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 v = row_ok ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sm.q + sw128_offset(r, ch)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.q_full);
    }

    float m_run = -INFINITY, l_run = 0.f;
    float sv[kKeys];
    for (int it = 0; it < n_tiles; ++it) {
      const int buf = it & 1;
      if (!mbar_wait(&sm.s_full[buf], (uint32_t)((it >> 1) & 1), abort_flag))
        note_timeout(sm, a.dev_err);
      umma::fence_after_sync();
      const uint32_t s_col = buf ? kColS1 : kColS0;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) umma::tmem_ld32(lane_addr + s_col + 32 * c4, sv + 32 * c4);
      umma::tmem_ld_wait();

      const int t0 = it * kKeys;
      const int lim = a.causal ? min(kv_len, qpos + 1) : kv_len;  // keys [t0, lim) count
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        const float x = (t0 + c < lim) ? sv[c] * a.scale_log2 : -INFINITY;
        sv[c] = x;
        mt = fmaxf(mt, x);
      }
      float m_use, alpha;
      bool rescale = false;
      if (it == 0) {
        m_use = mt;
        alpha = 0.f;
      } else if (mt > m_run + kRescaleThreshold) {
        m_use = mt;
        alpha = fast_exp2(m_run - mt);
        rescale = true;
      } else {
        m_use = m_run;
        alpha = 1.f;
      }
      const float m_safe = (m_use == -INFINITY) ? 0.f : m_use;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        const float p = fast_exp2(sv[c] - m_safe);
        sv[c] = p;
        rs += p;
      }
      l_run = l_run * alpha + rs;
      m_run = m_use;

      // O and the P buffer belong to PV(it-1) until it completes
      if (it > 0) {
        if (!mbar_wait(&sm.o_done, (uint32_t)((it - 1) & 1), abort_flag))
          note_timeout(sm, a.dev_err);
        umma::fence_after_sync();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        float ob[32];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          umma::tmem_ld32(lane_addr + kColO + 32 * c4, ob);
          umma::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ob[e] *= alpha;
          umma::tmem_st32(lane_addr + kColO + 32 * c4, ob);
        }
        umma::tmem_st_wait();
      }
      // rows of the last V tile beyond the sequence: zero them (never multiply a stale row)
      if (t0 + kKeys > kv_len) {
        const int st = it & 1;
        if (!mbar_wait(&sm.v_full[st], (uint32_t)((it >> 1) & 1), abort_flag))
          note_timeout(sm, a.dev_err);
        if (r >= kv_len - t0) {
#pragma unroll
          for (int ch = 0; ch < 16; ++ch)
            *reinterpret_cast<uint4*>(sm.v[st] + (ch >> 3) * kHalfBytes + r * 128 + (ch & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // P row (bf16) -> shared memory, 128-byte swizzled K-major
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        uint4 pk;
        pk.x = f32x2_to_bf16x2(sv[8 * ch + 0], sv[8 * ch + 1]);
        pk.y = f32x2_to_bf16x2(sv[8 * ch + 2], sv[8 * ch + 3]);
        pk.z = f32x2_to_bf16x2(sv[8 * ch + 4], sv[8 * ch + 5]);
        pk.w = f32x2_to_bf16x2(sv[8 * ch + 6], sv[8 * ch + 7]);
        *reinterpret_cast<uint4*>(sm.p + sw128_offset(r, ch)) = pk;
      }
      fence_proxy_async_smem();
      umma::fence_before_sync();
      mbar_arrive(&sm.p_full);
    }

    // ---- epilogue: O / l -> bf16 rows ------------------------------------------------
    if (!mbar_wait(&sm.o_done, (uint32_t)((n_tiles - 1) & 1), abort_flag))
      note_timeout(sm, a.dev_err);
    umma::fence_after_sync();
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                          ((int64_t)(q0 + qi) * H + j * G + hh) * kHeadDim);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      float ob[32];
      umma::tmem_ld32(lane_addr + kColO + 32 * c4, ob);
      umma::tmem_ld_wait();
      if (row_ok) {
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          uint4 pk;
          pk.x = f32x2_to_bf16x2(ob[8 * q8 + 0] * inv, ob[8 * q8 + 1] * inv);
          pk.y = f32x2_to_bf16x2(ob[8 * q8 + 2] * inv, ob[8 * q8 + 3] * inv);
          pk.z = f32x2_to_bf16x2(ob[8 * q8 + 4] * inv, ob[8 * q8 + 5] * inv);
          pk.w = f32x2_to_bf16x2(ob[8 * q8 + 6] * inv, ob[8 * q8 + 7] * inv);
          dst[c4 * 4 + q8] = pk;
        }
      }
    }
  }

  // ---- teardown: every role is done with tensor memory ----------------------------------
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_cache_map(CUtensorMap* map, const void* base, int num_kv_heads, int block_size,
                    int64_t num_blocks) {
  auto encode = get_encode();
  if (!encode) return false;
  const int box_rows = block_size < kKeys ? block_size : kKeys;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)num_kv_heads, (cuuint64_t)block_size,
                        (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)num_kv_heads * kHeadDim * 2,
                           (cuuint64_t)block_size * num_kv_heads * kHeadDim * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult rc = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                       strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

template <int G>
int launch_prefill_t(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                     const CUtensorMap& mk, const CUtensorMap& mv) {
  constexpr int P = kRows / G;
  const size_t smem = sizeof(PrefillSmem) + 1024;
  static bool attr_done[64] = {false};
  if (info.device < 0 || info.device >= 64) return PA_ERR_CUDA;
  if (!attr_done[info.device]) {
    if (cudaFuncSetAttribute(paged_prefill_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[info.device] = true;
  }
  const int q_tiles = (a.max_seqlen_q + P - 1) / P;
  if (q_tiles > 65535) return PA_ERR_UNSUPPORTED;
  dim3 grid((unsigned)a.num_kv_heads, (unsigned)a.num_seqs, (unsigned)q_tiles);
  paged_prefill_kernel<G><<<grid, kThreads, smem, stream>>>(mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

bool prefill_supported(int num_heads, int num_kv_heads, int block_size) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return false;
  const int g = num_heads / num_kv_heads;
  if (!(g == 1 || g == 2 || g == 4 || g == 8)) return false;
  if (block_size % kKeys == 0) return true;
  return block_size >= 8 && block_size % 8 == 0 && kKeys % block_size == 0;
}

int launch_prefill(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  if (a.num_seqs > 65535 || a.max_seqlen_q <= 0) return PA_ERR_UNSUPPORTED;
  CUtensorMap mk, mv;
  if (!make_cache_map(&mk, a.k_cache, a.num_kv_heads, a.block_size, a.num_blocks) ||
      !make_cache_map(&mv, a.v_cache, a.num_kv_heads, a.block_size, a.num_blocks))
    return PA_ERR_CUDA;
  switch (a.num_heads / a.num_kv_heads) {
    case 1: return launch_prefill_t<1>(a, info, stream, mk, mv);
    case 2: return launch_prefill_t<2>(a, info, stream, mk, mv);
    case 4: return launch_prefill_t<4>(a, info, stream, mk, mv);
    case 8: return launch_prefill_t<8>(a, info, stream, mk, mv);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace pa
