// prefill_kernel.cuh — chunked (varlen, causal) prefill attention over the paged cache on
// the tcgen05 tensor cores: the kernel template (head_dim 64 or 128, bf16 or IEEE fp16).
// prefill.cu instantiates head_dim 128 with bf16; prefill_d*_*.cu the other combinations.
//
// What it computes ("nano-vllm解读", section "如何适配不同请求不同序列长度"; "3.6 ModelRunner、
// CUDA Graph 与性能基准", section 2): for sequence s with n_s new tokens (rows
// cu_seqlens_q[s]..) and k_s = cu_seqlens_k[s+1]-cu_seqlens_k[s] keys (c_s = k_s - n_s cached
// ones first), new token i sits at absolute position c_s + i and attends, per query head
// h, over keys t <= c_s + i (causal) or all k_s keys, read through block_tables[s]:
// o = softmax(scale * q K^T) V.
//
// GB300 design (one CTA per (KV head j, sequence s, pair of 128-row query tiles)):
//  * A 128-row query tile is 128/G positions x the G query heads of KV group j (G = H/H_kv),
//    so every K/V tile fetched for the group serves all of its heads. A CTA holds two such
//    tiles (A: the earlier positions, B: the next ones) that take turns on the tensor core:
//    while one softmax warpgroup works, the other tile's products run.
//  * TMA: K and V are described by 4-D tensor maps over [num_blocks, block_size, H_kv, D];
//    a box of (64 dims x 1 head x R rows x 1 block), 128-byte swizzled, takes the physical
//    block id from the block table as a coordinate. A K/V tile is 128 keys (R = 128 when
//    block_size >= 128, else several blocks). K has a 3-deep ring, V a 2-deep one; K runs
//    one tile ahead of V.
//  * tcgen05.mma (kind::f16, bf16 operands, fp32 accumulators in tensor memory, all 512
//    columns): S_g = Q_g K^T (A = Q and B = K from shared memory, K-major) in 128 columns per
//    tile; the softmax writes P back over S as packed bf16 and O_g += P V reads P straight
//    from tensor memory (B = V, MN-major) into 128 more columns per tile. On the tensor core
//    the order per key tile is PV_A(i), S_A(i+1), PV_B(i), S_B(i+1): each S is issued only
//    after the PV that reads the P it overwrites, and S_g(i) completes after PV_g(i-1), so
//    O_g is stable whenever the softmax sees a new S_g. Key tiles past the causal limit of
//    tile A are not multiplied for A.
//  * Softmax: 8 warps, thread r of a warpgroup owns row r of its tile (TMEM lane r): scores
//    are masked by key index (causal and length) on boundary tiles only, reduced with tree
//    max/sum, the running max is only moved when it grows by more than 2^8 (then O is
//    rescaled in tensor memory), and p = 2^(s*scale - m) comes from one packed fma per pair.
//    Rows of the last V tile past the sequence are zeroed, so stale or poisoned rows never
//    meet a zero probability.
//  * Every wait is bounded; on a timeout the kernel records PA_DEV_ERR_TIMEOUT, runs to
//    the end of its protocol and frees its tensor memory.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "umma.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;                 // query rows per tile (TMEM lanes)
constexpr int kKeys = 128;                 // keys per K/V tile
constexpr int kKStages = 3, kVStages = 2;  // ring depths
constexpr int kHalf = 128 * 128;           // 128 rows x 64 dims: one swizzled column block
constexpr int kThreads = 320;              // warps 0-3 tile A, 4-7 tile B, 8 TMA, 9 MMA
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows 256x

// TMEM columns: S (then P) of tile g at g*128, O of tile g at 256 + g*128.
__host__ __device__ constexpr uint32_t col_s(int g) { return (uint32_t)(g * 128); }
__host__ __device__ constexpr uint32_t col_o(int g) { return (uint32_t)(256 + g * 128); }

// Shared memory of a CTA for head_dim D: tiles of 128 rows x D dims, D/64 swizzled column
// blocks each.
template <int D>
struct PrefillSmem {
  static constexpr int kTile = (D / 64) * kHalf;
  // 1024-byte aligned tiles (128-byte swizzle atoms are 1024 bytes)
  unsigned char q[2][kTile];         // [tile]
  unsigned char k[kKStages][kTile];  // [stage]
  unsigned char v[kVStages][kTile];
  uint64_t q_full;
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];        // S products of that K stage done
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];        // PV products of that V stage done
  uint64_t s_full[2];                // [tile]
  uint64_t p_full[2];
  uint64_t o_done[2];                // the tile's last PV done
  uint32_t tmem_base;
  int abort;
};

template <typename Smem>
__device__ __forceinline__ void note_timeout(Smem& sm, int* dev_err) {
  sm.abort = 1;
  set_dev_err(dev_err, PA_DEV_ERR_TIMEOUT);
}

// Two 16-bit elements packed from an fp32 pair (round to nearest even): bf16 or IEEE fp16.
template <bool F16>
__device__ __forceinline__ uint32_t pack_elt2(float lo, float hi) {
  if constexpr (F16) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  } else {
    return f32x2_to_bf16x2(lo, hi);
  }
}

template <int G, int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  constexpr int P = kRows / G;  // query positions per tile
  constexpr int NH = D / 64;    // 64-dim swizzled column blocks per row
  using Smem = PrefillSmem<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
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
  const int i0 = qt * 2 * P;
  if (i0 >= n) return;  // nothing to do (before any barrier or tensor memory)
  // keys needed by each tile (causal: up to its last position); tile B may be empty
  int n_tiles[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int rows = min(P, n - (i0 + g * P));
    const int keys = rows <= 0 ? 0 : (a.causal ? c_len + i0 + g * P + rows : kv_len);
    n_tiles[g] = (keys + kKeys - 1) / kKeys;
  }
  const int n_all = max(n_tiles[0], n_tiles[1]);

  if (tid == 0) {
    mbar_init(&sm.q_full, 2 * kRows);
    for (int b = 0; b < kKStages; ++b) {
      mbar_init(&sm.k_full[b], 1);
      mbar_init(&sm.k_empty[b], 1);
    }
    for (int b = 0; b < kVStages; ++b) {
      mbar_init(&sm.v_full[b], 1);
      mbar_init(&sm.v_empty[b], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&sm.s_full[g], 1);
      mbar_init(&sm.p_full[g], kRows);
      mbar_init(&sm.o_done[g], 1);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    umma::tmem_alloc(&sm.tmem_base, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      umma::prefetch_tmap(&tm_k);
      umma::prefetch_tmap(&tm_v);
      const int bs = a.block_size;
      const int box_rows = bs < kKeys ? bs : kKeys;
      const int boxes = kKeys / box_rows;
      const int32_t* table = a.block_tables + (int64_t)s * a.max_blocks;
      auto load = [&](bool is_v, int it) {
        const int stages = is_v ? kVStages : kKStages;
        const int st = it % stages;
        uint64_t* empty = is_v ? &sm.v_empty[st] : &sm.k_empty[st];
        uint64_t* full = is_v ? &sm.v_full[st] : &sm.k_full[st];
        if (it >= stages && !mbar_wait(empty, (uint32_t)(((it / stages) - 1) & 1), abort_flag))
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
              bytes += (uint32_t)NH * box_rows * 128u;
            } else if (!is_v) {
              set_dev_err(a.dev_err, PA_DEV_ERR_BLOCK_ID);
            }
          }
        }
        const int row0 = (bs > kKeys) ? (t0 % bs) : 0;
        unsigned char* dst = is_v ? sm.v[st] : sm.k[st];
        const CUtensorMap* map = is_v ? &tm_v : &tm_k;
        mbar_arrive_expect_tx(full, bytes);
        for (int bx = 0; bx < boxes; ++bx) {
          if (blk[bx] < 0) continue;
          for (int h2 = 0; h2 < NH; ++h2)
            umma::tma_load_4d(dst + h2 * kHalf + bx * box_rows * 128, map, h2 * 64, j, row0,
                              blk[bx], full);
        }
      };
      // K runs one tile ahead of V: S(i+1) is issued right after PV(i)
      load(false, 0);
      for (int it = 0; it < n_all; ++it) {
        load(true, it);
        if (it + 1 < n_all) load(false, it + 1);
      }
      // the last copies of every stage land before the CTA may exit (the full limit even
      // after a timeout elsewhere: a copy must not outlive the CTA's shared memory)
      for (int it = n_all > kKStages ? n_all - kKStages : 0; it < n_all; ++it)
        mbar_wait_copies(&sm.k_full[it % kKStages], (uint32_t)((it / kKStages) & 1));
      for (int it = n_all > kVStages ? n_all - kVStages : 0; it < n_all; ++it)
        mbar_wait_copies(&sm.v_full[it % kVStages], (uint32_t)((it / kVStages) & 1));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma::idesc_f32acc(kRows, kKeys, false, F16);
      constexpr uint32_t idesc_o = umma::idesc_f32acc(kRows, D, true, F16);
      auto issue_s = [&](int g, int it) {  // S_g = Q_g K(it)^T
        const uint32_t k_addr = smem_u32(sm.k[it % kKStages]);
        const uint32_t q_addr = smem_u32(sm.q[g]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma::mma_bf16(tmem + col_s(g), umma::smem_desc(q_addr + off, 16, 1024),
                         umma::smem_desc(k_addr + off, 16, 1024), idesc_s, kk > 0);
        }
        umma::commit(&sm.s_full[g]);
      };
      auto issue_pv = [&](int g, int it) {  // O_g += P_g V(it), P_g read from tensor memory
        const uint32_t v_addr = smem_u32(sm.v[it % kVStages]);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma::mma_bf16_ts(tmem + col_o(g), tmem + col_s(g) + kk * 8,
                            umma::smem_desc(v_addr + kk * 16 * 128, kHalf, 1024), idesc_o,
                            (it > 0) || (kk > 0));
        if (it == n_tiles[g] - 1) umma::commit(&sm.o_done[g]);
      };
      auto wait_k = [&](int it) {
        if (!mbar_wait(&sm.k_full[it % kKStages], (uint32_t)((it / kKStages) & 1), abort_flag))
          note_timeout(sm, a.dev_err);
        umma::fence_after_sync();
      };
      if (!mbar_wait(&sm.q_full, 0, abort_flag)) note_timeout(sm, a.dev_err);
      umma::fence_after_sync();
      wait_k(0);
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (n_tiles[g] > 0) issue_s(g, 0);
      umma::commit(&sm.k_empty[0]);
      for (int it = 0; it < n_all; ++it) {
        bool v_ready = false, k_ready = false;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (it >= n_tiles[g]) continue;
          if (!mbar_wait(&sm.p_full[g], (uint32_t)(it & 1), abort_flag)) note_timeout(sm, a.dev_err);
          if (!v_ready) {
            if (!mbar_wait(&sm.v_full[it % kVStages], (uint32_t)((it / kVStages) & 1), abort_flag))
              note_timeout(sm, a.dev_err);
            v_ready = true;
          }
          umma::fence_after_sync();
          issue_pv(g, it);
          if (it + 1 < n_tiles[g]) {
            if (!k_ready) {
              wait_k(it + 1);
              k_ready = true;
            }
            issue_s(g, it + 1);
          }
        }
        umma::commit(&sm.v_empty[it % kVStages]);
        if (k_ready) umma::commit(&sm.k_empty[(it + 1) % kKStages]);
      }
      // the last products must land before tensor memory is released
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (n_tiles[g] > 0 && !mbar_wait(&sm.o_done[g], 0, abort_flag)) note_timeout(sm, a.dev_err);
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int g = warp >> 2;      // query tile of this warpgroup
    const int r = tid & 127;      // row == TMEM lane
    const int wq = warp & 3;      // warp within the warpgroup (TMEM lane quarter)
    const int pos = r / G, hh = r % G;
    const int qi = i0 + g * P + pos;     // new-token index within the sequence
    const bool row_ok = qi < n;
    const int qpos = c_len + qi;         // absolute position of this query row
    const int lim_row = a.causal ? min(kv_len, qpos + 1) : kv_len;  // keys [0, lim_row) count
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const int nt = n_tiles[g];

    // Q row -> shared memory (128-byte swizzled, K-major)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(a.q) + ((int64_t)(q0 + qi) * H + j * G + hh) * D);
      uint4 qv[D / 8];
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) qv[ch] = row_ok ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch)
        *reinterpret_cast<uint4*>(sm.q[g] + (ch >> 3) * kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) =
            qv[ch];
      fence_proxy_async_smem();
      mbar_arrive(&sm.q_full);
    }

    float m_run = -INFINITY, l_run = 0.f;
    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
    for (int it = 0; it < nt; ++it) {
      if (!mbar_wait(&sm.s_full[g], (uint32_t)(it & 1), abort_flag)) note_timeout(sm, a.dev_err);
      umma::fence_after_sync();
      float sv[kKeys];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) umma::tmem_ld32(lane_addr + col_s(g) + 32 * c4, sv + 32 * c4);
      umma::tmem_ld_wait();

      const int t0 = it * kKeys;
      // only tiles that reach past this row's last visible key need a mask
      if (__any_sync(0xffffffffu, t0 + kKeys > lim_row)) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c)
          if (t0 + c >= lim_row) sv[c] = -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mx[c] = sv[c];
#pragma unroll
      for (int c = 8; c < kKeys; ++c) mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
      // the scale is positive, so the max of the scaled scores is the scaled max
      const float mt = a.scale_log2 * fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                            fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
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
      // p = 2^(s*scale - m): one packed fma per pair, then ex2; P packed as 16-bit pairs over
      // S, in the element type of V (the PV product takes both operands in one type)
      const float2 nm2 = make_float2(-m_safe, -m_safe);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < kKeys / 2; ++c) {
        const float2 x = umma::ffma2(make_float2(sv[2 * c], sv[2 * c + 1]), sc2, nm2);
        const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        acc[c & 3] = umma::fadd2(acc[c & 3], p);
        sv[c] = __uint_as_float(pack_elt2<F16>(p.x, p.y));  // c <= 2c: in place is safe
      }
      const float2 t01 = umma::fadd2(acc[0], acc[1]), t23 = umma::fadd2(acc[2], acc[3]);
      const float2 tt = umma::fadd2(t01, t23);
      l_run = l_run * alpha + (tt.x + tt.y);
      m_run = m_use;
      umma::tmem_st32(lane_addr + col_s(g), sv);
      umma::tmem_st32(lane_addr + col_s(g) + 32, sv + 32);
      // O_g is stable here (S_g(it) completed after PV_g(it-1)); PV_g(it) waits for p_full
      if (__any_sync(0xffffffffu, rescale)) {
        float ob[32];
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          umma::tmem_ld32(lane_addr + col_o(g) + 32 * c4, ob);
          umma::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ob[e] *= alpha;
          umma::tmem_st32(lane_addr + col_o(g) + 32 * c4, ob);
        }
      }
      // rows of the last V tile beyond the sequence: zero them (never multiply a stale row)
      if (t0 + kKeys > kv_len) {
        const int st = it % kVStages;
        if (!mbar_wait(&sm.v_full[st], (uint32_t)((it / kVStages) & 1), abort_flag))
          note_timeout(sm, a.dev_err);
        const int first_bad = kv_len - t0;
        if (r >= first_bad) {
#pragma unroll
          for (int ch = 0; ch < D / 8; ++ch)
            *reinterpret_cast<uint4*>(sm.v[st] + (ch >> 3) * kHalf + r * 128 + (ch & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      umma::tmem_st_wait();
      umma::fence_before_sync();
      mbar_arrive(&sm.p_full[g]);
    }

    // ---- epilogue: O / l -> 16-bit rows ----------------------------------------------
    if (nt > 0) {
      if (!mbar_wait(&sm.o_done[g], 0, abort_flag)) note_timeout(sm, a.dev_err);
      umma::fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                            ((int64_t)(q0 + qi) * H + j * G + hh) * D);
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        float ob[32];
        umma::tmem_ld32(lane_addr + col_o(g) + 32 * c4, ob);
        umma::tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint4 pk;
            pk.x = pack_elt2<F16>(ob[8 * q8 + 0] * inv, ob[8 * q8 + 1] * inv);
            pk.y = pack_elt2<F16>(ob[8 * q8 + 2] * inv, ob[8 * q8 + 3] * inv);
            pk.z = pack_elt2<F16>(ob[8 * q8 + 4] * inv, ob[8 * q8 + 5] * inv);
            pk.w = pack_elt2<F16>(ob[8 * q8 + 6] * inv, ob[8 * q8 + 7] * inv);
            dst[c4 * 4 + q8] = pk;
          }
        }
      }
    }
  }

  // ---- teardown: every role is done with tensor memory ----------------------------------
  umma::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int G, int D, bool F16>
int launch_prefill_t(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                     const CUtensorMap& mk, const CUtensorMap& mv) {
  constexpr int P = kRows / G;
  const size_t smem = sizeof(PrefillSmem<D>) + 1024;
  static_assert(sizeof(PrefillSmem<D>) + 1024 <= 227 * 1024, "shared memory budget");
  static std::atomic<bool> attr_done[64];  // zero-initialised: false
  if (info.device < 0 || info.device >= 64) return PA_ERR_CUDA;
  if (!attr_done[info.device].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(paged_prefill_kernel<G, D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[info.device].store(true, std::memory_order_release);
  }
  const int q_tiles = (a.max_seqlen_q + 2 * P - 1) / (2 * P);  // pairs of query tiles
  if (q_tiles > 65535) return PA_ERR_UNSUPPORTED;
  dim3 grid((unsigned)a.num_kv_heads, (unsigned)a.num_seqs, (unsigned)q_tiles);
  paged_prefill_kernel<G, D, F16><<<grid, kThreads, smem, stream>>>(mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Every GQA group size for one (head_dim, element type) combination.
template <int D, bool F16>
int dispatch_prefill(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                     const CUtensorMap& mk, const CUtensorMap& mv) {
  switch (a.num_heads / a.num_kv_heads) {
    case 1: return launch_prefill_t<1, D, F16>(a, info, stream, mk, mv);
    case 2: return launch_prefill_t<2, D, F16>(a, info, stream, mk, mv);
    case 4: return launch_prefill_t<4, D, F16>(a, info, stream, mk, mv);
    case 8: return launch_prefill_t<8, D, F16>(a, info, stream, mk, mv);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace
}  // namespace pa
