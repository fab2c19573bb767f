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
// GB300 design: a persistent grid, one CTA per SM, each walking its own list of work units.
//  * A work unit is (sequence s, KV head j, pair of 128-row query tiles). A 128-row tile is
//    128/G positions x the G query heads of KV group j (G = H/H_kv), so every K/V tile
//    fetched for the group serves all of its heads. The pair's tiles (A: the earlier
//    positions, B: the next ones) take turns on the tensor core: while one softmax
//    warpgroup works, the other tile's products run.
//  * Schedule: every CTA reads cu_seqlens at entry and builds the same list of (sequence,
//    query-tile pair) entries sorted by cost (key tiles, heaviest first) with a bitonic
//    sort in shared memory; the units (entries x KV heads) are dealt to the CTAs in a
//    serpentine (round r runs over CTAs 0..G-1, round r+1 back from G-1), which keeps the
//    per-SM sums of the longest-first order even. Each CTA keeps its own units as records
//    in shared memory. Batches whose bounds (sequences, query-tile pairs, units per CTA)
//    exceed what the in-kernel sort and the records hold run the same code one unit per
//    CTA, on a grid of (KV head, sequence, pair), latest pairs first.
//  * Units follow each other without draining the pipeline: the K/V ring runs on across
//    units, a Q warp copies a tile's next Q (TMA, one box per 64 dims of the tile's 128/G
//    positions x G heads) as soon as the tile's last S product of the current unit has
//    completed, and the next unit's first S products are issued right after the current
//    unit's last P.V products, while the softmax warpgroups write out the finished rows
//    (32-byte stores).
//  * TMA: K and V are described by 4-D tensor maps over [num_blocks, block_size, H_kv, D];
//    a box of (64 dims x 1 head x R rows x 1 block), 128-byte swizzled, takes the physical
//    block id from the block table as a coordinate. A K/V tile is 128 keys (R = 128 when
//    block_size >= 128, else several blocks, one box per block, copied by one lane each).
//    The producer warp reads each tile's block ids two tiles ahead of their first use. K
//    has a 2-deep ring, V a 3-deep one (a V tile waits longest: from its copy to the P.V
//    product of both tiles); K runs one tile ahead of V.
//  * tcgen05.mma (kind::f16, 16-bit operands, fp32 accumulators in tensor memory, all 512
//    columns): S_g = Q_g K^T (A = Q and B = K from shared memory, K-major) in 128 columns per
//    tile; the softmax writes P back over S as packed 16-bit values and O_g += P V reads P
//    straight from tensor memory (B = V, MN-major) into 128 more columns per tile. On the
//    tensor core the order per key tile is PV_A(i), S_A(i+1), PV_B(i), S_B(i+1): each S is
//    issued only after the PV that reads the P it overwrites, and S_g(i) completes after
//    PV_g(i-1), so O_g is stable whenever the softmax sees a new S_g. At head_dim 64 P has
//    columns of its own: S_A(i+1), S_B(i+1) follow the softmax's read of S(i) and come
//    before PV_A(i), PV_B(i); the softmax touches P and O only after the previous PV has
//    landed. Key tiles past the causal limit of tile A are not multiplied for A.
//  * Softmax: 8 warps, thread r of a warpgroup owns row r of its tile (TMEM lane r): scores
//    are masked by key index (causal and length) on boundary tiles only, reduced with tree
//    max/sum, the running max is only moved when it grows by more than 2^8 (then O is
//    rescaled in tensor memory), and p = 2^(s*scale - m) comes from one packed fma per pair.
//    Rows of the last V tile past the sequence are zeroed, so stale or poisoned rows never
//    meet a zero probability.
//  * Every wait is bounded; on a timeout the kernel records PA_DEV_ERR_TIMEOUT, runs to
//    the end of its protocol (the K/V and Q warps still wait for their own copies) and
//    frees its tensor memory.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "tensor_map.h"
#include "umma.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;                 // query rows per tile (TMEM lanes)
constexpr int kKeys = 128;                 // keys per K/V tile
constexpr int kKStages = 2, kVStages = 3;  // ring depths
constexpr int kHalf = 128 * 128;           // 128 rows x 64 dims: one swizzled column block
constexpr int kThreads = 384;  // warps 0-3 tile A, 4-7 tile B, 8 K/V TMA, 9 MMA, 10 Q, 11 idle
constexpr int kTmaWarp = 8, kMmaWarp = 9, kQWarp = 10;
// Registers per thread after the set-up: the softmax warpgroups hold a 128-key score row
// each; the third warpgroup (producers, MMA issuer, an idle warp) needs few. The sums per
// SM sub-partition (one warp of each warpgroup) and per CTA match the launch's 168 x 384.
constexpr int kSoftmaxRegs = 200, kControlRegs = 104;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= 168 * kThreads, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows 256x
// The in-kernel sort is used when the batch has at most kMaxSortSeqs sequences and
// kMaxSortPairs (sequence, query-tile pair) entries and every CTA's share of units fits its
// records; otherwise the plain order.
constexpr int kMaxSortSeqs = 1024;
constexpr int kMaxSortPairs = 2048;
constexpr int kRankSortMax = 512;  // up to this many entries a rank sort, else bitonic

// TMEM columns: S (then P) of tile g at g*128, O of tile g at 256 + g*128. At head_dim 64,
// O takes the first 64 of its 128 columns and P gets the other 64 (320 + g*128), so that
// the next S product may be issued as soon as the softmax has read this one (not after
// this tile's P.V).
__host__ __device__ constexpr uint32_t col_s(int g) { return (uint32_t)(g * 128); }
__host__ __device__ constexpr uint32_t col_o(int g) { return (uint32_t)(256 + g * 128); }
__host__ __device__ constexpr uint32_t col_p(int g) { return (uint32_t)(320 + g * 128); }

// One work unit of a CTA, as a record in shared memory.
struct UnitRec {
  int q0;      // first row of the sequence in q / out
  int n;       // new tokens of the sequence
  int kv_len;  // keys of the sequence (cached + new)
  int s;       // sequence
  int i0;      // first new token of the unit's tile A
  int j;       // KV head
  int vbase;   // K/V tiles of this CTA's earlier units (ring position of the unit's first)
  int nt;      // key tiles of tile A (bits 0..15) and of tile B (bits 16..31; may be 0)
};

// Barriers and schedule state; first in shared memory, then the unit records, then the
// tiles from the next 1024-byte boundary (128-byte swizzle atoms are 1024 bytes).
struct PrefillCtl {
  uint64_t q_full[2];          // [tile] the Q rows of a unit landed
  uint64_t q_empty[2];         // [tile] the last S product of a unit done: Q buffer free
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];  // S products of that K stage done
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];  // PV products of that V stage done
  uint64_t s_full[2];          // [tile]
  uint64_t s_free[2];          // [tile] head_dim 64: the softmax has read its S
  uint64_t p_full[2];
  uint64_t pv_done[2];         // [tile] head_dim 64: a P.V product done (one phase each)
  uint64_t o_done[2];          // the tile's last PV of a unit done
  uint32_t tmem_base;
  int abort;
  int n_units;                 // unit records of this CTA
  int warp_sums[kThreads / 32];
};

template <int D>
struct PrefillTiles {
  static constexpr int kTile = (D / 64) * kHalf;
  unsigned char q[2][kTile];         // [tile]
  unsigned char k[kKStages][kTile];  // [stage]; the schedule is built here at entry
  unsigned char v[kVStages][kTile];
};

constexpr int kCtlBytes = 256;
constexpr int kRecBytes = 1792;  // fills the opt-in limit at head_dim 128 with the slack below
// (56 records)
constexpr int kMaxUnitRecs = kRecBytes / (int)sizeof(UnitRec);
static_assert(sizeof(PrefillCtl) <= kCtlBytes, "control block");

template <int D>
constexpr size_t prefill_smem_bytes() {
  return 1023 /* alignment of the tiles */ + kCtlBytes + kRecBytes + sizeof(PrefillTiles<D>);
}

// Rows of q that the Q tensor map spans (a bound on the batch's tokens known to the host).
__host__ __device__ inline int64_t q_map_rows(const PrefillArgs& a) {
  const int64_t r = (int64_t)a.num_seqs * a.max_seqlen_q;
  return r < INT32_MAX ? r : INT32_MAX;
}

__device__ __forceinline__ void note_timeout(PrefillCtl& c, int* dev_err) {
  c.abort = 1;
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

// true in one lane of the (fully active) warp: the lowest
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// 16-byte global -> shared copy (cp.async, cached in L2 only); src_bytes 0 writes 16 zeros.
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Serpentine deal: the k-th unit of CTA c among G CTAs is entry k*G + c (k even) or
// k*G + G-1-c (k odd) of the ordered list; increasing in k.
__device__ __forceinline__ int64_t serp_index(int k, int c, int G) {
  return (int64_t)k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Shape checks of a sequence (false: the sequence is skipped and flagged).
__device__ __forceinline__ bool seq_ok(int n, int kv_len, int cap, int max_q) {
  return n >= 0 && kv_len >= n && kv_len <= cap && n <= max_q;
}

// Estimated time of a unit (the longest-first order's key), given its first new token i0:
// a key-tile step that both tiles take costs about 2.1 us on GB300, a step of one tile
// alone about 1.8 us, and a unit's start and end about 5 us (measured per unit with clock
// traces of this kernel on the chunked-prefill workload); in units of 0.1 us.
template <int P>
__device__ __forceinline__ uint32_t pair_cost(int n, int kv_len, int i0, bool causal) {
  const int c_len = kv_len - n;
  int nt[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int rows = min(P, n - (i0 + g * P));
    const int keys = rows <= 0 ? 0 : (causal ? c_len + i0 + g * P + rows : kv_len);
    nt[g] = (keys + kKeys - 1) / kKeys;
  }
  const uint32_t both = (uint32_t)min(nt[0], nt[1]);
  const uint32_t single = (uint32_t)abs(nt[0] - nt[1]);
  return 21u * both + 18u * single + 50u;
}

// Key tiles each tile of a unit multiplies (causal: up to its last position); tile B may
// have none.
template <int P>
__device__ __forceinline__ int unit_tiles(int n, int kv_len, int i0, bool causal) {
  const int c_len = kv_len - n;
  int packed = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int rows = min(P, n - (i0 + g * P));
    const int keys = rows <= 0 ? 0 : (causal ? c_len + i0 + g * P + rows : kv_len);
    packed |= ((keys + kKeys - 1) / kKeys) << (16 * g);
  }
  return packed;
}
__device__ __forceinline__ int nt_of(int nt, int g) { return (nt >> (16 * g)) & 0xFFFF; }
__device__ __forceinline__ int nt_all(int nt) { return max(nt & 0xFFFF, nt >> 16); }

// Completes this CTA's records (ring positions and tile counts; thread 0) and publishes the
// count. Ends with a block-wide barrier.
template <int P>
__device__ void finish_records(PrefillCtl& ctl, UnitRec* recs, int count, bool causal) {
  if (threadIdx.x == 0) {
    int v = 0;
    for (int k = 0; k < count; ++k) {
      recs[k].nt = unit_tiles<P>(recs[k].n, recs[k].kv_len, recs[k].i0, causal);
      recs[k].vbase = v;
      v += nt_all(recs[k].nt);
    }
    ctl.n_units = count;
  }
  __syncthreads();
}

// One unit per CTA: (KV head, sequence, pair) from the grid, latest pairs first.
template <int P>
__device__ void single_schedule(PrefillCtl& ctl, UnitRec* recs, const PrefillArgs& a) {
  int count = 0;
  if (threadIdx.x == 0) {
    const int j = blockIdx.x, s = blockIdx.y;
    const int qt = (int)gridDim.z - 1 - (int)blockIdx.z;
    const int q0 = __ldg(a.cu_seqlens_q + s);
    const int n = __ldg(a.cu_seqlens_q + s + 1) - q0;
    const int kv = __ldg(a.cu_seqlens_k + s + 1) - __ldg(a.cu_seqlens_k + s);
    if (!seq_ok(n, kv, a.max_blocks * a.block_size, a.max_seqlen_q)) {
      if (qt == 0 && j == 0) set_dev_err(a.dev_err, PA_DEV_ERR_SEQLENS);
    } else if (qt * 2 * P < n) {
      recs[0] = UnitRec{q0, n, kv, s, qt * 2 * P, j, 0, 0};
      count = 1;
    }
    ctl.n_units = count;
  }
  __syncthreads();
  finish_records<P>(ctl, recs, ctl.n_units, a.causal != 0);
}

// Builds the sorted schedule (all threads of the CTA take part; ends with a block-wide
// barrier). The scratch (cu_seqlens copies, per-sequence pair offsets, sort keys) lives in
// the K ring, which no copy has touched yet. The launcher takes this schedule only when
// the batch's bounds (num_seqs, max_seqlen_q, KV heads) guarantee that it fits.
template <int P>
__device__ void build_schedule(PrefillCtl& ctl, UnitRec* recs, unsigned char* scratch,
                               const PrefillArgs& a, int cu_q0, int cu_k0) {
  const int tid = threadIdx.x;
  const int S = a.num_seqs, Hk = a.num_kv_heads;
  if (S > kMaxSortSeqs) {  // excluded by the launcher
    if (tid == 0) {
      ctl.n_units = 0;
      if (blockIdx.x == 0) set_dev_err(a.dev_err, PA_DEV_ERR_SEQLENS);
    }
    __syncthreads();
    return;
  }
  int* cuq = reinterpret_cast<int*>(scratch);  // [S+1]
  int* cuk = cuq + (kMaxSortSeqs + 1);         // [S+1]
  int* poff = cuk + (kMaxSortSeqs + 1);        // [S+1]: pairs of the sequences before s
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(
      scratch + ((3 * (kMaxSortSeqs + 1) * 4 + 15) & ~15));
  const int cap = a.max_blocks * a.block_size;

  if (tid <= S) {  // loaded at kernel entry
    cuq[tid] = cu_q0;
    cuk[tid] = cu_k0;
  }
  for (int i = tid + kThreads; i <= S; i += kThreads) {
    cuq[i] = __ldg(a.cu_seqlens_q + i);
    cuk[i] = __ldg(a.cu_seqlens_k + i);
  }
  __syncthreads();
  // pairs per sequence and their exclusive prefix, one chunk of kThreads sequences a pass
  int carry = 0;
  const int lane = tid & 31, w = tid >> 5;
  for (int base = 0; base < S; base += kThreads) {
    const int s = base + tid;
    int cnt = 0;
    if (s < S) {
      const int n = cuq[s + 1] - cuq[s];
      const int kv = cuk[s + 1] - cuk[s];
      const bool ok = seq_ok(n, kv, cap, a.max_seqlen_q);
      if (!ok && blockIdx.x == 0) set_dev_err(a.dev_err, PA_DEV_ERR_SEQLENS);
      cnt = ok ? (n + 2 * P - 1) / (2 * P) : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) ctl.warp_sums[w] = incl;
    __syncthreads();
    int before = 0, chunk = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
      if (i < w) before += ctl.warp_sums[i];
      chunk += ctl.warp_sums[i];
    }
    if (s < S) poff[s] = carry + before + incl - cnt;
    carry += chunk;
    __syncthreads();
  }
  const int npairs = carry;
  const int64_t nunits = (int64_t)npairs * Hk;
  const int64_t per_cta = (nunits + gridDim.x - 1) / gridDim.x + 1;
  if (npairs > kMaxSortPairs || per_cta > kMaxUnitRecs) {  // excluded by the launcher
    if (tid == 0) {
      ctl.n_units = 0;
      if (blockIdx.x == 0) set_dev_err(a.dev_err, PA_DEV_ERR_SEQLENS);
    }
    __syncthreads();
    return;
  }
  if (tid == 0) poff[S] = npairs;
  int n2 = 1;
  while (n2 < npairs) n2 <<= 1;
  __syncthreads();
  // key: cost (key tiles) in the high word, then ~(s, pair) so that equal costs keep the
  // sequence order; padding keys are 0 and sort last
  for (int p = tid; p < npairs; p += kThreads) {
    // the sequence of pair p: the last s with poff[s] <= p (poff is non-decreasing)
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (poff[mid] <= p) lo = mid;
      else hi = mid - 1;
    }
    const int s = lo, qt = p - poff[s];
    const int n = cuq[s + 1] - cuq[s];
    const int kv = cuk[s + 1] - cuk[s];
    const uint32_t id = ((uint32_t)s << 12) | (uint32_t)qt;
    const uint32_t cost = pair_cost<P>(n, kv, qt * 2 * P, a.causal != 0);
    keys[p] = ((unsigned long long)cost << 32) | (unsigned long long)(0xFFFFFFFFu - id);
  }
  for (int i = npairs + tid; i < n2; i += kThreads) keys[i] = 0ull;
  __syncthreads();
  if (npairs <= kRankSortMax) {
    // small batches: each key's place is the number of larger keys (keys are distinct),
    // a few hundred shared-memory reads per thread instead of the network's barriers
    unsigned long long* sorted = keys + n2;
    for (int p = tid; p < npairs; p += kThreads) {
      const unsigned long long x = keys[p];
      int rank = 0;
      for (int q = 0; q < npairs; ++q) rank += keys[q] > x;
      sorted[rank] = x;
    }
    __syncthreads();
    keys = sorted;
  } else {
    // bitonic sort, descending
    for (int kk = 2; kk <= n2; kk <<= 1) {
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < n2; i += kThreads) {
          const int ixj = i ^ jj;
          if (ixj > i) {
            const unsigned long long x = keys[i], y = keys[ixj];
            if ((i & kk) == 0 ? (x < y) : (x > y)) {
              keys[i] = y;
              keys[ixj] = x;
            }
          }
        }
        __syncthreads();
      }
    }
  }
  // this CTA's units: the deal indices k with serp_index(k) < nunits form a prefix
  const int c = (int)blockIdx.x, G = (int)gridDim.x;
  for (int k = tid; k < kMaxUnitRecs; k += kThreads) {
    const int64_t idx = serp_index(k, c, G);
    if (idx >= nunits) continue;
    const unsigned long long key = keys[idx / Hk];
    const uint32_t id = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
    const int s = (int)(id >> 12), qt = (int)(id & 4095u);
    recs[k] = UnitRec{cuq[s], cuq[s + 1] - cuq[s], cuk[s + 1] - cuk[s], s, qt * 2 * P,
                      (int)(idx % Hk), 0, 0};
  }
  int count = 0;
  while (count < kMaxUnitRecs && serp_index(count, c, G) < nunits) ++count;
  __syncthreads();
  finish_records<P>(ctl, recs, count, a.causal != 0);
}

template <int G, int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q, const PrefillArgs a) {
  constexpr int P = kRows / G;  // query positions per tile
  constexpr int NH = D / 64;    // 64-dim swizzled column blocks per row
  constexpr bool kSepP = D == 64;  // P in its own tensor-memory columns (see col_p)
  using Tiles = PrefillTiles<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  PrefillCtl& ctl = *reinterpret_cast<PrefillCtl*>(smem_raw);
  UnitRec* recs = reinterpret_cast<UnitRec*>(smem_raw + kCtlBytes);
  Tiles& sm = *reinterpret_cast<Tiles*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + kCtlBytes + kRecBytes + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int H = a.num_heads;
  const bool causal = a.causal != 0;
  // the schedule's first inputs, requested before the set-up below so that their latency
  // overlaps it (entries past kThreads are loaded by the schedule itself)
  int cu_q0 = 0, cu_k0 = 0;
  if (a.persistent && tid <= a.num_seqs && a.num_seqs <= kMaxSortSeqs) {
    cu_q0 = __ldg(a.cu_seqlens_q + tid);
    cu_k0 = __ldg(a.cu_seqlens_k + tid);
  }

  if (tid == 0) {
    for (int g = 0; g < 2; ++g) {
      mbar_init(&ctl.q_full[g], 1);
      mbar_init(&ctl.q_empty[g], 1);
    }
    for (int b = 0; b < kKStages; ++b) {
      mbar_init(&ctl.k_full[b], 1);
      mbar_init(&ctl.k_empty[b], 1);
    }
    for (int b = 0; b < kVStages; ++b) {
      mbar_init(&ctl.v_full[b], 1);
      mbar_init(&ctl.v_empty[b], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&ctl.s_full[g], 1);
      mbar_init(&ctl.s_free[g], kRows);
      mbar_init(&ctl.p_full[g], kRows);
      mbar_init(&ctl.pv_done[g], 1);
      mbar_init(&ctl.o_done[g], 1);
    }
    ctl.abort = 0;
    ctl.n_units = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    umma::tmem_alloc(&ctl.tmem_base, kTmemCols);
    umma::tmem_relinquish();
  }
  __syncthreads();
  if (a.persistent) build_schedule<P>(ctl, recs, &sm.k[0][0], a, cu_q0, cu_k0);
  else single_schedule<P>(ctl, recs, a);
  // the schedule's scratch in the K ring was written through the generic proxy; TMA (the
  // async proxy) writes there next
  fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort;
  const int n_units = ctl.n_units;

  // Registers move from the control warpgroup (warps 8-11) to the softmax warpgroups; each
  // branch then runs to its own end (teardown included), so the compiler keeps the two
  // register budgets apart.
  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp walks the stream of key tiles (units in order, tiles in order): lane b
    // reads box b's block id, two tiles ahead of the K load that first needs it (the V load
    // of the same tile reuses it), so the table's latency stays off the copies' path; lane
    // 0 waits for free stages, and each box's lane issues its copy.
    if (lane == 0) {
      umma::prefetch_tmap(&tm_k);
      umma::prefetch_tmap(&tm_v);
    }
    const int bs = a.block_size;
    const int box_rows = bs < kKeys ? bs : kKeys;
    const int boxes = kKeys / box_rows;  // at most 16 (block_size 8)
    // this lane's block id of tile `it` of unit k: -1 past the keys (or past the stream),
    // -2 out of the pool
    auto read_id = [&](int k, int it) {
      if (k >= n_units || lane >= boxes) return -1;
      const UnitRec& u = recs[k];
      const int key0 = it * kKeys + lane * box_rows;
      if (key0 >= u.kv_len) return -1;
      const int id = __ldg(a.block_tables + (int64_t)u.s * a.max_blocks + key0 / bs);
      return (id >= 0 && (int64_t)id < a.num_blocks) ? id : -2;
    };
    auto advance = [&](int& k, int& it) {
      if (k < n_units && ++it >= nt_all(recs[k].nt)) {
        ++k;
        it = 0;
      }
    };
    int kl = 0, vl = 0;  // K and V loads issued so far (ring slot and phase)
    // lane-held ids of the current tile, the next one and the one after (being read)
    int k1 = 0, it1 = 0;
    advance(k1, it1);
    int k2 = k1, it2 = it1;
    advance(k2, it2);
    int id0 = read_id(0, 0), id1 = read_id(k1, it1), id2 = read_id(k2, it2);
    auto load = [&](bool is_v, int hj, int it, int id) {
      const int stages = is_v ? kVStages : kKStages;
      const int cnt = is_v ? vl++ : kl++;
      const int st = cnt % stages;
      uint64_t* empty = is_v ? &ctl.v_empty[st] : &ctl.k_empty[st];
      uint64_t* full = is_v ? &ctl.v_full[st] : &ctl.k_full[st];
      if (lane == 0 && cnt >= stages &&
          !mbar_wait(empty, (uint32_t)(((cnt / stages) - 1) & 1), abort_flag))
        note_timeout(ctl, a.dev_err);
      if (!is_v && __any_sync(0xffffffffu, id == -2) && lane == 0)
        set_dev_err(a.dev_err, PA_DEV_ERR_BLOCK_ID);
      const uint32_t valid = __ballot_sync(0xffffffffu, id >= 0);  // boxes with a block
      if (lane == 0)
        mbar_arrive_expect_tx(full, (uint32_t)__popc(valid) * NH * box_rows * 128u);
      __syncwarp();  // the stage is free and its bytes are expected: each box's lane copies
      if (id >= 0) {
        const int row0 = (bs > kKeys) ? ((it * kKeys) % bs) : 0;
        unsigned char* dst = (is_v ? sm.v[st] : sm.k[st]) + lane * box_rows * 128;
        const CUtensorMap* map = is_v ? &tm_v : &tm_k;
        for (int h2 = 0; h2 < NH; ++h2)
          umma::tma_load_4d(dst + h2 * kHalf, map, h2 * 64, hj, row0, id, full);
      }
      __syncwarp();
    };
    for (int k = 0; k < n_units; ++k) {
      const int n_all = nt_all(recs[k].nt);
      const int hj = recs[k].j;
      // K runs one tile ahead of V: S(i+1) is issued right after PV(i)
      load(false, hj, 0, id0);
      for (int it = 0; it < n_all; ++it) {
        load(true, hj, it, id0);
        if (it + 1 < n_all) load(false, hj, it + 1, id1);
        // shift the window one tile along the stream
        id0 = id1;
        id1 = id2;
        advance(k2, it2);
        id2 = read_id(k2, it2);
      }
    }
    // the last copies of every stage land before the CTA may exit (the full limit even
    // after a timeout elsewhere: a copy must not outlive the CTA's shared memory)
    if (lane == 0) {
      for (int c = kl > kKStages ? kl - kKStages : 0; c < kl; ++c)
        mbar_wait_copies(&ctl.k_full[c % kKStages], (uint32_t)((c / kKStages) & 1));
      for (int c = vl > kVStages ? vl - kVStages : 0; c < vl; ++c)
        mbar_wait_copies(&ctl.v_full[c % kVStages], (uint32_t)((c / kVStages) & 1));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (its descriptors are warp-uniform); one elected lane
    // issues the products and commits.
    {
      constexpr uint32_t idesc_s = umma::idesc_f32acc(kRows, kKeys, false, F16);
      constexpr uint32_t idesc_o = umma::idesc_f32acc(kRows, D, true, F16);
      int kc = 0, vc = 0;      // K and V loads consumed
      int qc[2] = {0, 0};      // Q tiles consumed, per tile slot
      int pc[2] = {0, 0};      // P tiles consumed, per tile slot
      int s_cnt[2] = {0, 0};   // head_dim 64: S products issued, per tile slot
      auto commit1 = [&](uint64_t* bar) {  // arrival on bar once the products so far are done
        if (elect_one()) umma::commit(bar);
        __syncwarp();
      };
      auto issue_s = [&](int g, int kstage) {  // S_g = Q_g K^T
        if constexpr (kSepP) {
          // S_g is overwritten once the softmax has read the previous one
          if (s_cnt[g] > 0 &&
              !mbar_wait(&ctl.s_free[g], (uint32_t)((s_cnt[g] - 1) & 1), abort_flag))
            note_timeout(ctl, a.dev_err);
          umma::fence_after_sync();
          ++s_cnt[g];
        }
        // descriptors of the K-slice kk: the tile's base descriptor plus the slice's offset
        // in 16-byte units (the address field cannot carry: shared addresses are < 256 KB)
        const uint64_t qd = umma::smem_desc(smem_u32(sm.q[g]), 16, 1024);
        const uint64_t kd = umma::smem_desc(smem_u32(sm.k[kstage]), 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off16 = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            umma::mma_bf16(tmem + col_s(g), qd + off16, kd + off16, idesc_s, kk > 0);
          }
          umma::commit(&ctl.s_full[g]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int g, int vstage, bool first) {  // O_g (+)= P_g V, P from TMEM
        const uint64_t vd = umma::smem_desc(smem_u32(sm.v[vstage]), kHalf, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            umma::mma_bf16_ts(tmem + col_o(g), tmem + (kSepP ? col_p(g) : col_s(g)) + kk * 8,
                              vd + ((kk * 16 * 128) >> 4), idesc_o, !first || (kk > 0));
          if constexpr (kSepP) umma::commit(&ctl.pv_done[g]);
        }
        __syncwarp();
      };
      auto wait_k = [&]() {
        if (!mbar_wait(&ctl.k_full[kc % kKStages], (uint32_t)((kc / kKStages) & 1), abort_flag))
          note_timeout(ctl, a.dev_err);
        umma::fence_after_sync();
      };
      // a unit's first S products: its Q tiles and K(0)
      auto start_unit = [&](int nt) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (nt_of(nt, g) == 0) continue;
          if (!mbar_wait(&ctl.q_full[g], (uint32_t)(qc[g] & 1), abort_flag))
            note_timeout(ctl, a.dev_err);
          ++qc[g];
        }
        wait_k();
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (nt_of(nt, g) == 0) continue;
          issue_s(g, kc % kKStages);
          if (nt_of(nt, g) == 1) commit1(&ctl.q_empty[g]);  // the unit's last S_g
        }
        commit1(&ctl.k_empty[kc % kKStages]);
        ++kc;
      };
      if (n_units > 0) start_unit(recs[0].nt);
      for (int k = 0; k < n_units; ++k) {
        const int nt = recs[k].nt;
        const int n_all = nt_all(nt);
        for (int it = 0; it < n_all; ++it) {
          if constexpr (kSepP) {
            // S(it+1) of each tile first (each waits only for its softmax to have read
            // S(it)), then PV(it) of each tile once its P is written
            if (it + 1 < n_all) {
              wait_k();
#pragma unroll
              for (int g = 0; g < 2; ++g) {
                const int ntg = nt_of(nt, g);
                if (it + 1 >= ntg) continue;
                issue_s(g, kc % kKStages);
                if (it + 2 == ntg) commit1(&ctl.q_empty[g]);  // the unit's last S_g
              }
              commit1(&ctl.k_empty[kc % kKStages]);
              ++kc;
            }
            bool vr = false;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const int ntg = nt_of(nt, g);
              if (it >= ntg) continue;
              if (!mbar_wait(&ctl.p_full[g], (uint32_t)(pc[g] & 1), abort_flag))
                note_timeout(ctl, a.dev_err);
              ++pc[g];
              if (!vr) {
                if (!mbar_wait(&ctl.v_full[vc % kVStages], (uint32_t)((vc / kVStages) & 1),
                               abort_flag))
                  note_timeout(ctl, a.dev_err);
                vr = true;
              }
              umma::fence_after_sync();
              issue_pv(g, vc % kVStages, it == 0);
              if (it == ntg - 1) commit1(&ctl.o_done[g]);
            }
            commit1(&ctl.v_empty[vc % kVStages]);
            ++vc;
            continue;
          }
          bool v_ready = false, k_ready = false;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int ntg = nt_of(nt, g);
            if (it >= ntg) continue;
            if (!mbar_wait(&ctl.p_full[g], (uint32_t)(pc[g] & 1), abort_flag))
              note_timeout(ctl, a.dev_err);
            ++pc[g];
            if (!v_ready) {
              if (!mbar_wait(&ctl.v_full[vc % kVStages], (uint32_t)((vc / kVStages) & 1),
                             abort_flag))
                note_timeout(ctl, a.dev_err);
              v_ready = true;
            }
            umma::fence_after_sync();
            issue_pv(g, vc % kVStages, it == 0);
            if (it == ntg - 1) commit1(&ctl.o_done[g]);
            if (it + 1 < ntg) {
              if (!k_ready) {
                wait_k();
                k_ready = true;
              }
              issue_s(g, kc % kKStages);
              if (it + 2 == ntg) commit1(&ctl.q_empty[g]);  // the unit's last S_g
            }
          }
          commit1(&ctl.v_empty[vc % kVStages]);
          ++vc;
          if (k_ready) {
            commit1(&ctl.k_empty[kc % kKStages]);
            ++kc;
          }
        }
        // the next unit's first S products follow this unit's last P.V products
        if (k + 1 < n_units) start_unit(recs[k + 1].nt);
      }
    }
  } else if (warp == kQWarp) {
    // ------------------------------------------------------------------ Q loader
    // Tile g of each unit is copied into its buffer as soon as the tile's last S product of
    // the previous unit has completed: one TMA box per 64 dims (128/G positions x the G heads
    // of the group) when every row of the box lies inside q, else (the batch's last rows)
    // plain 16-byte copies of the sequence's rows with zeros past it.
    const int64_t q_rows = min((int64_t)__ldg(a.cu_seqlens_q + a.num_seqs), q_map_rows(a));
    if (lane == 0) umma::prefetch_tmap(&tm_q);
    uint32_t qep = 0, started = 0;  // per tile: parity of its next q_empty phase; first done
    int qn[2] = {0, 0};             // Q copies issued per tile (one q_full phase each)
    auto box_ok = [&](const UnitRec& u, int g) {
      return (int64_t)u.q0 + u.i0 + g * P + P <= q_rows;
    };
    for (int k = 0; k < n_units; ++k) {
      const UnitRec& u = recs[k];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (nt_of(u.nt, g) == 0) continue;
        if ((started >> g) & 1u) {
          if (lane == 0 && !mbar_wait(&ctl.q_empty[g], (qep >> g) & 1u, abort_flag))
            note_timeout(ctl, a.dev_err);
          qep ^= 1u << g;
        }
        started |= 1u << g;
        ++qn[g];
        __syncwarp();
        unsigned char* qbuf = sm.q[g];
        const int i0 = u.i0 + g * P;  // the tile's first position in the sequence
        if (box_ok(u, g)) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&ctl.q_full[g], (uint32_t)(kRows * D * 2));
#pragma unroll
            for (int h2 = 0; h2 < NH; ++h2)
              umma::tma_load_3d(qbuf + h2 * kHalf, &tm_q, h2 * 64, u.j * G, u.q0 + i0,
                                &ctl.q_full[g]);
          }
        } else {
          for (int r = lane; r < kRows; r += 32) {
            const int qi = i0 + r / G;
            const bool ok = qi < u.n;
            const uint16_t* src = static_cast<const uint16_t*>(a.q) +
                                  (ok ? ((int64_t)(u.q0 + qi) * H + u.j * G + r % G) * D : 0);
#pragma unroll
            for (int ch = 0; ch < D / 8; ++ch)
              cp_async16_zfill(qbuf + (ch >> 3) * kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4),
                               src + (ok ? ch * 8 : 0), ok ? 16u : 0u);
          }
          cp_async_wait_all();
          fence_proxy_async_smem();  // written through the generic proxy, read by the MMA
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.q_full[g]);
        }
      }
    }
    // each tile's last copy lands before the CTA may exit (the full limit even after a
    // timeout elsewhere: a copy must not outlive the CTA's shared memory)
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (qn[g] > 0) mbar_wait_copies(&ctl.q_full[g], (uint32_t)((qn[g] - 1) & 1));
    }
  }
    // ---- teardown: every role is done with tensor memory
    umma::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
      umma::fence_after_sync();
      umma::tmem_dealloc(tmem, kTmemCols);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------------ softmax warpgroups
    const int g = warp >> 2;      // query tile of this warpgroup
    const int r = tid & 127;      // row == TMEM lane
    const int wq = warp & 3;      // warp within the warpgroup (TMEM lane quarter)
    const int pos = r / G, hh = r % G;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    int sc = 0, oc = 0;  // s_full and o_done phases consumed (sc: S tiles of this query tile)

    // the first unit after k (k = -1: the first unit) in which this tile has rows
    auto next_unit = [&](int k) {
      for (++k; k < n_units; ++k)
        if (nt_of(recs[k].nt, g) > 0) break;
      return k;
    };
    int k = next_unit(-1);
    while (k < n_units) {
      const int kn = next_unit(k);
      int lim_row, kv_len, vbase, my_nt;
      {
        const UnitRec& u = recs[k];
        const int qpos = (u.kv_len - u.n) + u.i0 + g * P + pos;  // absolute position of the row
        kv_len = u.kv_len;
        lim_row = causal ? min(kv_len, qpos + 1) : kv_len;  // keys [0, lim_row) count
        vbase = u.vbase;
        my_nt = nt_of(u.nt, g);
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int it = 0; it < my_nt; ++it) {
        if (!mbar_wait(&ctl.s_full[g], (uint32_t)(sc & 1), abort_flag)) note_timeout(ctl, a.dev_err);
        ++sc;
        umma::fence_after_sync();
        float sv[kKeys];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) umma::tmem_ld32(lane_addr + col_s(g) + 32 * c4, sv + 32 * c4);
        umma::tmem_ld_wait();
        if constexpr (kSepP) {  // S_g may be overwritten by the next product
          umma::fence_before_sync();
          mbar_arrive(&ctl.s_free[g]);
        }

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
        // p = 2^(s*scale - m): one packed fma per pair, then ex2; P packed as 16-bit pairs
        // over S, in the element type of V (the PV product takes both operands in one type)
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
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
        if constexpr (kSepP) {
          // the previous P.V of this tile has read P_g and landed in O_g (its pv_done phase;
          // the one before completed before this S product was issued)
          if (sc > 1 &&
              !mbar_wait(&ctl.pv_done[g], (uint32_t)((sc - 2) & 1), abort_flag))
            note_timeout(ctl, a.dev_err);
          umma::fence_after_sync();
          umma::tmem_st32(lane_addr + col_p(g), sv);
          umma::tmem_st32(lane_addr + col_p(g) + 32, sv + 32);
        } else {
          umma::tmem_st32(lane_addr + col_s(g), sv);
          umma::tmem_st32(lane_addr + col_s(g) + 32, sv + 32);
        }
        // O_g is stable here (head_dim 128: S_g(it) completed after PV_g(it-1); 64: waited
        // above); PV_g(it) waits for p_full
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
          const int vi = vbase + it;
          const int st = vi % kVStages;
          if (!mbar_wait(&ctl.v_full[st], (uint32_t)((vi / kVStages) & 1), abort_flag))
            note_timeout(ctl, a.dev_err);
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
        mbar_arrive(&ctl.p_full[g]);
      }

      // ---- epilogue: O / l -> 16-bit rows --------------------------------------------
      if (!mbar_wait(&ctl.o_done[g], (uint32_t)(oc & 1), abort_flag)) note_timeout(ctl, a.dev_err);
      ++oc;
      umma::fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const UnitRec& u = recs[k];
      const int qi = u.i0 + g * P + pos;
      const bool row_ok = qi < u.n;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                            ((int64_t)(u.q0 + qi) * H + u.j * G + hh) * D);
      float ob[D];  // the whole row at once: one tensor-memory round trip
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) umma::tmem_ld32(lane_addr + col_o(g) + 32 * c4, ob + 32 * c4);
      umma::tmem_ld_wait();
      if (row_ok && (reinterpret_cast<uintptr_t>(a.out) & 31) == 0) {
        // 32 bytes per store: one full sector each
#pragma unroll
        for (int q16 = 0; q16 < D / 16; ++q16) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = pack_elt2<F16>(ob[16 * q16 + 2 * e] * inv, ob[16 * q16 + 2 * e + 1] * inv);
          asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 2 * q16),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                       "r"(w[6]), "r"(w[7])
                       : "memory");
        }
      } else if (row_ok) {
#pragma unroll
        for (int q8 = 0; q8 < D / 8; ++q8) {
          uint4 pk;
          pk.x = pack_elt2<F16>(ob[8 * q8 + 0] * inv, ob[8 * q8 + 1] * inv);
          pk.y = pack_elt2<F16>(ob[8 * q8 + 2] * inv, ob[8 * q8 + 3] * inv);
          pk.z = pack_elt2<F16>(ob[8 * q8 + 4] * inv, ob[8 * q8 + 5] * inv);
          pk.w = pack_elt2<F16>(ob[8 * q8 + 6] * inv, ob[8 * q8 + 7] * inv);
          dst[q8] = pk;
        }
      }
      // the next unit's first P.V overwrites O_g only after this warpgroup's p_full of that
      // unit, which follows these reads
      k = kn;
    }
    // ---- teardown: every role is done with tensor memory
    umma::fence_before_sync();
    __syncthreads();
  }

}

template <int G, int D, bool F16>
int launch_prefill_t(const PrefillArgs& a, const DeviceInfo& info, cudaStream_t stream,
                     const CUtensorMap& mk, const CUtensorMap& mv) {
  constexpr int P = kRows / G;
  constexpr size_t smem = prefill_smem_bytes<D>();
  static_assert(prefill_smem_bytes<D>() <= 232448, "shared memory budget (opt-in maximum)");
  static std::atomic<bool> attr_done[64];  // zero-initialised: false
  if (info.device < 0 || info.device >= 64) return PA_ERR_CUDA;
  if ((size_t)info.max_smem_optin < smem) return PA_ERR_UNSUPPORTED;
  if (!attr_done[info.device].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(paged_prefill_kernel<G, D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[info.device].store(true, std::memory_order_release);
  }
  const int64_t qt_n = (a.max_seqlen_q + 2 * P - 1) / (2 * P);  // pairs per sequence at most
  const int64_t max_pairs = qt_n * a.num_seqs;
  const int64_t max_units = max_pairs * a.num_kv_heads;
  PrefillArgs args = a;
  CUtensorMap mq;
  if (!make_rows_map(&mq, a.q, q_map_rows(a), a.num_heads, D, F16, G, P)) return PA_ERR_CUDA;
  // persistent (one CTA per SM, fewer when the batch has fewer units) when the in-kernel
  // sort and every CTA's records are sure to hold the batch; else one unit per CTA
  const int grid1 = (int)(max_units < info.num_sms ? max_units : info.num_sms);
  args.persistent = a.num_seqs <= kMaxSortSeqs && max_pairs <= kMaxSortPairs && grid1 > 0 &&
                    (max_units + grid1 - 1) / grid1 + 1 <= kMaxUnitRecs;
  if (args.persistent) {
    paged_prefill_kernel<G, D, F16><<<grid1, kThreads, smem, stream>>>(mk, mv, mq, args);
  } else {
    if (qt_n > 65535) return PA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)a.num_kv_heads, (unsigned)a.num_seqs, (unsigned)qt_n);
    paged_prefill_kernel<G, D, F16><<<grid, kThreads, smem, stream>>>(mk, mv, mq, args);
  }
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
