// sample.cu — Gumbel-max sampling of one token per row of logits [B, V].
//
// "nano-vllm解读", section "Gumbel-Max采样": sampling from softmax(logits / T) equals taking
// argmax_i (ln p_i + G_i) with G_i = -ln(-ln u_i), u_i independent U(0,1); ln p_i and
// logits_i / T differ by a constant of the row, so the score is logits_i / T + G_i.
// "Model Runner V2 设计文档", section 6 ("Gumbel 采样内核"): no softmax is materialised and
// the random numbers come from a stateless in-kernel generator keyed by a seed input.
//
// Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC 2011). Element i of a row draws word i % 4 of the block at counter
// (i / 4, i / 2^34, offset lo, offset hi) under key (seed lo, seed hi); u = (2k + 1) / 2^24
// from the top 23 bits k (exact in binary32, never 0 or 1). T <= 0 samples greedily (the
// logit alone), a NaN logit never wins, ties go to the lowest index. The kernels rank by
// log2(e) * score - log2(log2(e)), which orders the elements exactly as the score does.
//
// Design (the logits are read once; the arithmetic is one Philox block per 4 elements and
// two special-function operations per element):
//  * Rows that start on 16 bytes: a persistent CTA per SM takes an even share of the
//    (row, tile of 40 KB for fp32, 24 KB for bf16) stream. A producer warp moves tiles with cp.async.bulk into a
//    4-stage shared-memory ring (mbarrier full/empty pairs, bounded waits); consumer
//    warps score them from shared memory, one 16-byte group per thread at a time.
//  * Other rows: one CTA per (row, 8192-element chunk) with plain loads.
//  * The running best is a 64-bit key: order-preserving bits of the score in the high
//    word, ~index in the low word, so an unsigned max picks the largest score and, among
//    equal scores, the lowest index. When a CTA leaves a row it reduces its key (warps,
//    then one thread), does one atomicMax into the row's key and adds its tile count to the
//    row's arrival counter; the CTA that completes the count writes the index and resets
//    key and counter to zero for the next call. One launch, deterministic.
#include <atomic>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleChunk = 8192;  // elements per CTA of the plain-load kernel
// consumer warps of the ring kernel (measured on B=256, V=151936: fp32 59.6-60.4 us at 20
// against 61.3-61.9 at 16 and 61.4 at 24; bf16 58.8-59.2 us at 12 against 61.4-63.4 at 16,
// where 20 warps leave too few registers and spill)
constexpr int kRingWarpsF32 = 20, kRingWarpsBf16 = 12;

__device__ __forceinline__ void philox4x32_10(uint32_t& c0, uint32_t& c1, uint32_t& c2,
                                              uint32_t& c3, uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint64_t p0, p1;  // full 32x32 -> 64-bit products
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(M0), "r"(c0));
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(M1), "r"(c2));
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c0 = n0;
    c1 = (uint32_t)p1;
    c2 = n2;
    c3 = (uint32_t)p0;
    k0 += W0;
    k1 += W1;
  }
}

// log2(u) (negative) for u = (2k + 1) / 2^24, k the top 23 bits of `bits`, with relative
// accuracy over the whole range. u = (1 + k/2^23) - (1 - 2^-24) is exact in binary32, and
// so is w = 1 - u (Sterbenz: u >= 1/2 where it is used). For u <= 0.9 the hardware log2
// (absolute error about 2^-22 on [1/2, 2], and |log2 u| >= 0.15, so at most about 2e-6
// relative); for u > 0.9, log2(1 - w) = -w P(w) with P the cubic below, fitted to
// -log2(1 - w) / w on [0, 0.1] by least squares on Chebyshev nodes reweighted toward the
// largest relative error, the sign carried by the coefficients: at most 3e-7 relative in
// binary32 over every uniform above 0.9 (an exhaustive CPU test evaluates these
// coefficients).
// log2-uniform-cubic: -0.425869345664978f -0.4766629934310913f -0.7214337587356567f -1.4426947832107544f
__device__ __forceinline__ float log2_uniform(uint32_t bits) {
  const float u = __uint_as_float(0x3F800000u + (bits >> 9)) - 0.99999994039535522f;
  const float w = 1.f - u;
  const float a = fast_log2(u);
  float p = -0.425869345664978f;
  p = fmaf(p, w, -0.4766629934310913f);
  p = fmaf(p, w, -0.7214337587356567f);
  p = fmaf(p, w, -1.4426947832107544f);
  // u <= 0.9 exactly when k <= 7549746 (u = (2k + 1) / 2^24), i.e. bits < 7549747 * 2^9
  return bits < 3865470464u ? a : w * p;
}

// Ranking score of one element in log2 units: l * (log2(e) / T) - log2(-log2 u).
__device__ __forceinline__ float rank_score(float l, float scale, uint32_t bits) {
  return fmaf(l, scale, -fast_log2(-log2_uniform(bits)));
}

__device__ __forceinline__ uint64_t score_key(float x, int64_t i) {
  uint32_t b = __float_as_uint(x);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)b << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

struct SampleArgs {
  const void* logits;
  int64_t row_stride;
  int vocab;
  int num_rows;
  int chunks;
  const float* temperatures;
  const uint64_t* seeds;
  const uint64_t* offsets;
  int64_t* out;
  unsigned long long* keys;  // [num_rows], zero between calls
  int* counters;             // [num_rows], zero between calls
  int* dev_err;
};

// T: float (4 elements per 16-byte group) or uint16_t bf16 bits (8 per group).
// Key of a CTA's best: reduce over the consumer threads (warp shuffles, then one thread
// over the warps' keys in `slots`; `sync` is the barrier over those threads), then one
// atomicMax into the row's key and `tiles` added to its arrival counter. The thread that
// completes the count (tiles of the row = chunks) writes the index and zeroes both.
template <typename Sync>
__device__ __forceinline__ void flush_row(const SampleArgs& a, int row, int tiles, float best_x,
                                          int64_t best_i, uint64_t* slots, int nwarps,
                                          int ctid, Sync sync) {
  uint64_t key = score_key(best_x, best_i);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) key = umax64(key, __shfl_xor_sync(0xffffffffu, key, m));
  if ((ctid & 31) == 0) slots[ctid >> 5] = key;
  sync();
  if (ctid == 0) {
    uint64_t k = slots[0];
    for (int w = 1; w < nwarps; ++w) k = umax64(k, slots[w]);
    atomicMax(a.keys + row, (unsigned long long)k);
    __threadfence();
    const int before = atomicAdd(a.counters + row, tiles);
    if (before + tiles == a.chunks) {
      __threadfence();
      const unsigned long long fin = atomicExch(a.keys + row, 0ull);
      a.out[row] = (int64_t)(0xFFFFFFFFu - (uint32_t)(fin & 0xFFFFFFFFull));
      a.counters[row] = 0;
    }
  }
}

__device__ __forceinline__ float widen(float v) { return v; }
__device__ __forceinline__ float widen(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// Score the n (<= 4) elements i0.. of a Philox block (i0 a multiple of 4) and keep the best.
__device__ __forceinline__ void score_block(const float* l, int64_t i0, int n, bool greedy,
                                           float scale, uint32_t k0, uint32_t k1, uint32_t o0,
                                           uint32_t o1, float& best_x, int64_t& best_i) {
  uint32_t r0 = 0, r1 = 0, r2 = 0, r3 = 0;
  if (!greedy) {
    const uint64_t g = (uint64_t)i0 >> 2;
    r0 = (uint32_t)g;
    r1 = (uint32_t)(g >> 32);
    r2 = o0;
    r3 = o1;
    philox4x32_10(r0, r1, r2, r3, k0, k1);
  }
  const uint32_t rw[4] = {r0, r1, r2, r3};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (e < n) {
      const float x = greedy ? l[e] : rank_score(l[e], scale, rw[e]);
      if (x > best_x) {  // NaN never passes; equal scores keep the earlier index
        best_x = x;
        best_i = i0 + e;
      }
    }
  }
}

// Rows that do not start on 16 bytes: one CTA per (row, chunk of kSampleChunk elements),
// plain loads of 4 consecutive elements per thread at a time.
template <typename T>
__global__ void __launch_bounds__(kSampleThreads) gumbel_sample_chunk_kernel(const SampleArgs a) {
  const int b = blockIdx.x / a.chunks;
  const int chunk = blockIdx.x - b * a.chunks;
  const int64_t c_begin = (int64_t)chunk * kSampleChunk;
  const int64_t c_end = min((int64_t)a.vocab, c_begin + kSampleChunk);
  const T* row = static_cast<const T*>(a.logits) + (int64_t)b * a.row_stride;
  const float temp = __ldg(a.temperatures + b);
  const bool greedy = !(temp > 0.f);
  const float scale = greedy ? 1.f : 1.4426950408889634f / temp;  // log2(e) / T
  const uint64_t seed = __ldg(reinterpret_cast<const unsigned long long*>(a.seeds) + b);
  const uint64_t off = __ldg(reinterpret_cast<const unsigned long long*>(a.offsets) + b);
  float best_x = -INFINITY;
  int64_t best_i = c_begin + (int64_t)threadIdx.x * 4;  // all -inf / NaN: the first element
  for (int64_t q = c_begin + (int64_t)threadIdx.x * 4; q < c_end; q += 4 * kSampleThreads) {
    float l[4];
    const int n = (int)min((int64_t)4, c_end - q);
#pragma unroll
    for (int e = 0; e < 4; ++e) l[e] = e < n ? widen(row[q + e]) : 0.f;
    score_block(l, q, n, greedy, scale, (uint32_t)seed, (uint32_t)(seed >> 32), (uint32_t)off,
                (uint32_t)(off >> 32), best_x, best_i);
  }
  __shared__ uint64_t slots[kSampleThreads / 32];
  flush_row(a, b, 1, best_x, best_i, slots, kSampleThreads / 32, threadIdx.x,
            [] { __syncthreads(); });
}

// ---------------------------------------------------------------- ring kernel
// Maximum of the NE (a power of two) scores of a thread's tile by a pairwise tree: node v
// (1 <= v < NE) holds the maximum of its children 2v and 2v + 1, nodes NE..2NE-1 are the
// leaves xs[0..NE-1]. fmaxf skips NaN, so a node is NaN only if all leaves under it are.
template <int NE>
__device__ __forceinline__ float tree_node(const float (&xs)[NE], const float (&t)[NE], int v) {
  return v >= NE ? xs[v - NE] : t[v];
}

template <int NE>
__device__ __forceinline__ float tree_max(const float (&xs)[NE], float (&t)[NE]) {
#pragma unroll
  for (int v = NE - 1; v >= 1; --v) t[v] = fmaxf(tree_node(xs, t, 2 * v), tree_node(xs, t, 2 * v + 1));
  return t[1];
}

// The first leaf holding the (non-NaN) maximum t[1]: from the root down, the left child
// when it equals the maximum (then a leaf under it does), else the right one. The left
// child of the node reached so far is picked out of its level by selects on the decisions
// already taken, so no array is indexed at run time.
template <int NE>
__device__ __forceinline__ int first_index_of_max(const float (&xs)[NE], const float (&t)[NE]) {
  constexpr int kLevels = __builtin_ctz(NE);
  static_assert((1 << kLevels) == NE, "power of two");
  const float m = t[1];
  bool right[kLevels];
#pragma unroll
  for (int lev = 0; lev < kLevels; ++lev) {
    // left children of the 2^lev nodes of this level, in order (constant trip counts, so
    // that every loop unrolls and c stays in registers)
    float c[NE / 2];
#pragma unroll
    for (int i = 0; i < NE / 2; ++i)
      if (i < (1 << lev)) c[i] = tree_node(xs, t, 2 * ((1 << lev) + i));
#pragma unroll
    for (int b = 0; b < kLevels; ++b)  // fold by the latest decision first
      if (b < lev) {
#pragma unroll
        for (int i = 0; i < NE / 4; ++i)
          if (i < (1 << (lev - b - 1))) c[i] = right[lev - 1 - b] ? c[2 * i + 1] : c[2 * i];
      }
    right[lev] = !(c[0] == m);
  }
  int j = 0;
#pragma unroll
  for (int lev = 0; lev < kLevels; ++lev) j = 2 * j + (right[lev] ? 1 : 0);
  return j;
}

constexpr int kRingStages = 4;
// a tile is four 16-byte groups per consumer thread (40 KB with 20 consumer warps, 24 KB
// with 12)
template <int CW>
constexpr int ring_tile_bytes() { return CW * 32 * 16 * 4; }

struct RingCtrl {
  uint64_t full[kRingStages];
  uint64_t empty[kRingStages];
  uint64_t slots[2][32];  // one key per consumer warp
  int abort;
};

// Rows that start on 16 bytes: persistent CTAs over the (row, tile) stream, tiles moved
// into shared memory by a producer warp, CW consumer warps.
template <typename T, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 1) gumbel_sample_ring_kernel(const SampleArgs a) {
  constexpr int EPG = 16 / sizeof(T);            // elements per 16-byte group
  constexpr int kTileBytes = ring_tile_bytes<CW>();
  static_assert(CW <= 32, "one key slot per consumer warp");
  constexpr int TE = kTileBytes / sizeof(T);     // elements per tile
  constexpr int CT = CW * 32;                    // consumer threads
  constexpr int GPT = kTileBytes / 16 / CT;      // groups per consumer thread per tile
  static_assert(GPT * CT * 16 == kTileBytes, "tile split");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  RingCtrl& ctl = *reinterpret_cast<RingCtrl*>(smem + kRingStages * kTileBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int64_t nt = (int64_t)a.num_rows * a.chunks;
  const int64_t x0 = (int64_t)blockIdx.x * nt / gridDim.x;
  const int64_t x1 = (int64_t)(blockIdx.x + 1) * nt / gridDim.x;
  if (x0 >= x1) return;  // no tiles: nothing initialised, nothing in flight
  if (tid == 0) {
    for (int st = 0; st < kRingStages; ++st) {
      mbar_init(&ctl.full[st], 1);
      mbar_init(&ctl.empty[st], CW);
    }
    ctl.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t n_tiles = x1 - x0;
  volatile int* abort_flag = &ctl.abort;

  if (warp == CW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      int b = (int)(x0 / a.chunks), ci = (int)(x0 - (int64_t)b * a.chunks);  // row, tile in row
      for (int64_t it = 0; it < n_tiles; ++it, ci = ci + 1 == a.chunks ? 0 : ci + 1,
                   b += ci == 0 ? 1 : 0) {
        const int64_t start = (int64_t)ci * TE;
        const int64_t n = min((int64_t)TE, (int64_t)a.vocab - start);
        const uint32_t bytes = (uint32_t)(n * (int64_t)sizeof(T)) & ~15u;
        const int st = (int)(it % kRingStages);
        if (it >= kRingStages &&
            !mbar_wait(&ctl.empty[st], (uint32_t)(((it / kRingStages) - 1) & 1), abort_flag)) {
          ctl.abort = 1;
          set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
        }
        mbar_arrive_expect_tx(&ctl.full[st], bytes);
        if (bytes)
          bulk_g2s_hint(smem + (size_t)st * kTileBytes,
                        static_cast<const T*>(a.logits) + (int64_t)b * a.row_stride + start, bytes,
                        &ctl.full[st], policy);
      }
      // the last stages must land before the CTA may exit
      const int64_t first = n_tiles > kRingStages ? n_tiles - kRingStages : 0;
      for (int64_t it = first; it < n_tiles; ++it)
        mbar_wait(&ctl.full[it % kRingStages], (uint32_t)((it / kRingStages) & 1), abort_flag);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  int cur = -1, row_tiles = 0, parity = 0;
  float best_x = -INFINITY, scale = 1.f;
  int64_t best_i = 0;
  bool greedy = true;
  uint32_t k0 = 0, k1 = 0, o0 = 0, o1 = 0;
  uint32_t rk0[10], rk1[10];  // Philox round keys of the current row
  // Counter words 1-3 of every block of a row are (0, offset lo, offset hi), so part of
  // rounds 0 and 1 is the same for the whole row. Round 0 leaves c0 = h0, c1 = h1,
  // c2 = hi(M0 ctr) ^ hb, c3 = lo(M0 ctr); round 1 then gives c0 = hi(M1 c2) ^ h2,
  // c1 = lo(M1 c2), c2 = c3 ^ h3 and c3 = h4, where h0..h4 and hb depend on the row only.
  uint32_t h0 = 0, h1 = 0, h2 = 0, h3 = 0, h4 = 0, hb = 0;
  auto sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(CT) : "memory"); };
  // row and tile within the row of tile x0 + it, advanced without a division per tile
  int b = (int)(x0 / a.chunks), ci = (int)(x0 - (int64_t)b * a.chunks);
  for (int64_t it = 0; it < n_tiles; ++it, ci = ci + 1 == a.chunks ? 0 : ci + 1,
               b += ci == 0 ? 1 : 0) {
    const int64_t start = (int64_t)ci * TE;
    const int64_t n = min((int64_t)TE, (int64_t)a.vocab - start);
    const int64_t n_bulk = ((n * (int64_t)sizeof(T)) & ~int64_t(15)) / (int64_t)sizeof(T);
    if (b != cur) {
      if (cur >= 0) {
        flush_row(a, cur, row_tiles, best_x, best_i, ctl.slots[parity], CW, tid, sync);
        parity ^= 1;
      }
      cur = b;
      row_tiles = 0;
      const float temp = __ldg(a.temperatures + b);
      greedy = !(temp > 0.f);
      scale = greedy ? 1.f : 1.4426950408889634f / temp;  // log2(e) / T
      const uint64_t seed = __ldg(reinterpret_cast<const unsigned long long*>(a.seeds) + b);
      const uint64_t off = __ldg(reinterpret_cast<const unsigned long long*>(a.offsets) + b);
      k0 = (uint32_t)seed;
      k1 = (uint32_t)(seed >> 32);
#pragma unroll
      for (int r = 0; r < 10; ++r) {
        rk0[r] = k0 + (uint32_t)r * 0x9E3779B9u;
        rk1[r] = k1 + (uint32_t)r * 0xBB67AE85u;
      }
      o0 = (uint32_t)off;
      o1 = (uint32_t)(off >> 32);
      {
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * o0;  // round 0: M1 * c2, c2 = offset lo
        h0 = (uint32_t)(p1 >> 32) ^ rk0[0];              // c1 = 0
        h1 = (uint32_t)p1;
        hb = o1 ^ rk1[0];                                // round 0: c3 ^ k1
        const uint64_t p0 = (uint64_t)0xD2511F53u * h0;  // round 1: M0 * c0
        h2 = h1 ^ rk0[1];
        h3 = (uint32_t)(p0 >> 32) ^ rk1[1];
        h4 = (uint32_t)p0;
      }
      best_x = -INFINITY;
      best_i = start + (int64_t)tid * EPG;  // all -inf / NaN: the row's first element
    }
    const int st = (int)(it % kRingStages);
    if (!mbar_wait(&ctl.full[st], (uint32_t)((it / kRingStages) & 1), abort_flag)) {
      if (lane == 0) {
        ctl.abort = 1;
        set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
      }
    }
    const unsigned char* tile = smem + (size_t)st * kTileBytes;
    uint4 raw[GPT];
#pragma unroll
    for (int k = 0; k < GPT; ++k) raw[k] = lds128(tile + ((size_t)k * CT + tid) * 16);
    // the stage is released before these loads are used: order them before the producer's
    // next bulk copy (async proxy) into it
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.empty[st]);  // the tile is in registers
    // scores of this thread's elements, in increasing index order; the tile's maximum is
    // located (first index holding it) only when it beats the running best
    constexpr int NE = GPT * EPG;
    float xs[NE];
    const int s0 = (int)start;
    const int nb = (int)n_bulk;
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      float l[EPG];
      if constexpr (sizeof(T) == 4) {
        l[0] = __uint_as_float(raw[k].x);
        l[1] = __uint_as_float(raw[k].y);
        l[2] = __uint_as_float(raw[k].z);
        l[3] = __uint_as_float(raw[k].w);
      } else {
        const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          l[2 * q] = __uint_as_float(w4[q] << 16);
          l[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
        }
      }
#pragma unroll
      for (int e = 0; e < EPG; ++e) xs[k * EPG + e] = l[e];  // the noise is added below
    }
    if (!greedy) {
      // the thread's Philox blocks advanced together, round by round (NB independent
      // chains interleaved), then the noise of each element
      constexpr int NB = NE / 4;
      uint32_t c0[NB], c1[NB], c2[NB], c3[NB];
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const int k = q / (EPG / 4), h = q % (EPG / 4);
        const uint32_t ctr = (uint32_t)((s0 + (k * CT + tid) * EPG) >> 2) + h;
        uint64_t p0, p1;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(0xD2511F53u), "r"(ctr));  // round 0
        const uint32_t x2 = (uint32_t)(p0 >> 32) ^ hb;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(0xCD9E8D57u), "r"(x2));   // round 1
        c0[q] = (uint32_t)(p1 >> 32) ^ h2;
        c1[q] = (uint32_t)p1;
        c2[q] = (uint32_t)p0 ^ h3;
        c3[q] = h4;
      }
#pragma unroll
      for (int r = 2; r < 10; ++r) {
#pragma unroll
        for (int q = 0; q < NB; ++q) {
          uint64_t p0, p1;
          asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(0xD2511F53u), "r"(c0[q]));
          asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(0xCD9E8D57u), "r"(c2[q]));
          const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1[q] ^ rk0[r];
          const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3[q] ^ rk1[r];
          c0[q] = n0;
          c1[q] = (uint32_t)p1;
          c2[q] = n2;
          c3[q] = (uint32_t)p0;
        }
      }
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        xs[4 * q + 0] = rank_score(xs[4 * q + 0], scale, c0[q]);
        xs[4 * q + 1] = rank_score(xs[4 * q + 1], scale, c1[q]);
        xs[4 * q + 2] = rank_score(xs[4 * q + 2], scale, c2[q]);
        xs[4 * q + 3] = rank_score(xs[4 * q + 3], scale, c3[q]);
      }
    }
    if (nb < TE) {  // only a row's last tile is short
#pragma unroll
      for (int k = 0; k < GPT; ++k)
        if ((k * CT + tid) * EPG >= nb) {
#pragma unroll
          for (int e = 0; e < EPG; ++e) xs[k * EPG + e] = -INFINITY;  // past the bulk part
        }
    }
    float t[NE];
    const float m = tree_max(xs, t);
    if (m > best_x) {
      const int jj = first_index_of_max(xs, t);
      best_x = m;
      best_i = s0 + ((jj / EPG) * CT + tid) * EPG + (jj % EPG);
    }
    // a ragged end of the row (fewer than 16 bytes): plain loads, one element per thread
    if (tid < n - n_bulk) {
      const int i = s0 + nb + tid;
      const T* rowp = static_cast<const T*>(a.logits) + (int64_t)b * a.row_stride;
      const float lv = widen(rowp[i]);
      float xv = lv;
      if (!greedy) {
        uint32_t r0 = (uint32_t)(i >> 2), r1 = 0, r2 = o0, r3 = o1;
        philox4x32_10(r0, r1, r2, r3, k0, k1);
        const int e = i & 3;
        xv = rank_score(lv, scale, e == 0 ? r0 : e == 1 ? r1 : e == 2 ? r2 : r3);
      }
      if (xv > best_x || (xv == best_x && i < best_i)) {
        best_x = xv;
        best_i = i;
      }
    }
    ++row_tiles;
  }
  flush_row(a, cur, row_tiles, best_x, best_i, ctl.slots[parity], CW, tid, sync);
}

}  // namespace

size_t sample_workspace_bytes(int num_rows) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  return up((size_t)num_rows * 8) + up((size_t)num_rows * 4);
}

namespace {
template <typename T, int CW>
int launch_ring(const SampleArgs& a, cudaStream_t stream, int num_sms) {
  const size_t smem = (size_t)kRingStages * ring_tile_bytes<CW>() + sizeof(RingCtrl) + 128;
  static std::atomic<bool> attr_done[64];  // zero-initialised: false
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(gumbel_sample_ring_kernel<T, CW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int64_t nt = (int64_t)a.num_rows * a.chunks;
  const int grid = (int)(nt < num_sms ? nt : num_sms);
  gumbel_sample_ring_kernel<T, CW><<<grid, (CW + 1) * 32, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
}  // namespace

int launch_gumbel_sample(int64_t* out, const void* logits, int64_t row_stride, int is_bf16,
                         int num_rows, int vocab, const float* temperatures,
                         const uint64_t* seeds, const uint64_t* offsets, void* workspace,
                         int* dev_err, cudaStream_t stream, int num_sms) {
  SampleArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.vocab = vocab;
  a.num_rows = num_rows;
  a.temperatures = temperatures;
  a.seeds = seeds;
  a.offsets = offsets;
  a.out = out;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.keys = reinterpret_cast<unsigned long long*>(ws);
  a.counters = reinterpret_cast<int*>(ws + (((size_t)num_rows * 8 + 255) & ~size_t(255)));
  a.dev_err = dev_err;
  const int esz = is_bf16 ? 2 : 4;
  const bool ring = (reinterpret_cast<uintptr_t>(logits) & 15) == 0 && ((row_stride * esz) & 15) == 0;
  if (ring) {
    const int tile = is_bf16 ? ring_tile_bytes<kRingWarpsBf16>() : ring_tile_bytes<kRingWarpsF32>();
    a.chunks = (int)(((int64_t)vocab * esz + tile - 1) / tile);
    return is_bf16 ? launch_ring<uint16_t, kRingWarpsBf16>(a, stream, num_sms)
                   : launch_ring<float, kRingWarpsF32>(a, stream, num_sms);
  }
  a.chunks = (vocab + kSampleChunk - 1) / kSampleChunk;
  const int64_t grid = (int64_t)a.chunks * num_rows;
  if (grid > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (is_bf16) gumbel_sample_chunk_kernel<uint16_t><<<(unsigned)grid, kSampleThreads, 0, stream>>>(a);
  else gumbel_sample_chunk_kernel<float><<<(unsigned)grid, kSampleThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
