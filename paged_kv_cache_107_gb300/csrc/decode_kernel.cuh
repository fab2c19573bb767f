// decode_kernel.cuh — paged GQA decode attention on CUDA cores (bandwidth-bound GEMV).
// The kernel template; decode.cu instantiates the plain call and decode_step.cu the one
// fused with the store of the new tokens.
//
// What it computes ("nano-vllm解读", sections "PageAttention原理" and "Nano-vllm中的使用";
// "3.6 ModelRunner、CUDA Graph 与性能基准", section 2): for every sequence b and query head
// h, o = softmax(scale * q_h K^T) V over the first context_lens[b] cached tokens of KV
// head h / (H/H_kv), where token t lives at row block_tables[b][t / bs] * bs + t % bs.
// The softmax is evaluated online, tile by tile, as the FlashAttention description on the
// nano-vllm overview page ("FlashAttention 核心思想") lays out: load a K/V tile into on-chip
// memory, update the running max and sum, accumulate, discard the tile.
//
// GB300 design
//  * Work split ("stream-K" over key tiles). Every sequence is cut into tiles of T tokens;
//    all tiles of all sequences form one stream of NT tiles, and CTA c of the grid takes
//    tiles [c*NT/G, (c+1)*NT/G). Every CTA therefore reads the same number of bytes
//    whatever the length mix. A sequence whose tiles all fall in one CTA is written
//    directly; a sequence cut between CTAs leaves one partial (o, log-sum-exp) per CTA,
//    and the last CTA to finish it (arrival counter) combines them in CTA order, so the
//    result is deterministic.
//  * FUSED (pa_decode_step): the new token of sequence b (k_new/v_new row b) is stored at
//    slot_mapping[b] by the CTA that owns the sequence's last tile. Its producer copies
//    that row into the tile straight from k_new/v_new (the cache rows before it come from
//    the cache), and the half-warp that loads the row from shared memory also writes it to
//    the cache slot. Store and attention are one launch, and the new row is read once.
//  * One CTA handles a slab of HS KV heads (all of them when H_kv <= 8), so one token's
//    rows for the slab are HS*256 contiguous bytes: the producer warp moves a tile's rows
//    into a STAGES-deep shared-memory ring guarded by mbarriers, with one cp.async.bulk
//    (TMA engine) per K and V when they form one run of cache rows (the slab is every KV
//    head and the tile lies in one block), else one per token row. Tiles never need block
//    alignment: each token's row can be addressed through the block table on its own.
//  * Launched as a programmatic dependent of the previous kernel on the stream: the
//    prologue reads context_lens (and, in the fused step, slot_mapping for its checks),
//    the producer reads the block-table rows of its first tiles to prefetch their K/V
//    runs into L2, and everything that reads q, the new rows or the caches, or writes the
//    output or the workspace, waits for the previous grid first.
//  * The last CTA of a split sequence combines the partials in CTA order
//    (combine_partials): the LSEs of every head and segment in one round trip per batch,
//    the partial outputs of up to four heads per segment together.
//  * 8 consumer warps (+1 producer warp: 9 warps keep 168 registers per thread):
//    warp (j, w) owns KV head j of the slab and 16 tokens of every tile; a half-warp
//    holds one token row (16 lanes x 16 bytes), so each K row is read from shared memory
//    once and reused for all G = H/H_kv query heads of the group. Partial
//    dot products are reduced with a butterfly that halves the value count at every
//    shuffle stage (about one shuffle per score). fp32 online softmax with exp2 on
//    pre-scaled q; fp32 accumulation; one bf16 rounding at the end.
#pragma once

#include <atomic>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kTokPerWarp = 16;
constexpr int kPairs = kTokPerWarp / 2;  // token pairs (one per half-warp) per warp and tile
constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagWhole = 4;

template <int HS, int G, int D>
struct DecCfg {
  static constexpr int DPL = D / 16;                // dims per lane (a half-warp per row)
  static constexpr int T = 128 / HS;                // tokens per stage
  static constexpr int WPH = kConsumerWarps / HS;   // consumer warps per KV head
  static constexpr int ROW = HS * D * 2;            // bytes of one token row of the slab
  static constexpr int KV_BYTES = T * ROW;          // K (or V) bytes per stage
  static constexpr int Q_BYTES = HS * G * D * 2;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES + Q_BYTES;
  static constexpr int STAGES = (3 * STAGE_BYTES + 8192 <= 227 * 1024) ? 3 : 2;
  static constexpr int NV = kPairs * G;             // partial scores per lane per tile
  static constexpr int CF = NV >= 16 ? NV / 16 : 1;  // scores per lane after the reduction
  static constexpr int MERGE_FLOATS = G * (D + 2);
  static constexpr int PBUF_FLOATS = 2 * kPairs * G;  // per warp: [half][pair][head]
  static constexpr int CTRL_BYTES = 4096 + kConsumerWarps * PBUF_FLOATS * 4;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + CTRL_BYTES + 128;
  static_assert(T == WPH * kTokPerWarp, "tile / warp split");
  static_assert((kConsumerWarps - HS) * MERGE_FLOATS * 4 <= 2 * KV_BYTES, "merge scratch");
};

struct __align__(16) StageMeta {
  int64_t pb;     // first tile of the sequence in the global tile stream
  int64_t new_slot;  // FUSED: cache row that receives the tile's new token
  int b;          // sequence
  int tok0;       // first token of the tile
  int count;      // valid tokens in the tile
  int nb;         // tiles of the sequence
  int flags;
  int new_row;    // FUSED: row of the tile taken from k_new/v_new and stored; -1 = none
};

struct Ctrl {
  uint64_t full[3];
  uint64_t empty[3];
  uint64_t seg_bar;
  uint64_t merge_bar[8];
  StageMeta meta[3];
  int64_t nt;      // tiles in the stream
  int64_t x0, x1;  // this CTA's tile range
  int64_t pb0;     // first tile of the sequence holding x0
  int b0;
  int g_eff;       // CTAs that own tiles
  int found;
  int abort;
  int64_t red[32];
};

__device__ __forceinline__ int load_ctx(const int32_t* ctx, int b, int cap) {
  const int n = __ldg(ctx + b);
  return (n < 0 || n > cap) ? 0 : n;
}

// CTA of the balanced split that owns tile x: the largest c with floor(c*NT/G) <= x.
__device__ __forceinline__ int64_t cta_of(int64_t x, int64_t nt, int g) {
  return ((x + 1) * g - 1) / nt;
}
__device__ __forceinline__ int64_t tile_begin(int64_t c, int64_t nt, int g) {
  return (c * nt) / g;
}

// One butterfly stage over the 16 lanes of a half-warp: N values -> N/2 values, or a plain
// all-reduce once a single value is left.
template <int N>
__device__ __forceinline__ void bfly(float* v, int sub, int mask) {
  if constexpr (N > 1) {
    const bool up = (sub & mask) != 0;
#pragma unroll
    for (int k = 0; k < N / 2; ++k) {
      const float send = up ? v[k] : v[k + N / 2];
      const float keep = up ? v[k + N / 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
  }
}

template <int N>
struct Half {
  static constexpr int v = N > 1 ? N / 2 : 1;
};

// After the butterfly, lane value r holds flattened index kb + r, kb from the lane bits.
template <int NV>
__device__ __forceinline__ int bfly_base(int sub) {
  int kb = 0, c = NV;
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) {
    if (c > 1) {
      c >>= 1;
      if (sub & m) kb += c;
    }
  }
  return kb;
}

// Value for head hh taken from the lane that owns it. After the butterfly the flattened
// index is kk = pair*G + hh, the pair bits sit in sub-lane bits 3..1 and the head in
// sub-lane bit 0 and the value index r: hh = (sub & 1) * CF + r.
template <int G, int CF>
__device__ __forceinline__ float head_bcast(const float* vals, int hh, int lane) {
  if constexpr (G == 1) {
    return vals[0];
  } else {
    // hh is a compile-time constant at every (unrolled) call site
    return __shfl_sync(0xffffffffu, vals[hh % CF], (lane & ~1) | (hh / CF));
  }
}

// Packed fp32x2 arithmetic (two independent fp32 lanes per instruction).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<const float2*>(&d);
}
// Two 16-bit elements (element 0 in the low half) widened to an fp32 pair: bf16 is the
// top half of an fp32 (a shift or a mask), IEEE fp16 converts in hardware.
template <bool F16>
__device__ __forceinline__ float2 elt2_f2(uint32_t w) {
  if constexpr (F16) {
    float lo, hi;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
    return make_float2(lo, hi);
  } else {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
}
// Round-to-nearest-even packing of an fp32 pair into two 16-bit elements.
template <bool F16>
__device__ __forceinline__ uint32_t f2_elt2(float lo, float hi) {
  if constexpr (F16) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  } else {
    return f32x2_to_bf16x2(lo, hi);
  }
}

// DPL consecutive 16-bit elements of one lane (DPL/2 words): 16 or 8 bytes.
template <int DPL>
struct LaneVec {
  uint32_t w[DPL / 2];
};
template <int DPL>
__device__ __forceinline__ LaneVec<DPL> ld_lane(const void* p) {
  LaneVec<DPL> v;
  if constexpr (DPL == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    v.w[0] = u.x, v.w[1] = u.y, v.w[2] = u.z, v.w[3] = u.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v.w[0] = u.x, v.w[1] = u.y;
  }
  return v;
}
template <int DPL>
__device__ __forceinline__ void st_lane(void* p, const LaneVec<DPL>& v) {
  if constexpr (DPL == 8) *reinterpret_cast<uint4*>(p) = make_uint4(v.w[0], v.w[1], v.w[2], v.w[3]);
  else *reinterpret_cast<uint2*>(p) = make_uint2(v.w[0], v.w[1]);
}
template <int DPL>
__device__ __forceinline__ LaneVec<DPL> zero_lane() {
  LaneVec<DPL> v;
#pragma unroll
  for (int i = 0; i < DPL / 2; ++i) v.w[i] = 0u;
  return v;
}

// Last arrival for (sequence b, KV head kvh): combine the partials of the nseg CTAs
// c_lo.. that processed parts of sequence b, in CTA order, for the G query heads of the
// group, and write the G output rows. One warp. Lane h + G*j holds the LSE of head h in
// segment j of a batch of 32/G segments, so the LSEs of every head arrive in one round
// trip per batch and the per-head maxima come from shuffles; then the partial outputs of
// up to four heads and of SU consecutive segments are loaded together before any of them
// is accumulated (one round trip per SU segments and group of four heads; the sums still
// run in CTA order, so the result does not depend on SU). GMAX bounds G.
template <int D, bool F16, int GMAX>
__device__ __forceinline__ void combine_partials(const DecodeArgs& a, int b, int kvh, int G,
                                                 int64_t c_lo, int nseg, int64_t NT, int g_eff,
                                                 int64_t pb, int lane) {
  constexpr int CPL = D / 32;                 // combined dims per lane
  constexpr int HG = GMAX < 4 ? GMAX : 4;     // heads combined together
  // segments whose loads are in flight together, within the registers the kernel has
  // left: eight for groups of 1-2 heads (the CUDA-core kernel), two for four heads of 64
  // dims, one for four heads of 128 dims (the tensor-core kernel)
  constexpr int SU = HG <= 2 ? 8 : (HG * CPL <= 8 ? 2 : 1);
  const int H = a.num_heads;
  const int SB = 32 / G;                      // segments per batch
  const int my_h = lane % G, my_j = lane / G;
#pragma unroll 1
  for (int h0 = 0; h0 < G; h0 += HG) {
    float acc[HG][CPL], m_h[HG], den[HG];
#pragma unroll
    for (int q = 0; q < HG; ++q) {
      m_h[q] = -INFINITY;
      den[q] = 0.f;
#pragma unroll
      for (int e = 0; e < CPL; ++e) acc[q][e] = 0.f;
    }
    for (int s0 = 0; s0 < nseg; s0 += SB) {
      float ls = -INFINITY;
      int sl = 0;
      if (my_j < SB && s0 + my_j < nseg) {
        const int64_t c2 = c_lo + s0 + my_j;
        sl = (tile_begin(c2, NT, g_eff) < pb) ? 1 : 0;
        ls = __ldcg(a.part_lse + (c2 * 2 + sl) * H + kvh * G + my_h);
      }
      const int nb = min(SB, nseg - s0);
      // move each head's running state to the batch maximum
#pragma unroll
      for (int q = 0; q < HG; ++q) {
        if (h0 + q < G) {
          float bm = -INFINITY;
          for (int j = 0; j < nb; ++j)
            bm = fmaxf(bm, __shfl_sync(0xffffffffu, ls, h0 + q + G * j));
          const float nm = fmaxf(m_h[q], bm);
          const float al = (m_h[q] == -INFINITY) ? 0.f : fast_exp2(m_h[q] - nm);
          den[q] *= al;
#pragma unroll
          for (int e = 0; e < CPL; ++e) acc[q][e] *= al;
          m_h[q] = nm;
        }
      }
      for (int j0 = 0; j0 < nb; j0 += SU) {
        float w[SU][HG];
        float po[SU][HG][CPL];
#pragma unroll
        for (int u = 0; u < SU; ++u) {
          const int j = j0 + u;
          const bool seg = j < nb;
          const int64_t cj = c_lo + s0 + j;
          const int slj = __shfl_sync(0xffffffffu, sl, seg ? G * j : 0);
#pragma unroll
          for (int q = 0; q < HG; ++q) {
            w[u][q] = 0.f;
#pragma unroll
            for (int e = 0; e < CPL; ++e) po[u][q][e] = 0.f;
            const float l = __shfl_sync(0xffffffffu, ls, seg ? h0 + q + G * j : 0);
            if (seg && h0 + q < G) {
              w[u][q] = (m_h[q] == -INFINITY || l == -INFINITY) ? 0.f : fast_exp2(l - m_h[q]);
              if (w[u][q] != 0.f) {
                const float* src =
                    a.part_o + ((cj * 2 + slj) * H + kvh * G + h0 + q) * D + lane * CPL;
                if constexpr (CPL == 4) {
                  const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
                  po[u][q][0] = v.x;
                  po[u][q][1] = v.y;
                  po[u][q][2] = v.z;
                  po[u][q][3] = v.w;
                } else {
                  const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
                  po[u][q][0] = v.x;
                  po[u][q][1] = v.y;
                }
              }
            }
          }
        }
        // accumulate in segment (CTA) order
#pragma unroll
        for (int u = 0; u < SU; ++u) {
#pragma unroll
          for (int q = 0; q < HG; ++q) {
            den[q] += w[u][q];
#pragma unroll
            for (int e = 0; e < CPL; ++e) acc[q][e] = fmaf(w[u][q], po[u][q][e], acc[q][e]);
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < HG; ++q) {
      if (h0 + q < G) {
        const float inv = den[q] > 0.f ? 1.f / den[q] : 0.f;
        uint16_t* dst =
            static_cast<uint16_t*>(a.out) + ((int64_t)b * H + kvh * G + h0 + q) * D + lane * CPL;
        if constexpr (CPL == 4) {
          *reinterpret_cast<uint2*>(dst) =
              make_uint2(f2_elt2<F16>(acc[q][0] * inv, acc[q][1] * inv),
                         f2_elt2<F16>(acc[q][2] * inv, acc[q][3] * inv));
        } else {
          *reinterpret_cast<uint32_t*>(dst) = f2_elt2<F16>(acc[q][0] * inv, acc[q][1] * inv);
        }
      }
    }
  }
}

template <int HS, int G, bool FUSED, int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_kernel(const DecodeArgs a) {
  using C = DecCfg<HS, G, D>;
  constexpr int DPL = C::DPL;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem + (size_t)C::STAGES * C::STAGE_BYTES);
  float* pbuf_all = reinterpret_cast<float*>(smem + (size_t)C::STAGES * C::STAGE_BYTES + 4096);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;
  const int slab = blockIdx.y;
  const int H = a.num_heads;
  const int Hk = a.num_kv_heads;
  const int cap = a.max_blocks * a.block_size;
  const int B = a.num_seqs;
  constexpr int T = C::T;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kConsumerWarps);
    }
    mbar_init(&ctl.seg_bar, kConsumerWarps);
    if (C::WPH > 1)
      for (int j = 0; j < HS; ++j) mbar_init(&ctl.merge_bar[j], C::WPH - 1);
    ctl.found = 0;
    ctl.abort = 0;
    ctl.b0 = 0;
    ctl.pb0 = 0;
    fence_mbar_init();
  }

  // the next kernel on the stream may be scheduled onto SMs as this grid's CTAs leave (it
  // waits for this grid before touching its results)
  pdl_launch_dependents();

  // ---- prologue: total tiles, then the sequence that holds this CTA's first tile -----
  int64_t local = 0;
  for (int b = tid; b < B; b += kThreads) {
    const int raw = __ldg(a.context_lens + b);
    if (raw < 0 || raw > cap) {
      if ((b % gridDim.x) == c && slab == 0) set_dev_err(a.dev_err, PA_DEV_ERR_CONTEXT);
    }
    // FUSED: a token of an empty sequence has no position to be stored at
    if (FUSED && (raw <= 0 || raw > cap) && __ldg(a.slot_mapping + b) != -1) {
      if ((b % gridDim.x) == c && slab == 0) set_dev_err(a.dev_err, PA_DEV_ERR_SLOT);
    }
    local += (load_ctx(a.context_lens, b, cap) + T - 1) / T;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) local += __shfl_xor_sync(0xffffffffu, local, m);
  if (lane == 0) ctl.red[warp] = local;
  __syncthreads();
  if (tid == 0) {
    int64_t nt = 0;
    for (int w = 0; w < kThreads / 32; ++w) nt += ctl.red[w];
    ctl.nt = nt;
    // CTAs that own tiles: every CTA of the grid, unless the stream is too short to give
    // each at least min_tiles
    const int64_t mt = a.min_tiles > 1 ? a.min_tiles : 1;
    const int64_t want = (nt + mt - 1) / mt;
    const int g_eff = (int)(want < (int64_t)gridDim.x ? want : (int64_t)gridDim.x);
    ctl.g_eff = g_eff;
    if (c < g_eff) {
      ctl.x0 = tile_begin(c, nt, g_eff);
      ctl.x1 = tile_begin(c + 1, nt, g_eff);
    } else {
      ctl.x0 = ctl.x1 = 0;
    }
  }
  __syncthreads();
  const int64_t NT = ctl.nt;
  const int g_eff = ctl.g_eff;
  const int64_t x0 = ctl.x0, x1 = ctl.x1;

  if (x0 < x1) {
    // chunked scan over the sequences until the one holding tile x0 is found
    int64_t running = 0;
    for (int base = 0; base < B; base += kConsumerWarps * 32) {
      int n = 0;
      const int b = base + tid;
      if (tid < kConsumerWarps * 32 && b < B) n = (load_ctx(a.context_lens, b, cap) + T - 1) / T;
      int incl = n;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, m);
        if (lane >= m) incl += y;
      }
      if (lane == 31) ctl.red[warp] = incl;
      __syncthreads();
      int64_t warp_off = 0;
      int64_t chunk_total = 0;
      for (int w = 0; w < kConsumerWarps; ++w) {
        if (w < warp) warp_off += ctl.red[w];
        chunk_total += ctl.red[w];
      }
      if (tid < kConsumerWarps * 32 && b < B && n > 0) {
        const int64_t p = running + warp_off + incl - n;
        if (p <= x0 && x0 < p + n) {
          ctl.b0 = b;
          ctl.pb0 = p;
          ctl.found = 1;
        }
      }
      running += chunk_total;
      __syncthreads();
      if (ctl.found) break;
    }
  }
  __syncthreads();
  // Before waiting, the producer warp warms L2 with the K/V runs of this CTA's first
  // tiles (lanes 2t, 2t+1: K, V of tile t). Block tables are inputs, and an L2 prefetch
  // leaves no stale copy: L2 is where the earlier grids' writes land. Only whole-row
  // runs inside one block are prefetched.
  if (warp == kProducerWarp && x0 < x1 && ctl.found && lane < 2 * C::STAGES) {
    const int64_t row_elems = (int64_t)Hk * D;
    if (slab == 0 && row_elems == (int64_t)HS * D && x0 + (lane >> 1) < x1) {
      const int64_t x = x0 + (lane >> 1);
      int b = ctl.b0;
      int64_t pb = ctl.pb0;
      int ctx_b = load_ctx(a.context_lens, b, cap);
      int nb = (ctx_b + T - 1) / T;
      while (x >= pb + nb && b + 1 < B) {
        pb += nb;
        ++b;
        ctx_b = load_ctx(a.context_lens, b, cap);
        nb = (ctx_b + T - 1) / T;
      }
      const int tok0 = (int)(x - pb) * T;
      const int count = min(T, ctx_b - tok0);
      if (count > 0 && tok0 / a.block_size == (tok0 + count - 1) / a.block_size) {
        const int blk = __ldg(a.block_tables + (int64_t)b * a.max_blocks + tok0 / a.block_size);
        if (blk >= 0 && (int64_t)blk < a.num_blocks) {
          const uint16_t* base = static_cast<const uint16_t*>((lane & 1) ? a.v_cache : a.k_cache);
          const uint16_t* src = base + ((int64_t)blk * a.block_size + tok0 % a.block_size) * row_elems;
          prefetch_l2_bulk(src, (uint32_t)(count * row_elems * 2));
        }
      }
    }
  }
  // everything above read only context_lens (an input no earlier kernel of the step
  // writes); from here on the kernel reads q, the new rows and the caches and writes out
  // and the workspace, so the grids launched before it must be complete
  pdl_wait();

  // zero rows of empty (or invalid) sequences assigned to this CTA: one warp per row
  {
    const int heads_per_slab = HS * G;
    for (int b = c + warp * (int)gridDim.x; b < B; b += (kThreads / 32) * (int)gridDim.x) {
      if (load_ctx(a.context_lens, b, cap) != 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                            ((int64_t)b * H + slab * heads_per_slab) * D);
      const int nvec = heads_per_slab * D / 8;
      for (int i = lane; i < nvec; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
    }
  }

  // no tiles (all barriers idle; nothing in flight); a start that cannot be located means
  // context_lens changed under the kernel: flag it and do nothing
  if (x0 >= x1) return;
  if (!ctl.found) {
    if (tid == 0) set_dev_err(a.dev_err, PA_DEV_ERR_CONTEXT);
    return;
  }

  const int64_t n_tiles = x1 - x0;
  volatile int* abort_flag = &ctl.abort;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    const uint64_t policy = policy_evict_first();
    const uint16_t* kc = static_cast<const uint16_t*>(a.k_cache);
    const uint16_t* vc = static_cast<const uint16_t*>(a.v_cache);
    const int64_t row_elems = (int64_t)Hk * D;
    const int64_t slab_off = (int64_t)slab * HS * D;
    int b = ctl.b0;
    int64_t pb = ctl.pb0;
    int ctx_b = load_ctx(a.context_lens, b, cap);
    int nb = (ctx_b + T - 1) / T;
    constexpr int ROWS_PER_LANE = (2 * T + 31) / 32;
    for (int64_t it = 0; it < n_tiles; ++it) {
      const int64_t x = x0 + it;
      while (x >= pb + nb && b + 1 < B) {
        pb += nb;
        ++b;
        ctx_b = load_ctx(a.context_lens, b, cap);
        nb = (ctx_b + T - 1) / T;
      }
      const int s = (int)(it % C::STAGES);
      const int lt = (int)(x - pb);
      const int tok0 = lt * T;
      const int count = min(T, ctx_b - tok0);  // <= 0 only if context_lens changed mid-run
      int flags = 0;
      if (x == x0 || lt == 0) flags |= kFlagFirst;
      if (x == x1 - 1 || lt == nb - 1) flags |= kFlagLast;
      if (pb >= x0 && pb + nb <= x1) flags |= kFlagWhole;

      // FUSED: the last tile of a sequence holds its newest position ctx_b - 1, always as
      // the tile's last row. It is taken from k_new/v_new and stored when slot_mapping[b]
      // is that position's slot; -1 leaves the cache row as it is; any other slot is an
      // error (flagged, not stored), because another row of the cache may be read by
      // this very launch.
      int new_row = -1;
      int64_t new_slot = -1;
      if (FUSED && lt == nb - 1 && count > 0) {
        const int pos = ctx_b - 1;
        const int32_t sl = __ldg(a.slot_mapping + b);
        if (sl != -1) {
          const int blk = __ldg(a.block_tables + (int64_t)b * a.max_blocks + pos / a.block_size);
          const int64_t want = (blk >= 0 && (int64_t)blk < a.num_blocks)
                                   ? (int64_t)blk * a.block_size + pos % a.block_size
                                   : -2;
          if ((int64_t)sl == want) {
            new_row = count - 1;
            new_slot = want;
          } else if (lane == 0 && slab == 0) {
            set_dev_err(a.dev_err, PA_DEV_ERR_SLOT);
          }
        }
      }

      // The rows of a tile are one contiguous run when the slab is every KV head and the
      // tile sits inside one block: then lane 0 moves K and V with one copy each.
      const int pos_first = tok0, pos_last = tok0 + count - 1;
      const bool one_run = slab_off == 0 && row_elems == (int64_t)HS * D &&
                           count > 0 && (pos_first / a.block_size) == (pos_last / a.block_size);
      const uint16_t* src[ROWS_PER_LANE];
      int ok_rows = 0;
      if (one_run) {
#pragma unroll
        for (int k = 0; k < ROWS_PER_LANE; ++k) src[k] = nullptr;
        const int blk = __ldg(a.block_tables + (int64_t)b * a.max_blocks + pos_first / a.block_size);
        // lanes 0 / 1: the K / V run from the cache; FUSED lanes 2 / 3: the new K / V row
        const int run_rows = new_row >= 0 ? count - 1 : count;
        if (blk >= 0 && (int64_t)blk < a.num_blocks) {
          const int64_t rowi = (int64_t)blk * a.block_size + pos_first % a.block_size;
          if (lane < 2 && run_rows > 0) {
            src[0] = (lane ? vc : kc) + rowi * row_elems;
            ok_rows = run_rows;
          }
        } else if (lane == 0) {
          set_dev_err(a.dev_err, PA_DEV_ERR_BLOCK_ID);
        }
        if (FUSED && new_row >= 0 && (lane == 2 || lane == 3)) {
          src[0] = lane == 2 ? static_cast<const uint16_t*>(a.k_new) + (int64_t)b * a.k_new_stride
                             : static_cast<const uint16_t*>(a.v_new) + (int64_t)b * a.v_new_stride;
          ok_rows = 1;
        }
      } else {
#pragma unroll
      for (int k = 0; k < ROWS_PER_LANE; ++k) {
        src[k] = nullptr;
        const int r = lane + 32 * k;
        if (r < 2 * T) {
          const int kv = r >= T;
          const int t = kv ? r - T : r;
          if (FUSED && t == new_row) {
            src[k] = (kv ? static_cast<const uint16_t*>(a.v_new) + (int64_t)b * a.v_new_stride
                         : static_cast<const uint16_t*>(a.k_new) + (int64_t)b * a.k_new_stride) +
                     slab_off;
            ++ok_rows;
          } else if (t < count) {
            const int pos = tok0 + t;
            const int blk = __ldg(a.block_tables + (int64_t)b * a.max_blocks + pos / a.block_size);
            if (blk >= 0 && (int64_t)blk < a.num_blocks) {
              const int64_t rowi = (int64_t)blk * a.block_size + pos % a.block_size;
              src[k] = (kv ? vc : kc) + rowi * row_elems + slab_off;
              ++ok_rows;
            } else if (kv == 0) {
              set_dev_err(a.dev_err, PA_DEV_ERR_BLOCK_ID);
            }
          }
        }
      }
      }
      const int total_rows = __reduce_add_sync(0xffffffffu, ok_rows);
      const bool first = flags & kFlagFirst;
      const uint32_t bytes = (uint32_t)total_rows * C::ROW + (first ? C::Q_BYTES : 0);

      if (it >= C::STAGES) {
        if (!mbar_wait(&ctl.empty[s], (uint32_t)(((it / C::STAGES) - 1) & 1), abort_flag)) {
          if (lane == 0) {
            ctl.abort = 1;
            set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
          }
        }
      }
#ifdef PA_TEST_DELAY_LAST_TILE_CYCLES
      // test build only: hold back the last tile's copies longer than the consumers' wait
      // limit, so that their wait on it runs out (the copies are still issued, late, and
      // drained below; nothing follows them in the ring)
      if (it == n_tiles - 1) {
        const long long t_hold = clock64();
        while (clock64() - t_hold < (long long)(PA_TEST_DELAY_LAST_TILE_CYCLES)) {
        }
      }
#endif
      unsigned char* st = smem + (size_t)s * C::STAGE_BYTES;
      if (lane == 0) {
        StageMeta& m = ctl.meta[s];
        m.pb = pb;
        m.b = b;
        m.tok0 = tok0;
        m.count = count;
        m.nb = nb;
        m.flags = flags;
        m.new_row = new_row;
        m.new_slot = new_slot;
        mbar_arrive_expect_tx(&ctl.full[s], bytes);
      }
      __syncwarp();
      if (one_run) {
        if (src[0] != nullptr) {
          const int kv = lane & 1;
          const int row0 = lane < 2 ? 0 : new_row;
          bulk_g2s_hint(st + kv * C::KV_BYTES + row0 * C::ROW, src[0], (uint32_t)ok_rows * C::ROW,
                        &ctl.full[s], policy);
        }
      } else {
#pragma unroll
      for (int k = 0; k < ROWS_PER_LANE; ++k) {
        const int r = lane + 32 * k;
        if (src[k] != nullptr) {
          const int kv = r >= T;
          const int t = kv ? r - T : r;
          bulk_g2s_hint(st + kv * C::KV_BYTES + t * C::ROW, src[k], C::ROW, &ctl.full[s], policy);
        }
      }
      }
      if (first && lane == 0) {
        const uint16_t* qsrc = static_cast<const uint16_t*>(a.q) +
                               ((int64_t)b * H + (int64_t)slab * HS * G) * D;
        bulk_g2s(st + 2 * C::KV_BYTES, qsrc, C::Q_BYTES, &ctl.full[s]);
      }
    }
    // drain: the last issued stages must land before the CTA may exit (waited with the
    // full limit even after a timeout elsewhere)
    const int64_t first_drain = n_tiles > C::STAGES ? n_tiles - C::STAGES : 0;
    for (int64_t it = first_drain; it < n_tiles; ++it) {
      const int s = (int)(it % C::STAGES);
      mbar_wait_copies(&ctl.full[s], (uint32_t)((it / C::STAGES) & 1));
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int j = warp / C::WPH;  // KV head within the slab
  const int w = warp % C::WPH;  // token group within the tile
  const int half = lane >> 4;
  const int sub = lane & 15;
  const int kvh = slab * HS + j;  // global KV head
  const int kb = bfly_base<C::NV>(sub);
  float* pbuf = pbuf_all + warp * C::PBUF_FLOATS;

  float2 qp[G][DPL / 2];  // q of the group's heads, this lane's DPL dims, pre-scaled
  float2 op[G][DPL / 2];  // running output, this lane's DPL dims
  float m_run[G];
  float m_own[C::CF];
  float l_loc[C::CF];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m_run[hh] = -INFINITY;
#pragma unroll
    for (int c2 = 0; c2 < DPL / 2; ++c2) op[hh][c2] = make_float2(0.f, 0.f), qp[hh][c2] = op[hh][c2];
  }
#pragma unroll
  for (int r = 0; r < C::CF; ++r) m_own[r] = -INFINITY, l_loc[r] = 0.f;
  const float2 scale2 = make_float2(a.scale_log2, a.scale_log2);

  int seg_count = 0;
  for (int64_t it = 0; it < n_tiles; ++it) {
    const int s = (int)(it % C::STAGES);
    if (!mbar_wait(&ctl.full[s], (uint32_t)((it / C::STAGES) & 1), abort_flag)) {
      if (lane == 0) {
        ctl.abort = 1;
        set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
      }
    }
    const StageMeta meta = ctl.meta[s];
    const unsigned char* Kst = smem + (size_t)s * C::STAGE_BYTES;
    const unsigned char* Vst = Kst + C::KV_BYTES;
    const int count = meta.count;

    if (meta.flags & kFlagFirst) {
      const unsigned char* Qst = Kst + 2 * C::KV_BYTES;
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const LaneVec<DPL> qv = ld_lane<DPL>(Qst + ((j * G + hh) * D + sub * DPL) * 2);
#pragma unroll
        for (int c2 = 0; c2 < DPL / 2; ++c2) qp[hh][c2] = mul2(elt2_f2<F16>(qv.w[c2]), scale2);
#pragma unroll
        for (int c2 = 0; c2 < DPL / 2; ++c2) op[hh][c2] = make_float2(0.f, 0.f);
        m_run[hh] = -INFINITY;
      }
#pragma unroll
      for (int r = 0; r < C::CF; ++r) m_own[r] = -INFINITY, l_loc[r] = 0.f;
    }

    // ---- this warp's rows of the tile: K now, V early (in-bounds shared loads) ---------
    LaneVec<DPL> kraw[kPairs], vraw[kPairs];
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const int t = w * kTokPerWarp + 2 * i + half;
      const size_t off = (size_t)(t * HS + j) * (D * 2) + sub * (DPL * 2);
      kraw[i] = ld_lane<DPL>(Kst + off);
      vraw[i] = ld_lane<DPL>(Vst + off);
      if (t >= count) vraw[i] = zero_lane<DPL>();  // stale rows must not reach p*v
    }
    if constexpr (FUSED) {
      // the new token's row of KV head kvh: its half-warp writes it to the cache slot
      if (meta.new_row >= 0) {
        const int64_t dst = meta.new_slot * ((int64_t)Hk * D) + (int64_t)kvh * D + sub * DPL;
#pragma unroll
        for (int i = 0; i < kPairs; ++i) {
          if (w * kTokPerWarp + 2 * i + half == meta.new_row) {
            st_lane<DPL>(static_cast<uint16_t*>(const_cast<void*>(a.k_cache)) + dst, kraw[i]);
            st_lane<DPL>(static_cast<uint16_t*>(const_cast<void*>(a.v_cache)) + dst, vraw[i]);
          }
        }
      }
    }

    // ---- scores: q . k, DPL dims per lane, reduced over the 16 lanes of a row ----------
    float sc[C::NV];
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      float2 kf[DPL / 2];
#pragma unroll
      for (int c2 = 0; c2 < DPL / 2; ++c2) kf[c2] = elt2_f2<F16>(kraw[i].w[c2]);
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float2 acc = mul2(qp[hh][0], kf[0]);
#pragma unroll
        for (int c2 = 1; c2 < DPL / 2; ++c2) acc = fma2(qp[hh][c2], kf[c2], acc);
        sc[i * G + hh] = acc.x + acc.y;
      }
    }
    bfly<C::NV>(sc, sub, 8);
    bfly<Half<C::NV>::v>(sc, sub, 4);
    bfly<Half<Half<C::NV>::v>::v>(sc, sub, 2);
    bfly<Half<Half<Half<C::NV>::v>::v>::v>(sc, sub, 1);

    // ---- online softmax --------------------------------------------------------------
    float tm[C::CF];
    bool valid[C::CF];
#pragma unroll
    for (int r = 0; r < C::CF; ++r) {
      const int kk = kb + r;
      const int i = kk / G;
      const int t = w * kTokPerWarp + 2 * i + half;
      valid[r] = t < count;
      sc[r] = valid[r] ? sc[r] : -INFINITY;
      float v = sc[r];
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
      tm[r] = v;
    }
    float alpha[G];
    bool rescale = false;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float t_max = head_bcast<G, C::CF>(tm, hh, lane);
      const float m_new = fmaxf(m_run[hh], t_max);
      alpha[hh] = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run[hh] - m_new);
      rescale |= (m_new != m_run[hh]);
      m_run[hh] = m_new;
    }
#pragma unroll
    for (int r = 0; r < C::CF; ++r) {
      const float m_new = fmaxf(m_own[r], tm[r]);
      const float al = (m_new == -INFINITY) ? 1.f : fast_exp2(m_own[r] - m_new);
      const float p = valid[r] ? fast_exp2(sc[r] - m_new) : 0.f;
      l_loc[r] = l_loc[r] * al + p;
      m_own[r] = m_new;
      pbuf[half * kPairs * G + kb + r] = p;
    }
    __syncwarp();
    float pv[kPairs * G];
#pragma unroll
    for (int k = 0; k < kPairs * G / 4; ++k) {
      const float4 f = *reinterpret_cast<const float4*>(pbuf + half * kPairs * G + 4 * k);
      pv[4 * k + 0] = f.x;
      pv[4 * k + 1] = f.y;
      pv[4 * k + 2] = f.z;
      pv[4 * k + 3] = f.w;
    }
    __syncwarp();
    if (rescale) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float2 al2 = make_float2(alpha[hh], alpha[hh]);
#pragma unroll
        for (int c2 = 0; c2 < DPL / 2; ++c2) op[hh][c2] = mul2(op[hh][c2], al2);
      }
    }
    // ---- o += p v ----------------------------------------------------------------------
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      float2 vf[DPL / 2];
#pragma unroll
      for (int c2 = 0; c2 < DPL / 2; ++c2) vf[c2] = elt2_f2<F16>(vraw[i].w[c2]);
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float2 p2 = make_float2(pv[i * G + hh], pv[i * G + hh]);
#pragma unroll
        for (int c2 = 0; c2 < DPL / 2; ++c2) op[hh][c2] = fma2(p2, vf[c2], op[hh][c2]);
      }
    }

    if (meta.flags & kFlagLast) {
      // ---- finalize the segment ----------------------------------------------------
      // (1) fold the two half-warps (tokens 2i and 2i+1) and total the softmax sums
      float o[G][DPL];
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int c2 = 0; c2 < DPL / 2; ++c2) {
          o[hh][2 * c2] = op[hh][c2].x + __shfl_xor_sync(0xffffffffu, op[hh][c2].x, 16);
          o[hh][2 * c2 + 1] = op[hh][c2].y + __shfl_xor_sync(0xffffffffu, op[hh][c2].y, 16);
        }
      float lt[C::CF];
#pragma unroll
      for (int r = 0; r < C::CF; ++r) {
        float v = l_loc[r];
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        lt[r] = v;
      }
      float l_all[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) l_all[hh] = head_bcast<G, C::CF>(lt, hh, lane);

      // (2) several warps per KV head (slabs below 8 heads): once every consumer warp is
      // done with this stage's K/V, reuse it as scratch to merge their softmax states
      if constexpr (C::WPH > 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.seg_bar);
        if (!mbar_wait(&ctl.seg_bar, (uint32_t)(seg_count & 1), abort_flag)) {
          if (lane == 0) {
            ctl.abort = 1;
            set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
          }
        }
      }
      float* merge = reinterpret_cast<float*>(smem + (size_t)s * C::STAGE_BYTES) +
                     (size_t)j * (C::WPH - 1) * C::MERGE_FLOATS;
      if (w != 0) {
        float* mine = merge + (size_t)(w - 1) * C::MERGE_FLOATS;
        if (half == 0) {
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float4* d4 = reinterpret_cast<float4*>(mine + hh * D + sub * DPL);
#pragma unroll
            for (int q4 = 0; q4 < DPL / 4; ++q4)
              d4[q4] = make_float4(o[hh][4 * q4], o[hh][4 * q4 + 1], o[hh][4 * q4 + 2], o[hh][4 * q4 + 3]);
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            mine[G * D + hh] = m_run[hh];
            mine[G * D + G + hh] = l_all[hh];
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.merge_bar[j]);
      } else {
        if constexpr (C::WPH > 1) {
          if (!mbar_wait(&ctl.merge_bar[j], (uint32_t)(seg_count & 1), abort_flag)) {
            if (lane == 0) {
              ctl.abort = 1;
              set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
            }
          }
        }
        for (int w2 = 1; w2 < C::WPH; ++w2) {
          const float* other = merge + (size_t)(w2 - 1) * C::MERGE_FLOATS;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const float m2 = other[G * D + hh];
            const float l2 = other[G * D + G + hh];
            const float mm = fmaxf(m_run[hh], m2);
            const float a1 = (mm == -INFINITY) ? 0.f : fast_exp2(m_run[hh] - mm);
            const float a2 = (mm == -INFINITY) ? 0.f : fast_exp2(m2 - mm);
            float ov[DPL];
#pragma unroll
            for (int q4 = 0; q4 < DPL / 4; ++q4) {
              const float4 p4 = lds128f(other + hh * D + sub * DPL + 4 * q4);
              ov[4 * q4] = p4.x, ov[4 * q4 + 1] = p4.y, ov[4 * q4 + 2] = p4.z, ov[4 * q4 + 3] = p4.w;
            }
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[hh][e] = o[hh][e] * a1 + ov[e] * a2;
            l_all[hh] = l_all[hh] * a1 + l2 * a2;
            m_run[hh] = mm;
          }
        }
        // (3) normalise and write the row, or the partial for the combine
        const int b = meta.b;
        if (meta.flags & kFlagWhole) {
          if (half == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
              const int hg = kvh * G + hh;
              const float inv = l_all[hh] > 0.f ? 1.f / l_all[hh] : 0.f;
              LaneVec<DPL> pk;
#pragma unroll
              for (int c2 = 0; c2 < DPL / 2; ++c2)
                pk.w[c2] = f2_elt2<F16>(o[hh][2 * c2] * inv, o[hh][2 * c2 + 1] * inv);
              st_lane<DPL>(static_cast<uint16_t*>(a.out) + ((int64_t)b * H + hg) * D + sub * DPL, pk);
            }
          }
        } else {
          const int slot = (x0 < meta.pb) ? 1 : 0;
          if (half == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
              const int hg = kvh * G + hh;
              const float inv = l_all[hh] > 0.f ? 1.f / l_all[hh] : 0.f;
              float4* d4 = reinterpret_cast<float4*>(
                  a.part_o + (((int64_t)c * 2 + slot) * H + hg) * D + sub * DPL);
#pragma unroll
              for (int q4 = 0; q4 < DPL / 4; ++q4)
                d4[q4] = make_float4(o[hh][4 * q4] * inv, o[hh][4 * q4 + 1] * inv,
                                     o[hh][4 * q4 + 2] * inv, o[hh][4 * q4 + 3] * inv);
            }
          }
          if (lane == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
              const int hg = kvh * G + hh;
              a.part_lse[((int64_t)c * 2 + slot) * H + hg] =
                  (l_all[hh] > 0.f) ? m_run[hh] + fast_log2(l_all[hh]) : -INFINITY;
            }
          }
          __threadfence();
          __syncwarp();
          int old = 0;
          int* counter = a.counters + (int64_t)b * Hk + kvh;
          if (lane == 0) old = atomicAdd(counter, 1);
          old = __shfl_sync(0xffffffffu, old, 0);
          const int64_t c_lo = cta_of(meta.pb, NT, g_eff);
          const int64_t c_hi = cta_of(meta.pb + meta.nb - 1, NT, g_eff);
          const int nseg = (int)(c_hi - c_lo + 1);
          if (old == nseg - 1) {
            // (4) last arrival: combine the partials of sequence b in CTA order
            __threadfence();
            combine_partials<D, F16, G>(a, b, kvh, G, c_lo, nseg, NT, g_eff, meta.pb, lane);
            if (lane == 0) *counter = 0;  // leave the counter zero for the next call
          }
        }
      }
      ++seg_count;
      fence_proxy_async_smem();
    }
    // order this tile's shared-memory reads before the producer's next copy into the stage
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.empty[s]);
  }
}

// Launch with programmatic stream serialization: the grid may be scheduled while the
// previous kernel on the stream is still running (its CTAs run the prologue, then wait in
// pdl_wait for that kernel to complete before using anything it wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

template <int HS, int G, bool FUSED, int D, bool F16>
int launch_decode_t(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  using C = DecCfg<HS, G, D>;
  static std::atomic<bool> attr_done[64];  // zero-initialised: false
  const int dev = info.device;
  if (dev < 0 || dev >= 64) return PA_ERR_CUDA;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(paged_decode_kernel<HS, G, FUSED, D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int slabs = a.num_kv_heads / HS;
  dim3 grid((unsigned)a.grid_ctas, (unsigned)slabs);
  if (launch_dependent(paged_decode_kernel<HS, G, FUSED, D, F16>, grid, dim3(kThreads), C::SMEM,
                       stream, a) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <int HS, bool FUSED, int D, bool F16>
int dispatch_group(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  switch (a.num_heads / a.num_kv_heads) {
    case 1: return launch_decode_t<HS, 1, FUSED, D, F16>(a, info, stream);
    case 2: return launch_decode_t<HS, 2, FUSED, D, F16>(a, info, stream);
    default: return PA_ERR_UNSUPPORTED;  // larger groups take the tensor-core kernel
  }
}

// Every head slab for one (FUSED, D, element type) combination.
template <bool FUSED, int D, bool F16>
int dispatch_slab(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  switch (decode_head_slab(a.num_kv_heads)) {
    case 8: return dispatch_group<8, FUSED, D, F16>(a, info, stream);
    case 4: return dispatch_group<4, FUSED, D, F16>(a, info, stream);
    case 2: return dispatch_group<2, FUSED, D, F16>(a, info, stream);
    default: return dispatch_group<1, FUSED, D, F16>(a, info, stream);
  }
}

}  // namespace
}  // namespace pa
