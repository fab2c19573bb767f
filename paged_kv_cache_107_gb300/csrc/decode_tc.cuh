// decode_tc.cuh — paged decode attention for groups of 1 to 8 query heads per KV head on
// the tensor cores (warp-level mma.sync m16n8k16, bf16 or fp16 operands, fp32 accumulators).
//
// Same computation and same work split as decode_kernel.cuh ("nano-vllm解读", sections
// "PageAttention原理" and "Nano-vllm中的使用"; stream-K over key tiles, partials combined in
// CTA order by the last CTA of a sequence). With G query heads per KV head the per-head work
// is a small dense product: S = Q_j K^T (G x T) and O += P V (G x D). On CUDA cores its dot
// products, reductions and accumulations outgrow the instruction budget of the HBM stream
// once G >= 4 (and G = 8 no longer fits in registers); here one warp runs them as
// 16-row tensor-core products, the G heads padded to 16 rows. The same kernel takes G = 1
// and 2 wherever its TMA boxes stream faster than the CUDA-core kernel's copies (head_dim
// 64, slabs narrower than the KV row).
//
//  * A stage holds T = 128 * SUB / HS tokens of the slab's HS KV heads (SUB = 2 at head_dim
//    64, else 1, so that a stage always carries 64 KB), K then V, each as D/64 halves laid
//    out [head][token][64 dims]: 128-byte rows with the 128-byte swizzle, so the 8 token
//    rows an ldmatrix reads sit in 8 different bank groups. The producer fills it with TMA
//    boxes of tb tokens x HS heads x 64 dims (tb = the largest power of two dividing
//    block_size, at most T), i.e. 2 * D/64 * T/tb copies per stage; a block size with no
//    such tb >= 8 is filled with 16-byte cp.async copies into the same layout.
//  * Launched as a programmatic dependent (decode_kernel.cuh's launch_dependent): the
//    prologue reads only context_lens; before waiting for the previous grid the producer
//    prefetches its first tiles' K/V runs into L2.
//  * The fused step's new token: its K and V rows of the slab come from k_new / v_new into
//    a side row of the stage; lanes whose token is the new one point ldmatrix there.
//  * Q of a segment goes to its own slot (two where shared memory allows), loaded once per
//    sequence and released as soon as every warp holds its fragments.
//  * Warp (j, w): KV head j of the slab, SUB blocks of 16 tokens of each tile. S: for every
//    16-dim chunk, ldmatrix.x4 gives the K fragments of two 8-token column tiles. Online
//    softmax in the accumulator layout (a row's 16 scores sit in one quad of lanes); the S
//    accumulators become the A operand of O += P V directly; V fragments come from
//    ldmatrix.x4.trans. Rows of V past the context are zeroed first, so no stale value
//    meets a zero probability.
#pragma once

#include <atomic>
#include <cuda.h>
#include <string.h>

#include "decode_kernel.cuh"
#include "tensor_map.h"

namespace pa {
namespace {

constexpr int kTcGMax = 8;   // query heads per KV head on this path (rows of the 16-row tile)

template <int S>
struct TcCtrl {
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t seg_bar;
  uint64_t merge_bar[8];
  StageMeta meta[S];
  int64_t nt;      // tiles in the stream
  int64_t x0, x1;  // this CTA's tile range
  int64_t pb0;     // first tile of the sequence holding x0
  int b0;
  int g_eff;       // CTAs that own tiles
  int found;
  int abort;
  int64_t red[32];
};

template <int HS, int D>
struct TcCfg {
  // a warp takes SUB blocks of 16 tokens per stage: two at head_dim 64, so that a stage
  // carries as many bytes as at head_dim 128 and the per-stage costs (barriers, block
  // lookups, copies) are spread over twice the tokens
  static constexpr int SUB = D == 64 ? 2 : 1;
  static constexpr int T = 128 * SUB / HS;         // tokens per stage (8 warps x 16 x SUB / HS)
  static constexpr int WPH = kConsumerWarps / HS;  // warps per KV head (token split)
  static constexpr int NH = D / 64;                // 64-dim halves of a head row
  static constexpr int HALF = HS * T * 128;        // bytes of one half: [head][token][64 dims]
  static constexpr int KV_BYTES = NH * HALF;
  static constexpr int SIDE_ROW = HS * D * 2;      // the new token's K (or V) row of the slab
  static constexpr int STAGE_BYTES = (2 * KV_BYTES + 2 * SIDE_ROW + 1023) / 1024 * 1024;
  static constexpr int Q_BYTES = HS * kTcGMax * D * 2;
  static constexpr int CTRL_BYTES = 1024;
  static constexpr int BUDGET = 227 * 1024 - 1024 - CTRL_BYTES;  // less the alignment slack
  static constexpr int QS = (3 * STAGE_BYTES + 2 * Q_BYTES <= BUDGET) ? 2 : 1;
  static constexpr int FIT = (BUDGET - QS * Q_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = FIT < 6 ? FIT : 6;
  static constexpr int MERGE_FLOATS = kTcGMax * (D + 2);
  static constexpr size_t SMEM =
      1024 + (size_t)STAGES * STAGE_BYTES + (size_t)QS * Q_BYTES + CTRL_BYTES;
  static_assert(STAGES >= 2, "at least two stages");
  static_assert(sizeof(TcCtrl<STAGES>) <= CTRL_BYTES, "control block");
  static_assert(HS * (WPH - 1) * MERGE_FLOATS * 4 <= 2 * KV_BYTES, "merge scratch");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// D (16x8) += A (16x16) B (16x8) with rows 8..15 of A zero (at most 8 heads per group):
// a0/a2 are this thread's A words of row gid, c0/c1 its accumulators of row gid; the
// accumulators of rows 8..15 go to the scratch pair z (written, never read).
template <bool F16>
__device__ __forceinline__ void mma16816(float& c0, float& c1, float2& z, uint32_t a0, uint32_t a2,
                                         uint32_t b0, uint32_t b1) {
  const uint32_t zero = 0u;
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c0), "+f"(c1), "+f"(z.x), "+f"(z.y)
        : "r"(a0), "r"(zero), "r"(a2), "r"(zero), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c0), "+f"(c1), "+f"(z.x), "+f"(z.y)
        : "r"(a0), "r"(zero), "r"(a2), "r"(zero), "r"(b0), "r"(b1));
  }
}
// ldmatrix x4 (plain and transposed) from a 32-bit shared-memory address
__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// One TMA box (4-D tensor map) into shared memory, completion counted on `bar` in bytes,
// with an L2 eviction-priority hint.
__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* map, int c0, int c1,
                                                 int c2, int c3, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 16-byte asynchronous copy global -> shared (both 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
// The barrier counts one more arrival, made when this thread's cp.async copies so far land.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int HS, bool FUSED, int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a,
                           const int tb) {
  using TC = TcCfg<HS, D>;
  constexpr int S = TC::STAGES;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* qbuf = smem + (size_t)S * TC::STAGE_BYTES;
  TcCtrl<S>& ctl = *reinterpret_cast<TcCtrl<S>*>(qbuf + (size_t)TC::QS * TC::Q_BYTES);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;
  const int slab = blockIdx.y;
  const int H = a.num_heads;
  const int Hk = a.num_kv_heads;
  const int G = H / Hk;  // 1..8
  const int cap = a.max_blocks * a.block_size;
  const int B = a.num_seqs;
  constexpr int T = TC::T;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kConsumerWarps);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&ctl.q_full[q], 1);
      mbar_init(&ctl.q_empty[q], kConsumerWarps);
    }
    mbar_init(&ctl.seg_bar, kConsumerWarps);
    if (TC::WPH > 1)
      for (int j = 0; j < HS; ++j) mbar_init(&ctl.merge_bar[j], TC::WPH - 1);
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
  // tiles (lanes 2t, 2t+1: K, V of tile t), as the CUDA-core kernel does; only when the
  // slab is every KV head, so that a tile inside one block is one run of cache rows.
  if (warp == kProducerWarp && x0 < x1 && ctl.found && lane < 2 * S) {
    const int64_t row_elems = (int64_t)Hk * D;
    if (slab == 0 && Hk == HS && x0 + (lane >> 1) < x1) {
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
    if (tb > 0 && lane == 0) {
      prefetch_tensor_map(&tm_k);
      prefetch_tensor_map(&tm_v);
    }
    const uint16_t* kc = static_cast<const uint16_t*>(a.k_cache);
    const uint16_t* vc = static_cast<const uint16_t*>(a.v_cache);
    const int64_t row_elems = (int64_t)Hk * D;
    const int64_t slab_off = (int64_t)slab * HS * D;
    const int box_bytes = HS * tb * 128;  // one box: HS heads x tb tokens x 64 dims
    const int nbx = tb > 0 ? T / tb : 0;  // boxes per half
    int b = ctl.b0;
    int64_t pb = ctl.pb0;
    int ctx_b = load_ctx(a.context_lens, b, cap);
    int nb = (ctx_b + T - 1) / T;
    int q_n = 0;  // segments whose Q has been issued
    for (int64_t it = 0; it < n_tiles; ++it) {
      const int64_t x = x0 + it;
      while (x >= pb + nb && b + 1 < B) {
        pb += nb;
        ++b;
        ctx_b = load_ctx(a.context_lens, b, cap);
        nb = (ctx_b + T - 1) / T;
      }
      const int s = (int)(it % S);
      const int lt = (int)(x - pb);
      const int tok0 = lt * T;
      const int count = min(T, ctx_b - tok0);
      int flags = 0;
      if (x == x0 || lt == 0) flags |= kFlagFirst;
      if (x == x1 - 1 || lt == nb - 1) flags |= kFlagLast;
      if (pb >= x0 && pb + nb <= x1) flags |= kFlagWhole;
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
      // this lane's box: tokens tok0 + lane*tb .. +tb-1, inside one block
      int blk = -1, off = 0;
      bool box_ok = false;
      if (lane < nbx && lane * tb < count) {
        const int pos = tok0 + lane * tb;
        blk = __ldg(a.block_tables + (int64_t)b * a.max_blocks + pos / a.block_size);
        off = pos % a.block_size;
        box_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
        if (!box_ok) set_dev_err(a.dev_err, PA_DEV_ERR_BLOCK_ID);
      }
      const int nbox = __popc(__ballot_sync(0xffffffffu, box_ok));
      if (it >= S) {
        if (!mbar_wait(&ctl.empty[s], (uint32_t)(((it / S) - 1) & 1), abort_flag)) {
          if (lane == 0) {
            ctl.abort = 1;
            set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
          }
        }
      }
      unsigned char* st = smem + (size_t)s * TC::STAGE_BYTES;
      unsigned char* side = st + 2 * TC::KV_BYTES;
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
        if (tb > 0)
          mbar_arrive_expect_tx(&ctl.full[s], (uint32_t)(nbox * 2 * TC::NH * box_bytes +
                                                         (new_row >= 0 ? 2 * TC::SIDE_ROW : 0)));
      }
      __syncwarp();
      if (tb > 0) {
        if (box_ok) {
#pragma unroll
          for (int h = 0; h < TC::NH; ++h) {
            tma_load_4d_hint(st + h * TC::HALF + lane * box_bytes, &tm_k, h * 64, off, slab * HS,
                             blk, &ctl.full[s], policy);
            tma_load_4d_hint(st + TC::KV_BYTES + h * TC::HALF + lane * box_bytes, &tm_v, h * 64,
                             off, slab * HS, blk, &ctl.full[s], policy);
          }
        }
        if (FUSED && new_row >= 0 && lane == 0) {
          bulk_g2s(side, static_cast<const uint16_t*>(a.k_new) + (int64_t)b * a.k_new_stride + slab_off,
                   TC::SIDE_ROW, &ctl.full[s]);
          bulk_g2s(side + TC::SIDE_ROW,
                   static_cast<const uint16_t*>(a.v_new) + (int64_t)b * a.v_new_stride + slab_off,
                   TC::SIDE_ROW, &ctl.full[s]);
        }
      } else {
        // 16-byte copies into the same swizzled layout, one box of T tokens per half
        constexpr int CH = D / 8;  // 16-byte chunks of one head's row
        const int per_kv = count * HS * CH;
        for (int i = lane; i < 2 * per_kv; i += 32) {
          const int kv = i >= per_kv;
          const int r = kv ? i - per_kv : i;
          const int t = r / (HS * CH);
          const int jj = (r / CH) % HS;
          const int ch = r % CH;
          if (FUSED && t == new_row) {
            const uint16_t* src =
                (kv ? static_cast<const uint16_t*>(a.v_new) + (int64_t)b * a.v_new_stride
                    : static_cast<const uint16_t*>(a.k_new) + (int64_t)b * a.k_new_stride) +
                slab_off + jj * D + ch * 8;
            cp_async16(side + kv * TC::SIDE_ROW + (jj * D + ch * 8) * 2, src);
          } else {
            const int pos = tok0 + t;
            const int bk = __ldg(a.block_tables + (int64_t)b * a.max_blocks + pos / a.block_size);
            if (bk < 0 || (int64_t)bk >= a.num_blocks) {
              if (kv == 0 && jj == 0 && ch == 0) set_dev_err(a.dev_err, PA_DEV_ERR_BLOCK_ID);
              continue;
            }
            const int64_t rowi = (int64_t)bk * a.block_size + pos % a.block_size;
            const uint16_t* src = (kv ? vc : kc) + rowi * row_elems + slab_off + jj * D + ch * 8;
            cp_async16(st + kv * TC::KV_BYTES + (ch >> 3) * TC::HALF + (jj * T + t) * 128 +
                           (((ch & 7) ^ (t & 7)) << 4),
                       src);
          }
        }
        cp_async_arrive(&ctl.full[s]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.full[s]);
      }
      if (flags & kFlagFirst) {
        // Q of the segment (HS*G rows of D, contiguous) into its slot
        const int qs = q_n % TC::QS;
        if (q_n >= TC::QS) {
          if (!mbar_wait(&ctl.q_empty[qs], (uint32_t)(((q_n / TC::QS) - 1) & 1), abort_flag)) {
            if (lane == 0) {
              ctl.abort = 1;
              set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
            }
          }
        }
        if (lane == 0) {
          const uint32_t q_bytes = (uint32_t)(HS * G * D * 2);
          mbar_arrive_expect_tx(&ctl.q_full[qs], q_bytes);
          bulk_g2s(qbuf + (size_t)qs * TC::Q_BYTES,
                   static_cast<const uint16_t*>(a.q) + ((int64_t)b * H + (int64_t)slab * HS * G) * D,
                   q_bytes, &ctl.q_full[qs]);
        }
        ++q_n;
      }
    }
    // copies still in flight land before the producer leaves (bounded waits, the full
    // limit even after a timeout elsewhere)
    const int64_t first_drain = n_tiles > S ? n_tiles - S : 0;
    for (int64_t it = first_drain; it < n_tiles; ++it) {
      const int s = (int)(it % S);
      mbar_wait_copies(&ctl.full[s], (uint32_t)((it / S) & 1));
    }
    for (int n = q_n > TC::QS ? q_n - TC::QS : 0; n < q_n; ++n)
      mbar_wait_copies(&ctl.q_full[n % TC::QS], (uint32_t)((n / TC::QS) & 1));
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int j = warp / TC::WPH;   // KV head within the slab
  const int w = warp % TC::WPH;   // token group within the tile
  const int kvh = slab * HS + j;  // global KV head
  // mma fragment coordinates: this thread holds row gid (a query head of the group; rows
  // 8..15 of the 16-row tile are padding) and columns 2tig, 2tig+1 of each 8-column tile
  const int gid = lane >> 2, tig = lane & 3;
  const bool row_ok = gid < G;
  constexpr int KC = D / 16;      // 16-dim chunks
  constexpr int NO = D / 8;       // 8-dim output column tiles
  uint32_t qa[KC][2];             // Q fragments of row gid: dims 16kc + 2tig(+1), +8
  float o[NO][2];                 // O accumulators of row gid: dims 8n + 2tig, +1
  float2 z = make_float2(0.f, 0.f);  // accumulators of the padding rows (never read)
  float m_run = -INFINITY, l_part = 0.f;  // row gid: running max (log2 units), partial sum
#pragma unroll
  for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = 0.f;
  const float sl2 = a.scale_log2;

  // shared-memory row of token t of head j within a half: boxes of tbl tokens, each
  // [head][token]; chunk c of the row sits at chunk c ^ (t % 8)
  const int tbl = tb > 0 ? tb : T;
  const int lg_tbl = __ffs(tbl) - 1;
  const int tw_base = w * 16 * TC::SUB;  // this warp's first token of the tile
  auto row_off = [&](int t) -> int {
    return ((((t >> lg_tbl) * HS + j) << lg_tbl) + (t & (tbl - 1))) * 128;
  };
  const int sw = lane & 7;                                   // = t % 8 of the ldmatrix rows
  const int k_hi = (lane >> 3) & 1, v_hi = lane >> 4;        // second 8 dims of a 16-dim chunk
  // byte offsets within a stage: 16-byte chunk c = 2*(chunk16 % 4) + hi of a 128-byte row sits
  // at (c ^ sw) * 16 = ((chunk16 % 4) * 32 ^ (sw & 6) * 16) + (hi ^ (sw & 1)) * 16
  const uint32_t x_sw = (uint32_t)(sw & 6) << 4;
  const uint32_t ks_lane = (uint32_t)(2 * TC::KV_BYTES + (j * D + k_hi * 8) * 2);
  const uint32_t vs_lane = (uint32_t)(2 * TC::KV_BYTES + TC::SIDE_ROW + (j * D + v_hi * 8) * 2);
  const uint32_t smem_base = smem_u32(smem);

  int seg_count = 0;
  int q_n = 0;
  for (int64_t it = 0; it < n_tiles; ++it) {
    const int s = (int)(it % S);
    if (!mbar_wait(&ctl.full[s], (uint32_t)((it / S) & 1), abort_flag)) {
      if (lane == 0) {
        ctl.abort = 1;
        set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
      }
    }
    const StageMeta meta = ctl.meta[s];
    unsigned char* Kst = smem + (size_t)s * TC::STAGE_BYTES;
    unsigned char* Vst = Kst + TC::KV_BYTES;
    unsigned char* side = Kst + 2 * TC::KV_BYTES;
    const int count = meta.count;

    if (meta.flags & kFlagFirst) {
      const int qs = q_n % TC::QS;
      if (!mbar_wait(&ctl.q_full[qs], (uint32_t)((q_n / TC::QS) & 1), abort_flag)) {
        if (lane == 0) {
          ctl.abort = 1;
          set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
        }
      }
      const unsigned char* Qst = qbuf + (size_t)qs * TC::Q_BYTES;
#pragma unroll
      for (int kc = 0; kc < KC; ++kc) {
        const unsigned char* r0 = Qst + ((j * G + gid) * D + kc * 16 + 2 * tig) * 2;
        qa[kc][0] = row_ok ? *reinterpret_cast<const uint32_t*>(r0) : 0u;
        qa[kc][1] = row_ok ? *reinterpret_cast<const uint32_t*>(r0 + 16) : 0u;
      }
      // the slot is released before these loads are used: order them before the next
      // segment's bulk copy (async proxy) into the slot
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.q_empty[qs]);
      ++q_n;
#pragma unroll
      for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = 0.f;
      m_run = -INFINITY;
      l_part = 0.f;
    }

#pragma unroll
    for (int u = 0; u < TC::SUB; ++u) {
      const int tw0 = tw_base + u * 16;  // first token of this 16-token block
      const int tK = tw0 + (lane & 7) + ((lane >> 4) << 3);        // ldmatrix row (K, S product)
      const int tV = tw0 + (lane & 7) + (((lane >> 3) & 1) << 3);  // ldmatrix row (V, trans)
      const uint32_t k_lane = (uint32_t)row_off(tK) + ((uint32_t)(k_hi ^ (sw & 1)) << 4);
      const uint32_t v_lane =
          (uint32_t)(TC::KV_BYTES + row_off(tV)) + ((uint32_t)(v_hi ^ (sw & 1)) << 4);
      // rows of this warp's V past the tile's valid tokens: zero them (head j's rows)
      if (tw0 + 16 > count) {
        for (int i = lane; i < 16 * TC::NH * 8; i += 32) {
          const int t = tw0 + i / (TC::NH * 8);
          if (t >= count)
            *reinterpret_cast<uint4*>(Vst + ((i >> 3) % TC::NH) * TC::HALF + row_off(t) + (i & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      bool k_new_lane = false, v_new_lane = false;
      if constexpr (FUSED) {
        // the new token's row of KV head kvh: from the side rows to its cache slot
        if (meta.new_row >= tw0 && meta.new_row < tw0 + 16) {
          const int64_t dst = meta.new_slot * ((int64_t)Hk * D) + (int64_t)kvh * D;
          const int half = lane >> 4, sub = lane & 15;
          if (sub < D / 8) {
            const unsigned char* srcp = side + half * TC::SIDE_ROW + j * D * 2 + sub * 16;
            uint16_t* cache = static_cast<uint16_t*>(const_cast<void*>(half ? a.v_cache : a.k_cache));
            *reinterpret_cast<uint4*>(cache + dst + sub * 8) = *reinterpret_cast<const uint4*>(srcp);
          }
        }
        k_new_lane = tK == meta.new_row;
        v_new_lane = tV == meta.new_row;
      }

      // ---- S = Q K^T for 16 tokens: two 8-token column tiles ----------------------------
      float sc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // row gid, tokens 8n + 2tig, +1
      const uint32_t st_u = smem_base + (uint32_t)s * TC::STAGE_BYTES;
      {
  #pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
          uint32_t r[4];
          uint32_t kp = st_u + k_lane + (kc >> 2) * TC::HALF + (((uint32_t)(kc & 3) << 5) ^ x_sw);
          if constexpr (FUSED) kp = k_new_lane ? st_u + ks_lane + kc * 32 : kp;
          ldsm_x4(r, kp);
          mma16816<F16>(sc[0][0], sc[0][1], z, qa[kc][0], qa[kc][1], r[0], r[1]);
          mma16816<F16>(sc[1][0], sc[1][1], z, qa[kc][0], qa[kc][1], r[2], r[3]);
        }
      }
      // ---- online softmax in the accumulator layout (a row's scores sit in one quad) -----
      float tmax = -INFINITY;
  #pragma unroll
      for (int n = 0; n < 2; ++n)
  #pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = tw0 + n * 8 + 2 * tig + e;
          const float v = t < count ? sc[n][e] * sl2 : -INFINITY;
          sc[n][e] = v;
          tmax = fmaxf(tmax, v);
        }
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float m_new = fmaxf(m_run, tmax);
      const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
      m_run = m_new;
      float p[2][2];
  #pragma unroll
      for (int n = 0; n < 2; ++n)
  #pragma unroll
        for (int e = 0; e < 2; ++e) p[n][e] = (m_new == -INFINITY) ? 0.f : fast_exp2(sc[n][e] - m_new);
      l_part = l_part * alpha + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
  #pragma unroll
        for (int n = 0; n < NO; ++n) {
          o[n][0] *= alpha;
          o[n][1] *= alpha;
        }
      }
      // ---- O += P V: P (row gid x 16 tokens) straight from the S accumulators ------------
      const uint32_t pa0 = f2_elt2<F16>(p[0][0], p[0][1]);  // tokens 2tig, +1
      const uint32_t pa2 = f2_elt2<F16>(p[1][0], p[1][1]);  // tokens 8 + 2tig, +1
      {
  #pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          uint32_t r[4];
          uint32_t vp = st_u + v_lane + (dn >> 2) * TC::HALF + (((uint32_t)(dn & 3) << 5) ^ x_sw);
          if constexpr (FUSED) vp = v_new_lane ? st_u + vs_lane + dn * 32 : vp;
          ldsm_x4_t(r, vp);
          mma16816<F16>(o[2 * dn][0], o[2 * dn][1], z, pa0, pa2, r[0], r[1]);
          mma16816<F16>(o[2 * dn + 1][0], o[2 * dn + 1][1], z, pa0, pa2, r[2], r[3]);
        }
      }

    }

    if (meta.flags & kFlagLast) {
      // ---- finalize the segment ----------------------------------------------------
      float l_all = l_part;
      l_all += __shfl_xor_sync(0xffffffffu, l_all, 1);
      l_all += __shfl_xor_sync(0xffffffffu, l_all, 2);
      // several warps per KV head: merge their softmax states through the stage's K/V
      // shared memory once every consumer warp is done with it
      if constexpr (TC::WPH > 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.seg_bar);
        if (!mbar_wait(&ctl.seg_bar, (uint32_t)(seg_count & 1), abort_flag)) {
          if (lane == 0) {
            ctl.abort = 1;
            set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
          }
        }
      }
      float* merge = reinterpret_cast<float*>(Kst) +
                     (size_t)j * (TC::WPH - 1) * TC::MERGE_FLOATS;
      if (w != 0) {
        float* mine = merge + (size_t)(w - 1) * TC::MERGE_FLOATS;
        if (row_ok) {
#pragma unroll
          for (int n = 0; n < NO; ++n)
            *reinterpret_cast<float2*>(mine + gid * D + n * 8 + 2 * tig) = make_float2(o[n][0], o[n][1]);
          if (tig == 0) {
            mine[kTcGMax * D + gid] = m_run;
            mine[kTcGMax * D + kTcGMax + gid] = l_all;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.merge_bar[j]);
      } else {
        if constexpr (TC::WPH > 1) {
          if (!mbar_wait(&ctl.merge_bar[j], (uint32_t)(seg_count & 1), abort_flag)) {
            if (lane == 0) {
              ctl.abort = 1;
              set_dev_err(a.dev_err, PA_DEV_ERR_TIMEOUT);
            }
          }
        }
        for (int w2 = 1; w2 < TC::WPH; ++w2) {
          const float* other = merge + (size_t)(w2 - 1) * TC::MERGE_FLOATS;
          if (row_ok) {
            const float m2 = other[kTcGMax * D + gid];
            const float l2 = other[kTcGMax * D + kTcGMax + gid];
            const float mm = fmaxf(m_run, m2);
            const float a1 = (mm == -INFINITY) ? 0.f : fast_exp2(m_run - mm);
            const float a2 = (mm == -INFINITY) ? 0.f : fast_exp2(m2 - mm);
#pragma unroll
            for (int n = 0; n < NO; ++n) {
              const float2 ov = *reinterpret_cast<const float2*>(other + gid * D + n * 8 + 2 * tig);
              o[n][0] = o[n][0] * a1 + ov.x * a2;
              o[n][1] = o[n][1] * a1 + ov.y * a2;
            }
            l_all = l_all * a1 + l2 * a2;
            m_run = mm;
          }
        }
        // normalise and write the rows, or the partials for the combine
        const int b = meta.b;
        if (meta.flags & kFlagWhole) {
          if (row_ok) {
            const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
            uint16_t* dst = static_cast<uint16_t*>(a.out) + ((int64_t)b * H + kvh * G + gid) * D;
#pragma unroll
            for (int n = 0; n < NO; ++n)
              *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * tig) =
                  f2_elt2<F16>(o[n][0] * inv, o[n][1] * inv);
          }
        } else {
          const int slot = (x0 < meta.pb) ? 1 : 0;
          if (row_ok) {
            const int hg = kvh * G + gid;
            const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
            float* dst = a.part_o + (((int64_t)c * 2 + slot) * H + hg) * D;
#pragma unroll
            for (int n = 0; n < NO; ++n)
              *reinterpret_cast<float2*>(dst + n * 8 + 2 * tig) = make_float2(o[n][0] * inv, o[n][1] * inv);
            if (tig == 0)
              a.part_lse[((int64_t)c * 2 + slot) * H + hg] =
                  (l_all > 0.f) ? m_run + fast_log2(l_all) : -INFINITY;
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
            combine_partials<D, F16, kTcGMax>(a, b, kvh, G, c_lo, nseg, NT, g_eff, meta.pb, lane);
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

template <int HS, bool FUSED, int D, bool F16>
int launch_decode_tc_t(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  using TC = TcCfg<HS, D>;
  static std::atomic<bool> attr_done[64];  // zero-initialised: false
  const int dev = info.device;
  if (dev < 0 || dev >= 64) return PA_ERR_CUDA;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(paged_decode_tc_kernel<HS, FUSED, D, F16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC::SMEM) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[dev].store(true, std::memory_order_release);
  }
  // tokens per TMA box: the largest power of two dividing block_size, at most a stage's
  // tokens; below 8 the stage is filled by 16-byte cp.async copies instead
  int tb = a.block_size & -a.block_size;
  if (tb > TC::T) tb = TC::T;
  if (tb < 8) tb = 0;
  CUtensorMap mk, mv;
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  if (tb > 0 && (!make_slab_map(&mk, a.k_cache, a.num_kv_heads, D, F16, a.block_size,
                                a.num_blocks, tb, HS) ||
                 !make_slab_map(&mv, a.v_cache, a.num_kv_heads, D, F16, a.block_size,
                                a.num_blocks, tb, HS)))
    return PA_ERR_CUDA;
  const int slabs = a.num_kv_heads / HS;
  dim3 grid((unsigned)a.grid_ctas, (unsigned)slabs);
  if (launch_dependent(paged_decode_tc_kernel<HS, FUSED, D, F16>, grid, dim3(kThreads), TC::SMEM,
                       stream, mk, mv, a, tb) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Every head slab of the tensor-core path for one (FUSED, D, element type) combination.
template <bool FUSED, int D, bool F16>
int dispatch_slab_tc(const DecodeArgs& a, const DeviceInfo& info, cudaStream_t stream) {
  switch (decode_head_slab(a.num_kv_heads)) {
    case 8: return launch_decode_tc_t<8, FUSED, D, F16>(a, info, stream);
    case 4: return launch_decode_tc_t<4, FUSED, D, F16>(a, info, stream);
    case 2: return launch_decode_tc_t<2, FUSED, D, F16>(a, info, stream);
    default: return launch_decode_tc_t<1, FUSED, D, F16>(a, info, stream);
  }
}

}  // namespace
}  // namespace pa
