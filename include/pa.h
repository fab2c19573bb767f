/*
 * pa.h — C ABI of the paged-KV attention library (GB300, sm_103a).
 *
 * The library implements the data-parallel hot path of a paged KV cache as the
 * nano-vllm pages describe it:
 *   - store:   each new token's K/V rows are scattered into k_cache/v_cache at the
 *              row index slot_mapping[i] ("nano-vllm解读", section "KVCache的写入";
 *              "3.6 ModelRunner、CUDA Graph 与性能基准", section 2, prepare_prefill /
 *              prepare_decode, where slot = block_table[pos / block_size] * block_size
 *              + pos % block_size and slot == -1 marks a padding row that is skipped).
 *   - decode:  one query token per sequence attends over the first context_lens[b]
 *              cached tokens, gathered through the -1-padded int32 block table
 *              ("nano-vllm解读", sections "PageAttention原理" and "Nano-vllm中的使用").
 *   - prefill: causal varlen attention of the new tokens of each sequence over its
 *              cached prefix plus the new tokens, the key/value rows read through the
 *              block table ("nano-vllm解读", section "如何适配不同请求不同序列长度";
 *              "3.6 ModelRunner…", section 2, cu_seqlens_q / cu_seqlens_k).
 *
 * Conventions shared by every entry point
 *   - Every pointer named as device memory is caller-owned CUDA device memory on the
 *     current device. The library allocates nothing and frees nothing.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL =
 *     the legacy default stream) and never synchronises the host.
 *   - Element type: 16-bit floats (raw 16-bit storage) for q, k, v, caches and outputs:
 *     bf16, or IEEE binary16 (fp16) where a call takes a `dtype` (pa_dtype). head_dim is
 *     64 or 128; anything else returns PA_ERR_UNSUPPORTED.
 *   - Layouts are C-contiguous unless a stride argument says otherwise:
 *       k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *       block_tables      [num_seqs, max_blocks_per_seq] int32, right-padded with -1
 *   - GQA: query head h reads KV head h / (num_heads / num_kv_heads). Decode (and the fused
 *     step) take 1 to 8 query heads per KV head; prefill takes 1, 2, 4 or 8.
 *   - Host-side validation happens before any launch; when it fails the call returns
 *     the status and launches nothing.
 *   - Data-dependent errors that only the device can see (a block id outside
 *     [0, num_blocks), a slot outside [-1, num_blocks*block_size), a context longer
 *     than max_blocks_per_seq*block_size, a pipeline wait that ran out) never fault:
 *     the offending access is skipped and, when `dev_err` is non-NULL, the matching
 *     PA_DEV_ERR_* bit is OR-ed into *dev_err (device memory, one int). The host reads
 *     it after synchronising. The output rows touched by such an error are undefined.
 */
#ifndef PAGED_KV_PA_H
#define PAGED_KV_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side status codes returned by every entry point. */
enum pa_status {
  PA_OK = 0,
  PA_ERR_NULL = 1,        /* a required pointer is NULL */
  PA_ERR_SHAPE = 2,       /* inconsistent sizes: H % Hk != 0, block_size <= 0, ... */
  PA_ERR_UNSUPPORTED = 3, /* head_dim not 64 or 128, an element type or query-head group
                             the call does not take, or a size beyond the kernels' limits */
  PA_ERR_WORKSPACE = 4,   /* decode workspace missing or too small */
  PA_ERR_CUDA = 5,        /* a CUDA runtime error (launch, attribute, tensor map) */
  PA_ERR_ALIGN = 6        /* a pointer or stride breaks the 16-byte alignment rule */
};

/* Bits OR-ed into *dev_err by the kernels. */
enum pa_dev_error {
  PA_DEV_ERR_BLOCK_ID = 1, /* block table entry outside [0, num_blocks) where a read needs it */
  PA_DEV_ERR_SLOT = 2,     /* slot_mapping entry outside [-1, num_blocks*block_size) */
  PA_DEV_ERR_CONTEXT = 4,  /* context length above max_blocks_per_seq*block_size, or negative */
  PA_DEV_ERR_TIMEOUT = 8,  /* a bounded pipeline wait gave up (the kernel returned early) */
  PA_DEV_ERR_SEQLENS = 16, /* cu_seqlens not non-decreasing, or a sequence shape out of range */
  PA_DEV_ERR_STAGED = 32   /* a staged run outside the tensor, or run offsets that decrease */
};

/* Element types: the sampler's logits (F32 or BF16) and the attention calls' q, caches
 * and outputs (BF16 or F16). */
enum pa_dtype { PA_DTYPE_F32 = 0, PA_DTYPE_BF16 = 1, PA_DTYPE_F16 = 2 };

/* Human-readable name of a pa_status value. Never NULL. */
const char* pa_status_str(int status);

/* Library ABI version, (major << 16) | minor. */
int pa_version(void);

/*
 * pa_store_kvcache — scatter new K/V rows into the paged cache.
 * Source: "nano-vllm解读", section "KVCache的写入" (one Triton kernel writes each
 * token's K/V at its slot); "3.6 ModelRunner…", section 2 (slot formula; slot == -1
 * is a padding row that writes nothing).
 *
 *   k, v            device, 16-bit elements (bf16 or fp16); token i's row starts at
 *                   k + i*k_tok_stride elements and holds num_kv_heads*head_dim
 *                   contiguous elements.
 *   k_tok_stride,
 *   v_tok_stride    token strides in ELEMENTS (>= num_kv_heads*head_dim).
 *   k_cache,v_cache device, the same element type [num_blocks, block_size, num_kv_heads,
 *                   head_dim],
 *                   updated in place: row s of the [num_blocks*block_size,
 *                   num_kv_heads*head_dim] view receives token i when slot_mapping[i]==s.
 *   slot_mapping    device, int32 [num_tokens]; -1 = skip this token.
 *   num_tokens      >= 0 (0 launches nothing and returns PA_OK).
 *
 * The copy is bit-exact for any 16-bit element type (bf16 or fp16). head_dim 64 or 128.
 * Two tokens with the same slot race (the pages never produce that). One warp moves one
 * token's K or V row; 16-byte vectors are used when k, v, both caches and both strides
 * are 16-byte aligned, otherwise 2-byte elements give the same bytes.
 */
int pa_store_kvcache(const void* k, const void* v, int64_t k_tok_stride, int64_t v_tok_stride,
                     void* k_cache, void* v_cache, const int32_t* slot_mapping, int num_tokens,
                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                     int* dev_err, void* stream);

/*
 * pa_staged_write_apply — apply a packed batch of staged runs to a device tensor.
 * Source: "Model Runner V2 设计文档", section "4. StagedWriteTensor" (the tensor stays on
 * the GPU; the host stages the differences, packs them into one contiguous buffer, copies
 * it to the GPU and launches one kernel that applies them; used for block tables and
 * other state written by both host and GPU).
 *
 *   base            device, [num_rows, row_stride] elements of elem_bytes bytes (1, 2, 4
 *                   or 8; int32 for block tables); columns 0..num_cols-1 of each row are
 *                   the tensor.
 *   rows, starts    device, int32 [num_writes]: run w writes row rows[w] from column
 *                   starts[w] on.
 *   offsets         device, int32 [num_writes+1], non-decreasing, offsets[0] = 0,
 *                   offsets[num_writes] = num_values: run w's values are
 *                   values[offsets[w] .. offsets[w+1]).
 *   values          device, [num_values] elements of elem_bytes bytes.
 *
 * Result: base[rows[w]][starts[w] + i] = values[offsets[w] + i] for every run w and
 * i < offsets[w+1] - offsets[w]; nothing else changes. Runs must not overlap
 * (pa_staged_pack merges overlapping writes, later ones winning, before packing); elements
 * that several runs write receive one of their values. A run outside the tensor (row out
 * of range, start < 0, start + length > num_cols) or decreasing offsets set
 * PA_DEV_ERR_STAGED and that run is not written. rows, starts, offsets and values may
 * all point into one packed buffer (each array aligned to its element size).
 */
int pa_staged_write_apply(void* base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
                          int elem_bytes, const int32_t* rows, const int32_t* starts,
                          const int32_t* offsets, const void* values, int num_writes,
                          int64_t num_values, int* dev_err, void* stream);

/*
 * Host-side staging for pa_staged_write_apply (no GPU involved): merges staged writes
 * and packs them into one buffer that a single host-to-device copy moves.
 *
 * pa_staged_pack_bound — bytes that suffice to pack num_writes writes holding num_values
 *   values in total (0 for invalid sizes).
 * pa_staged_pack — write k (host arrays, staging order) puts lens[k] values (taken in
 *   turn from `values`, elem_bytes each) at row rows[k] from column starts[k]. Writes of
 *   one row that overlap or touch become one run; where they overlap the later write
 *   wins. The runs go to `packed` (host memory, pinned for an asynchronous copy) as
 *   int32 rows[W], starts[W], offsets[W+1], then the values at a 16-byte aligned offset;
 *   *layout receives W, the value count, the byte offsets of the four arrays and the
 *   total bytes. If packed_bytes is too small it returns PA_ERR_WORKSPACE with
 *   layout->bytes set to the size needed. Negative lengths or starts: PA_ERR_SHAPE.
 *   Rows and column bounds are checked on the device by pa_staged_write_apply.
 */
typedef struct pa_staged_layout {
  int64_t rows_offset, starts_offset, offsets_offset, values_offset;
  int32_t num_writes;
  int64_t num_values;
  int64_t bytes;
} pa_staged_layout;

size_t pa_staged_pack_bound(int num_writes, int64_t num_values, int elem_bytes);
int pa_staged_pack(const int32_t* rows, const int32_t* starts, const int32_t* lens,
                   const void* values, int num_writes, int elem_bytes, void* packed,
                   size_t packed_bytes, pa_staged_layout* layout);

/*
 * pa_staged_upload_apply — one host-to-device copy of a packed buffer made by
 * pa_staged_pack (layout->bytes bytes from packed_host to packed_dev, asynchronous on
 * `stream`), then pa_staged_write_apply on the copy; base, num_rows, num_cols,
 * row_stride, elem_bytes and dev_err as there. packed_dev is device memory of at least
 * layout->bytes bytes, 16-byte aligned. packed_host should be pinned (page-locked) for
 * the copy to be asynchronous; the caller keeps it unchanged until the copy has ended
 * (an event recorded on `stream` after this call tells when).
 */
int pa_staged_upload_apply(void* base, int64_t num_rows, int64_t num_cols, int64_t row_stride,
                           int elem_bytes, const void* packed_host, void* packed_dev,
                           const pa_staged_layout* layout, int* dev_err, void* stream);

/*
 * pa_sample_workspace_size — bytes of scratch pa_gumbel_sample needs for num_seqs rows
 * (0 for num_seqs < 0).
 *
 * pa_gumbel_sample — one token per row of logits, drawn from softmax(logits / T) by the
 * Gumbel-max trick, without materialising the softmax.
 * Source: "nano-vllm解读", section "Gumbel-Max采样" (argmax_i (ln p_i + G_i),
 * G_i = -ln(-ln u_i), u_i ~ U(0,1) independent, has the law p); "Model Runner V2 设计文档",
 * section 6 "Gumbel 采样内核" (no softmax materialised; stateless in-kernel random numbers
 * from a seed input).
 *
 *   out             device, int64 [num_seqs]: the sampled index of each row.
 *   logits          device, [num_seqs, row_stride] of binary32 (PA_DTYPE_F32) or bf16
 *                   (PA_DTYPE_BF16); columns 0..vocab_size-1 are the logits.
 *   temperatures    device, fp32 [num_seqs]; T <= 0 (or NaN) samples greedily.
 *   seeds, offsets  device, uint64 [num_seqs]: the generator's key and stream position for
 *                   the row (for example a request's seed and its decode step).
 *   workspace       device, >= pa_sample_workspace_size(num_seqs) bytes, 256-byte aligned,
 *                   ZERO before the first call; every call leaves it zero again. Calls
 *                   that overlap in time need different workspaces.
 *
 * Definition (bit-reproducible across calls and launch shapes): element i of row b draws
 * the 32-bit word i % 4 of Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy
 * as 1, 2, 3", SC 2011) at counter (i/4 mod 2^32, i/2^34, offset mod 2^32, offset/2^32)
 * under key (seed mod 2^32, seed/2^32); k = that word >> 9 gives u = (2k + 1) / 2^24. The
 * score is logits[i] / T - ln(-ln u) in fp32 (the logit alone when T <= 0); a NaN score
 * never wins; the largest score wins, the lowest index among equal scores; a row whose
 * scores are all -inf or NaN gives 0.
 */
size_t pa_sample_workspace_size(int num_seqs);
int pa_gumbel_sample(int64_t* out, const void* logits, int64_t row_stride, int logits_dtype,
                     int num_seqs, int vocab_size, const float* temperatures,
                     const uint64_t* seeds, const uint64_t* offsets, void* workspace,
                     size_t workspace_bytes, int* dev_err, void* stream);

/*
 * pa_decode_workspace_size — bytes of scratch that pa_decode needs for num_seqs
 * sequences and num_heads query heads on the CURRENT device (the size depends on its
 * SM count). Returns 0 for invalid sizes.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim);

/*
 * pa_decode — paged GQA decode attention, one query token per sequence.
 * Source: "nano-vllm解读", sections "PageAttention原理" (address = base +
 * block_table[pos / block_size] * block_size + pos % block_size) and
 * "Nano-vllm中的使用" (q [B, H, d]; caches [max_blocks, block_size, H_kv, d];
 * cache_seqlens int32 [B]; block_table int32 [B, max_len_blocks] padded with -1;
 * softmax_scale = 1/sqrt(head_dim)); "3.6 ModelRunner…", section 2 (context_lens =
 * len(seq), i.e. the just-stored token is part of the context).
 *
 *   out             device, [num_seqs, num_heads, head_dim]; written for every row.
 *   q               device, [num_seqs, num_heads, head_dim].
 *   head_dim        64 or 128.
 *   dtype           element type of q, both caches and out: PA_DTYPE_BF16 or PA_DTYPE_F16
 *                   (nano-vllm overview page, section "PagedAttention：KV Cache": a
 *                   block's cache tensor takes head_dim and dtype as parameters).
 *   block_tables    device, int32 [num_seqs, max_blocks_per_seq]; entries at index
 *                   >= ceil(context_lens[b]/block_size) are never read.
 *   context_lens    device, int32 [num_seqs]; 0 writes a zero row and reads nothing.
 *   scale           softmax scale; <= 0 or NaN means 1/sqrt(head_dim).
 *   grid_ctas       number of CTAs that split the key stream (0 = automatic: one per SM,
 *                   but never fewer than four key tiles per CTA, so a short stream is cut
 *                   into fewer segments). The result does not depend on it beyond the
 *                   rounding of the final combine.
 *   workspace       device scratch of at least pa_decode_workspace_size(...) bytes,
 *                   256-byte aligned; zero it once when it is created. It holds the
 *                   partial results, then num_seqs*num_kv_heads int32 arrival counters
 *                   that must be zero before a call; every successful call leaves them
 *                   zero again (after a PA_DEV_ERR_TIMEOUT the caller must zero the
 *                   workspace). The counters' offset depends only on the device and
 *                   num_heads, so a workspace sized for B sequences serves any call
 *                   with num_seqs <= B and the same num_heads / num_kv_heads. Calls that
 *                   overlap in time must use different workspaces.
 *
 * Arithmetic: 16-bit inputs widened exactly, fp32 products, fp32 online softmax and
 * accumulation, one round-to-nearest-even to the element type at the end. Shapes that run
 * on the tensor cores (3 to 8 query heads per KV head, or head_dim 64) also round each
 * probability to the element type before the P V product (the softmax denominator stays
 * fp32): at most 2^-9 relative per probability.
 *
 * Launch: a programmatic dependent launch. The grid may start while the previous kernel
 * on the stream is still running, provided that kernel lets its dependents start early
 * (griddepcontrol.launch_dependents); an ordinary kernel does so only when it completes.
 * Before waiting for that kernel the grid reads context_lens and the block_tables rows of
 * its first tiles (to prefetch those tiles into L2; pa_decode_step also reads
 * slot_mapping); everything else is read and every output written after the wait. So
 * context_lens, block_tables and slot_mapping must not be written by a preceding kernel
 * that releases its dependents before it has written them (host copies and ordinary
 * kernels are fine; of this library's kernels only the decode kernels release early, and
 * they write none of these).
 */
int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int dtype,
              int block_size, int64_t num_blocks, float scale, int grid_ctas, void* workspace,
              size_t workspace_bytes, int* dev_err, void* stream);

/*
 * pa_decode_step — one decode step of the path in ONE launch: the store of every
 * sequence's new token followed by the decode over the cache that includes it.
 * Source: "nano-vllm解读", sections "KVCache的写入" (each layer first writes the new K/V at
 * slot_mapping, then attends) and "CUDAGraph优化" (the decode step is replayed from a
 * captured graph per batch bucket; padding rows carry slot -1 and context length 0);
 * "3.6 ModelRunner…", section 2 (the decode token of sequence b is stored at the slot of
 * its last position, context_lens[b] = len(seq)) and section 5 (graph buckets
 * 1, 2, 4, 8, 16, 32, …, padded with slot -1 / context 0).
 *
 * Same result, bit for bit, as pa_store_kvcache(k_new, v_new, ..., slot_mapping,
 * num_tokens = num_seqs) followed by pa_decode(...) with the other arguments, for every
 * input where each slot_mapping[b] is -1 or the slot of position context_lens[b]-1 of
 * sequence b (block_tables[b][p/bs]*bs + p%bs, p = context_lens[b]-1), which is how the
 * decode step builds it.
 *
 *   k_new, v_new    device, the element type of q (dtype); row b (start k_new +
 *                   b*k_new_stride elements) holds the num_kv_heads*head_dim values of
 *                   sequence b's new token.
 *   k_new_stride,
 *   v_new_stride    token strides in ELEMENTS, >= num_kv_heads*head_dim and multiples of 8
 *                   (k_new, v_new 16-byte aligned), else PA_ERR_ALIGN.
 *   k_cache,v_cache written at the new tokens' slots, read everywhere else.
 *   slot_mapping    device, int32 [num_seqs]. -1: nothing is stored and the cache row at
 *                   position context_lens[b]-1 is read as it is. Any other value that is
 *                   not the slot of that position (or a token of a sequence with context
 *                   length 0) sets PA_DEV_ERR_SLOT and that token is NOT stored (another
 *                   sequence of the same launch might be reading that row).
 *   everything else as pa_decode (head_dim, dtype, the workspace rules; one workspace per
 *   call in flight).
 *
 * The store and the attention share one read of each new row: the CTA that owns a
 * sequence's last key tile copies that row from k_new/v_new into its tile and writes it to
 * the cache. Rows of other sequences that alias the new token's slot (never the case when
 * the slot's block holds the newest position of only one sequence) race with the store.
 * Graph-capturable: no host synchronisation, no allocation, fixed grid for any batch.
 * Launched as a programmatic dependent, with the same rule on context_lens, block_tables
 * and slot_mapping as pa_decode.
 */
int pa_decode_step(void* out, const void* q, const void* k_new, const void* v_new,
                   int64_t k_new_stride, int64_t v_new_stride, void* k_cache, void* v_cache,
                   const int32_t* slot_mapping, const int32_t* block_tables,
                   int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                   int num_heads, int num_kv_heads, int head_dim, int dtype, int block_size,
                   int64_t num_blocks, float scale, int grid_ctas, void* workspace,
                   size_t workspace_bytes, int* dev_err, void* stream);

/*
 * pa_decode_noalloc — pa_decode for callers that cannot allocate device memory.
 * The pages have no counterpart: this is an interface convenience of the library.
 *
 * pa_decode needs a caller-provided workspace. Some callers cannot create one: code
 * running where no device allocator is available or allowed (a plugin inside a host
 * program that owns all device memory, a runtime that forbids allocation after start-up,
 * a caller with a fixed memory budget). This entry point computes exactly what pa_decode
 * computes with the same arguments and dtype PA_DTYPE_BF16, minus workspace/
 * workspace_bytes, and allocates
 * nothing: its scratch is one fixed array of 16 MiB in the library's device memory, held
 * by every GPU that loads the library until the process exits.
 *
 *   Limit           the scratch needed is round256(num_seqs*num_kv_heads*4)
 *                   + round256(G*2*num_heads*4) + round256(G*2*num_heads*128*4) bytes,
 *                   G = grid_ctas (0 = the SM count); more than 16 MiB returns
 *                   PA_ERR_WORKSPACE and launches nothing.
 *   First call      the first call on a device looks up the array's device address
 *                   (cudaGetSymbolAddress, with that device current); make that first
 *                   call before any stream capture. The address is kept per device and
 *                   CUDA context: after the context is destroyed and recreated (for
 *                   example by cudaDeviceReset) the next call looks it up again, so that
 *                   call too should come before any capture.
 *   Sharing         every call on a device uses the same array and it keeps the last
 *                   call's contents; each call clears the arrival counters with an
 *                   asynchronous memset on `stream` before its launch. Calls that overlap
 *                   on the GPU (other streams, or in flight together) race on the array:
 *                   serialise them.
 */
int pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs, int num_heads,
                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                      float scale, int grid_ctas, int* dev_err, void* stream);

/*
 * pa_prefill_varlen — causal (or full) varlen attention of new tokens over the paged
 * cache, on the tcgen05 tensor cores.
 * Source: "nano-vllm解读", section "如何适配不同请求不同序列长度" (q [sum_seq_lens, H, d];
 * cu_seqlens_q / cu_seqlens_k cumulative lengths; max_seqlen_q / max_seqlen_k;
 * causal=True; block_table given when a prefix is cached); "3.6 ModelRunner…",
 * section 2 (new token i of sequence s sits at absolute position
 * num_cached_tokens + i; cu_seqlens_k counts cached plus new tokens).
 *
 *   out             device, [cu_seqlens_q[num_seqs], num_heads, head_dim].
 *   q               device, same shape and element type as out.
 *   head_dim, dtype 64 or 128; PA_DTYPE_BF16 or PA_DTYPE_F16 (q, both caches and out).
 *   k_cache,v_cache device caches of that element type that ALREADY hold every key/value
 *                   row of the call, the new tokens included (run pa_store_kvcache first).
 *   block_tables    device, int32 [num_seqs, max_blocks_per_seq].
 *   cu_seqlens_q    device, int32 [num_seqs+1]; n_s = cu_seqlens_q[s+1]-cu_seqlens_q[s].
 *   cu_seqlens_k    device, int32 [num_seqs+1]; k_s = cu_seqlens_k[s+1]-cu_seqlens_k[s]
 *                   = cached + new tokens, so the cached count is c_s = k_s - n_s >= 0.
 *   max_seqlen_q    host bound on n_s (sizes the grid); sequences above it set
 *                   PA_DEV_ERR_SEQLENS and are left unwritten.
 *   max_seqlen_k    host bound on k_s, used for validation only.
 *   causal          non-zero: query i of sequence s (absolute position c_s + i) sees keys
 *                   t <= c_s + i. Zero: it sees all k_s keys.
 *   scale           softmax scale; <= 0 or NaN means 1/sqrt(head_dim).
 *
 * Requirements: block_size a multiple of 128, or a divisor of 128 that is a multiple of
 * 8; q, out and both caches 16-byte aligned. Arithmetic: 16-bit tensor-core products
 * (kind::f16, both operands of one type) with fp32 accumulation, fp32 softmax, P rounded
 * to the element type for the second product, one rounding of the output.
 */
int pa_prefill_varlen(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
                      int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                      int head_dim, int dtype, int block_size, int64_t num_blocks, int causal,
                      float scale, int* dev_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_PA_H */
