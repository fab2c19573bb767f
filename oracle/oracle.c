/*
 * oracle.c — plain, slow, fp64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path may include, link,
 * load or call this file. Only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it. It shares no code, header, table or helper with the CUDA
 * library: it is written from the definitions on the pages, one loop per definition,
 * with no tiling, fusion or reordering.
 *
 * Definitions followed (page title, section):
 *   - store: "nano-vllm解读", "KVCache的写入": each token's K/V row goes to row
 *     slot_mapping[i] of the cache viewed as [num_blocks*block_size, H_kv*D];
 *     "3.6 ModelRunner、CUDA Graph 与性能基准", section 2: slot == -1 writes nothing.
 *   - address translation: "nano-vllm解读", "PageAttention原理": the key/value of
 *     logical position t lives in physical block block_table[t / block_size] at
 *     offset t % block_size.
 *   - attention: nano-vllm overview page (ascendai.csdn.net), "FlashAttention 集成 /
 *     传统 Attention 的瓶颈": softmax(q k^T / sqrt(d)) v, evaluated here directly over
 *     the gathered keys; the maximum is subtracted before exp, which leaves the
 *     softmax unchanged and keeps exp finite.
 *   - decode context: "3.6 ModelRunner…", section 2: context_lens[b] = len(seq), the
 *     just-stored token included; a row with context length 0 (CUDA-graph padding,
 *     section 5) has no keys and its output is defined here as zeros.
 *   - prefill: "nano-vllm解读", "如何适配不同请求不同序列长度" and "3.6 ModelRunner…",
 *     section 2: new token i of sequence s sits at absolute position c_s + i with
 *     c_s = k_s - n_s cached tokens; causal means keys t <= c_s + i.
 *   - Gumbel-max sampling: "nano-vllm解读", "Gumbel-Max采样": the sample of row b is
 *     argmax_i (ln p_i + G_i), p = softmax(logits / T), G_i = -ln(-ln u_i) with u_i
 *     independent U(0,1); ln p_i differs from logits_i / T by a constant of the row, so
 *     the score used is logits_i / T + G_i. "Model Runner V2 设计文档", section 6
 *     ("Gumbel 采样内核"): the uniforms come from a stateless generator keyed by a seed
 *     input. The generator is Philox4x32-10 as published by Salmon, Moraes, Dror and
 *     Shaw ("Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011); the use of its
 *     counter, the uniform mapping and the greedy / NaN / tie rules are this library's
 *     definitions, restated in gumbel_score below.
 *   - staged writes: "Model Runner V2 设计文档", section "4. StagedWriteTensor": each
 *     staged write copies its values into one row of the tensor from a start column; the
 *     writes take effect one after another, in the order they were staged.
 *
 * bf16 (or IEEE binary16) values arrive as raw uint16 bits; each is widened exactly to
 * double.
 * Parity status: every function here is pinned by the CPU tests (closed forms,
 * invariants, textbook special cases, brute force); see the test suite.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes (oracle-local; independent of the library's codes). */
#define ORC_OK 0
#define ORC_BAD_SLOT 1
#define ORC_BAD_BLOCK 2
#define ORC_BAD_CONTEXT 3
#define ORC_BAD_SHAPE 4
#define ORC_BAD_SEQLENS 5

/* Exact widening of a bf16 bit pattern to double: bf16 is the top half of an fp32. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Exact widening of an IEEE 754 binary16 bit pattern to double: sign, 5-bit exponent
 * (bias 15), 10-bit fraction; exponent 0 holds the subnormals m * 2^-24, exponent 31 the
 * infinities and NaNs. */
static double f16_bits_to_double(uint16_t bits) {
  const int sign = bits >> 15, e = (bits >> 10) & 31, m = bits & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(1024 + m), e - 25);
  return sign ? -v : v;
}

/* The element types of q, k and v: bf16 (is_fp16 = 0) or IEEE binary16 (is_fp16 = 1). */
static double elem_to_double(uint16_t bits, int is_fp16) {
  return is_fp16 ? f16_bits_to_double(bits) : bf16_bits_to_double(bits);
}

double oracle_f16_to_double(uint16_t bits) { return f16_bits_to_double(bits); }

int oracle_version(void) { return 1; }

/*
 * Store: for every token i whose slot is not -1, copy its H_kv*D element row of k
 * (resp. v) into row slot of the flattened cache. Byte copy, so the result is exact.
 */
int oracle_store_kvcache(const uint16_t* k, const uint16_t* v, int64_t k_tok_stride,
                         int64_t v_tok_stride, uint16_t* k_cache, uint16_t* v_cache,
                         const int32_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                         int head_dim, int64_t num_slots) {
  int64_t row = (int64_t)num_kv_heads * head_dim;
  int status = ORC_OK;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      status = ORC_BAD_SLOT;
      continue;
    }
    for (int64_t e = 0; e < row; ++e) {
      k_cache[slot * row + e] = k[i * k_tok_stride + e];
      v_cache[slot * row + e] = v[i * v_tok_stride + e];
    }
  }
  return status;
}

/*
 * Physical cache row of logical position t of a sequence whose block-table row is
 * `table` (max_blocks entries): block_table[t / block_size] * block_size + t % block_size.
 * Returns -1 when the table entry is missing or out of range.
 */
static int64_t physical_row(const int32_t* table, int max_blocks, int64_t t, int block_size,
                            int64_t num_blocks) {
  int64_t logical_block = t / block_size;
  if (logical_block >= max_blocks) return -1;
  int64_t phys = table[logical_block];
  if (phys < 0 || phys >= num_blocks) return -1;
  return phys * block_size + t % block_size;
}

/*
 * One attention row: the query vector qv (D doubles) against keys at logical positions
 * 0..num_keys-1 of one sequence and one KV head. Writes D doubles to o and, if lse is
 * non-NULL, the natural log of sum_t exp(scale*q.k_t) to *lse.
 * Steps, in the definition's order: scores s_t = scale * q.k_t; softmax over t; o = sum_t p_t v_t.
 */
static int attend_row(double* o, double* lse, const double* qv, const uint16_t* k_cache,
                      const uint16_t* v_cache, const int32_t* table, int max_blocks,
                      int64_t num_keys, int num_kv_heads, int kv_head, int D, int block_size,
                      int64_t num_blocks, double scale, double* scores /* num_keys scratch */,
                      int is_fp16) {
  int64_t row_elems = (int64_t)num_kv_heads * D;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (num_keys <= 0) {
    if (lse) *lse = -INFINITY;
    return ORC_OK;
  }
  /* scores */
  for (int64_t t = 0; t < num_keys; ++t) {
    int64_t r = physical_row(table, max_blocks, t, block_size, num_blocks);
    if (r < 0) return ORC_BAD_BLOCK;
    const uint16_t* kt = k_cache + r * row_elems + (int64_t)kv_head * D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qv[d] * elem_to_double(kt[d], is_fp16);
    scores[t] = scale * dot;
  }
  /* softmax */
  double m = scores[0];
  for (int64_t t = 1; t < num_keys; ++t)
    if (scores[t] > m) m = scores[t];
  double l = 0.0;
  for (int64_t t = 0; t < num_keys; ++t) {
    scores[t] = exp(scores[t] - m);
    l += scores[t];
  }
  /* weighted sum of values */
  for (int64_t t = 0; t < num_keys; ++t) {
    int64_t r = physical_row(table, max_blocks, t, block_size, num_blocks);
    const uint16_t* vt = v_cache + r * row_elems + (int64_t)kv_head * D;
    double p = scores[t] / l;
    for (int d = 0; d < D; ++d) o[d] += p * elem_to_double(vt[d], is_fp16);
  }
  if (lse) *lse = m + log(l);
  return ORC_OK;
}

/* nthreads > 0: that many threads; 0: every host core (so a one-thread call before does
 * not leave later calls on one thread). */
static int set_threads(int nthreads) {
#ifdef _OPENMP
  omp_set_num_threads(nthreads > 0 ? nthreads : omp_get_num_procs());
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

int oracle_max_threads(int nthreads) { return set_threads(nthreads); }

/*
 * Decode: for every sequence b and query head h, attend over logical positions
 * 0..context_lens[b]-1 of KV head h / (H / H_kv). out is [B, H, D] doubles; lse (nullable)
 * is [B, H] (natural log). When `pairs` (b*H + h indices) is non-NULL only those rows are
 * computed and out/lse are compact: [num_pairs, D] and [num_pairs].
 */
int oracle_decode(double* out, double* lse, const uint16_t* q, const uint16_t* k_cache,
                  const uint16_t* v_cache, const int32_t* block_tables, int max_blocks,
                  const int32_t* context_lens, int B, int H, int Hk, int D, int block_size,
                  int64_t num_blocks, double scale, const int64_t* pairs, int64_t num_pairs,
                  int nthreads, int is_fp16) {
  if (B < 0 || H <= 0 || Hk <= 0 || H % Hk != 0 || D <= 0 || block_size <= 0)
    return ORC_BAD_SHAPE;
  int group = H / Hk;
  int64_t max_ctx = 0;
  for (int b = 0; b < B; ++b) {
    if (context_lens[b] < 0 || (int64_t)context_lens[b] > (int64_t)max_blocks * block_size)
      return ORC_BAD_CONTEXT;
    if (context_lens[b] > max_ctx) max_ctx = context_lens[b];
  }
  int64_t n = pairs ? num_pairs : (int64_t)B * H;
  int status = ORC_OK;
  set_threads(nthreads);
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
    for (int64_t idx = 0; idx < n; ++idx) {
      int64_t bh = pairs ? pairs[idx] : idx;
      int b = (int)(bh / H), h = (int)(bh % H);
      for (int d = 0; d < D; ++d)
        qv[d] = elem_to_double(q[((int64_t)b * H + h) * D + d], is_fp16);
      double row_lse;
      int64_t dst = pairs ? idx : bh; /* compact output when a subset is asked for */
      int rc = attend_row(out + dst * D, &row_lse, qv, k_cache, v_cache,
                          block_tables + (int64_t)b * max_blocks, max_blocks, context_lens[b],
                          Hk, h / group, D, block_size, num_blocks, scale, scores, is_fp16);
      if (lse) lse[dst] = row_lse;
      if (rc != ORC_OK) {
#pragma omp critical
        status = rc;
      }
    }
    free(scores);
    free(qv);
  }
  return status;
}

/*
 * Prefill: q and out are [cu_q[S], H, D]. For sequence s, new token i (0 <= i < n_s) is
 * at absolute position p = c_s + i, c_s = k_s - n_s. Causal: keys 0..p; otherwise keys
 * 0..k_s-1. When `rows` (token_row * H + h indices) is non-NULL only those rows are
 * computed and out/lse are compact: [num_rows, D] and [num_rows].
 */
int oracle_prefill(double* out, double* lse, const uint16_t* q, const uint16_t* k_cache,
                   const uint16_t* v_cache, const int32_t* block_tables, int max_blocks,
                   const int32_t* cu_q, const int32_t* cu_k, int S, int H, int Hk, int D,
                   int block_size, int64_t num_blocks, int causal, double scale,
                   const int64_t* rows, int64_t num_rows, int nthreads, int is_fp16) {
  if (S < 0 || H <= 0 || Hk <= 0 || H % Hk != 0 || D <= 0 || block_size <= 0)
    return ORC_BAD_SHAPE;
  int group = H / Hk;
  int64_t total_q = cu_q[S];
  int64_t max_k = 0;
  for (int s = 0; s < S; ++s) {
    int64_t n_s = (int64_t)cu_q[s + 1] - cu_q[s];
    int64_t k_s = (int64_t)cu_k[s + 1] - cu_k[s];
    if (n_s < 0 || k_s < n_s) return ORC_BAD_SEQLENS;
    if (k_s > (int64_t)max_blocks * block_size) return ORC_BAD_CONTEXT;
    if (k_s > max_k) max_k = k_s;
  }
  int64_t n = rows ? num_rows : total_q * H;
  int status = ORC_OK;
  set_threads(nthreads);
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(max_k > 0 ? max_k : 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
    for (int64_t idx = 0; idx < n; ++idx) {
      int64_t th = rows ? rows[idx] : idx;
      int64_t tok = th / H;
      int h = (int)(th % H);
      /* the sequence holding query row tok: cu_q[s] <= tok < cu_q[s+1] */
      int s = 0;
      while (s < S && !(tok >= cu_q[s] && tok < cu_q[s + 1])) ++s;
      if (s == S) {
#pragma omp critical
        status = ORC_BAD_SEQLENS;
        continue;
      }
      int64_t n_s = (int64_t)cu_q[s + 1] - cu_q[s];
      int64_t k_s = (int64_t)cu_k[s + 1] - cu_k[s];
      int64_t c_s = k_s - n_s;
      int64_t i = tok - cu_q[s];
      int64_t num_keys = causal ? (c_s + i + 1) : k_s;
      for (int d = 0; d < D; ++d) qv[d] = elem_to_double(q[(tok * H + h) * D + d], is_fp16);
      double row_lse;
      int64_t dst = rows ? idx : th; /* compact output when a subset is asked for */
      int rc = attend_row(out + dst * D, &row_lse, qv, k_cache, v_cache,
                          block_tables + (int64_t)s * max_blocks, max_blocks, num_keys, Hk,
                          h / group, D, block_size, num_blocks, scale, scores, is_fp16);
      if (lse) lse[dst] = row_lse;
      if (rc != ORC_OK) {
#pragma omp critical
        status = rc;
      }
    }
    free(scores);
    free(qv);
  }
  return status;
}

/* Slot of logical position pos of a sequence (host-side prepare step of section 2 of
 * "3.6 ModelRunner…"): block_table[pos / block_size] * block_size + pos % block_size.
 * Used by the tests to check the workload generator's slot_mapping. */
int64_t oracle_slot_of(const int32_t* table, int max_blocks, int64_t pos, int block_size) {
  int64_t logical_block = pos / block_size;
  if (pos < 0 || logical_block >= max_blocks || table[logical_block] < 0) return -1;
  return (int64_t)table[logical_block] * block_size + pos % block_size;
}

/*
 * Staged writes applied in staging order to a row-major [rows, cols] tensor of
 * elem_bytes-byte elements. Write w puts w_len[w] values (taken in turn from `values`)
 * at row w_row[w], columns w_start[w] .. w_start[w]+w_len[w]-1. A write that leaves the
 * tensor is an invalid input (ORC_BAD_SHAPE), nothing after it is applied.
 */
int oracle_staged_apply(unsigned char* base, int64_t rows, int64_t cols, int elem_bytes,
                        int nwrites, const int64_t* w_row, const int64_t* w_start,
                        const int64_t* w_len, const unsigned char* values) {
  int64_t taken = 0;
  for (int w = 0; w < nwrites; ++w) {
    if (w_row[w] < 0 || w_row[w] >= rows || w_start[w] < 0 || w_len[w] < 0 ||
        w_start[w] + w_len[w] > cols)
      return ORC_BAD_SHAPE;
    memcpy(base + (w_row[w] * cols + w_start[w]) * elem_bytes, values + taken * elem_bytes,
           (size_t)(w_len[w] * elem_bytes));
    taken += w_len[w];
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------- Philox4x32-10 */
/* One Philox4x32 round: two 32x32->64 products of counter words 0 and 2 by the round
 * multipliers; the new counter is (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1,
 * lo(M0*c0)). Ten rounds, the key advanced by the Weyl constants between rounds. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint64_t p0 = (uint64_t)M0 * c0;
    const uint64_t p1 = (uint64_t)M1 * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n1 = (uint32_t)p1;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    const uint32_t n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32 random bits of element i of a row with this seed and offset: word i % 4 of
 * Philox4x32-10 at counter (i/4 low 32 bits, i/4 high 32 bits, offset low, offset high),
 * key (seed low, seed high). */
uint32_t oracle_philox_bits(uint64_t seed, uint64_t offset, uint64_t i) {
  const uint64_t g = i >> 2;
  const uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), (uint32_t)offset,
                           (uint32_t)(offset >> 32)};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return out[i & 3];
}

/* Uniform in (0, 1) from 32 random bits: the top 23 bits k give u = (2k + 1) / 2^24, the
 * midpoints of 2^23 equal cells (exactly representable in binary32, never 0 or 1). */
double oracle_uniform(uint32_t bits) {
  return (double)(2u * (bits >> 9) + 1u) / 16777216.0;
}

/* Score of element i: logits/T + G with G = -ln(-ln u); T <= 0 (greedy) gives the logit
 * alone. A NaN logit scores -inf. */
static double gumbel_score(double logit, double temperature, uint64_t seed, uint64_t offset,
                           uint64_t i) {
  if (isnan(logit)) return -INFINITY;
  if (!(temperature > 0.0)) return logit;
  const double u = oracle_uniform(oracle_philox_bits(seed, offset, i));
  return logit / temperature - log(-log(u));
}

/* Gumbel-max sample of every row: the index of the largest score, the lowest index among
 * equal scores (a row of -inf scores gives 0). logits: row-major with row_stride elements
 * between rows, binary32 (is_bf16 = 0) or bf16 bits (is_bf16 = 1). Writes the index, the
 * largest score and the second largest (gap to the runner-up) per row. */
int oracle_gumbel_sample(int64_t* out, double* best, double* second, const void* logits,
                         int64_t row_stride, int is_bf16, int num_rows, int64_t vocab,
                         const float* temperatures, const uint64_t* seeds,
                         const uint64_t* offsets, int nthreads) {
  if (num_rows < 0 || vocab <= 0 || row_stride < vocab) return ORC_BAD_SHAPE;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < num_rows; ++b) {
    double m1 = -INFINITY, m2 = -INFINITY;
    int64_t arg = 0;
    for (int64_t i = 0; i < vocab; ++i) {
      double l;
      if (is_bf16) {
        l = bf16_bits_to_double(((const uint16_t*)logits)[(int64_t)b * row_stride + i]);
      } else {
        l = (double)((const float*)logits)[(int64_t)b * row_stride + i];
      }
      const double x = gumbel_score(l, (double)temperatures[b], seeds[b], offsets[b], i);
      if (x > m1) {
        m2 = m1;
        m1 = x;
        arg = i;
      } else if (x > m2) {
        m2 = x;
      }
    }
    out[b] = arg;
    if (best) best[b] = m1;
    if (second) second[b] = m2;
  }
  return ORC_OK;
}

/* Every score of one row (for tests that check a choice among near-equal scores). */
int oracle_gumbel_scores(double* scores, const void* logits, int is_bf16, int64_t vocab,
                         float temperature, uint64_t seed, uint64_t offset) {
  for (int64_t i = 0; i < vocab; ++i) {
    const double l = is_bf16 ? bf16_bits_to_double(((const uint16_t*)logits)[i])
                             : (double)((const float*)logits)[i];
    scores[i] = gumbel_score(l, (double)temperature, seed, offset, i);
  }
  return ORC_OK;
}
