/*
 * oracle.c -- plain, slow, obviously correct CPU reference for the hot path of one
 * continuous-batching iteration: paged decode/verify attention and speculative
 * rejection sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls
 * this file; only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or constant with the CUDA path.
 *
 * Precision: every quantity is computed in IEEE double from the exact input values
 * (fp32 inputs widened, bf16 inputs decoded bit-exactly, fp64 inputs as given).
 *
 * Sources (the pages this follows):
 *  - "Continuous Batching and Speculative Decoding: How Modern LLM Serving Engines
 *    Actually Work" (syslabs.in), sections "PagedAttention: making the KV cache
 *    schedulable" and "Speculative decoding" / "The core idea".
 *  - "llm-inference-optimization-batching" (tempatgunting.com), section "Anatomy of
 *    the KV Cache: Memory Layout, Paging and Quantization Trade-offs" (pool shape
 *    [num_blocks, block_size, num_heads, head_dim], block table per sequence) and
 *    section "Speculative Decoding: Turning Verification Parallelism into Latency
 *    Wins" (accept/resample/bonus, rollback).
 *  - "Continuous Batching & Speculative Decoding" (neuralmasteryai.com), section
 *    "3. Mathematical Proof: Exact Distributional Match" / "The Modified Rejection
 *    Sampling Algorithm" (accept iff r <= min(1, p/q); halt at the first rejection;
 *    resample from max(0, p - q) normalised).
 *  - Philox4x32-10: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
 *    Random Numbers: As Easy as 1, 2, 3", SC'11 (the published counter-based
 *    generator; the pages only say "random()").
 *
 * Readings where the pages are silent (the plainest one the rest supports):
 *  - seq_lens[i] counts every KV token of sequence i, including this step's query
 *    tokens; query token j of sequence i sits at absolute position L_i - ql_i + j and
 *    attends to positions 0..that position (causal inside the draft window).
 *  - query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups).
 *  - lse is the natural log of sum_t exp(scale * q.k_t).
 *  - acceptance uses "<=" (the neuralmasteryai page), evaluated as r*q <= p in double.
 *  - uniforms: u = (word + 0.5) * 2^-32 from Philox4x32-10 with
 *    counter = (position, sequence, 0, 0) and key = (seed low word, seed high word);
 *    word 0 drives the ratio test at that position, word 1 the resample / bonus draw.
 *  - inverse-CDF draw: emit the smallest x whose inclusive prefix sum exceeds s * S.
 *  - a rejection whose residual sums to zero (impossible in exact arithmetic) falls
 *    back to sampling from the target row p_j.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 2

#define ORC_OK 0
#define ORC_E_ARG (-1)
#define ORC_E_PAGE (-2)
#define ORC_E_LEN (-3)
#define ORC_E_TOKEN (-4)
#define ORC_E_DIST (-5)

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the parallel loops use from now on (timing a single-thread baseline); n < 1
 * leaves the setting as it is. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Element `idx` of an array of the given storage type, widened to double.
 * bf16 is the top half of an fp32 bit pattern, so the decode is exact. */
static double load_elem(const void* base, int dtype, size_t idx) {
  if (dtype == ORC_F32) return (double)((const float*)base)[idx];
  if (dtype == ORC_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return ((const double*)base)[idx];
}

/* ------------------------------------------------------------------------------
 * Paged attention, plain definition.
 *
 * Pool layout (tempatgunting.com, "Anatomy of the KV Cache"): k_pages and v_pages
 * are [num_pages, page_size, num_kv_heads, head_dim]; block_table is
 * [num_seqs, max_pages_per_seq]; logical position t of sequence i lives in physical
 * page block_table[i][t / page_size], slot t % page_size (syslabs.in,
 * "PagedAttention": a per-sequence table maps logical positions to blocks).
 *
 * q and out are [total_q_tokens, num_q_heads, head_dim], rows packed by sequence in
 * order; lse is [total_q_tokens, num_q_heads].  For every query row:
 *     s_t   = scale * <q, k_t>          for the visible positions t
 *     lse   = log sum_t exp(s_t)
 *     out   = sum_t exp(s_t - lse) v_t
 * Query token j of a sequence with context L and ql query tokens sits at position
 * L - ql + j.  Without a tree it sees positions 0 .. L - ql + j (causal within the
 * draft window).  With a draft tree (neuralmasteryai.com, "Tree Attention & Medusa
 * Heads": candidate paths verified in one pass), parents[row] is the index of the
 * token's parent among its sequence's query tokens (-1: the root, attached to the
 * context), and the token sees the context 0 .. L - ql - 1 and the positions of
 * its ancestors and itself.  A parent must come before its child.
 * Returns ORC_OK, or a negative code for arguments that make the result undefined.
 * ---------------------------------------------------------------------------- */
static int paged_attn_impl(const void* q, const void* k_pages, const void* v_pages, int dtype,
                           const int32_t* block_table, const int32_t* seq_lens,
                           const int32_t* query_lens, const int32_t* parents, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                           int num_pages, int max_pages_per_seq, double scale, double* out,
                           double* lse) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      page_size <= 0 || num_pages < 0 || max_pages_per_seq < 0)
    return ORC_E_ARG;
  if (num_q_heads % num_kv_heads != 0) return ORC_E_ARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16 && dtype != ORC_F64) return ORC_E_ARG;

  /* First query row of every sequence: exclusive prefix sum of query_lens. */
  int64_t* row0 = (int64_t*)malloc(sizeof(int64_t) * (size_t)(num_seqs + 1));
  if (!row0) return ORC_E_ARG;
  row0[0] = 0;
  for (int i = 0; i < num_seqs; ++i) {
    int L = seq_lens[i], ql = query_lens[i];
    if (ql < 0 || L < 0 || ql > L || (int64_t)L > (int64_t)max_pages_per_seq * page_size) {
      free(row0);
      return ORC_E_LEN;
    }
    int npages = (L + page_size - 1) / page_size;
    for (int pg = 0; pg < npages; ++pg) {
      int32_t id = block_table[(size_t)i * max_pages_per_seq + pg];
      if (id < 0 || id >= num_pages) {
        free(row0);
        return ORC_E_PAGE;
      }
    }
    row0[i + 1] = row0[i] + ql;
  }
  if (parents) {
    for (int i = 0; i < num_seqs; ++i)
      for (int j = 0; j < query_lens[i]; ++j) {
        const int32_t pj = parents[row0[i] + j];
        if (pj < -1 || pj >= j) {
          free(row0);
          return ORC_E_ARG;
        }
      }
  }

  const int group = num_q_heads / num_kv_heads;
  const int64_t work = (int64_t)num_seqs * num_q_heads;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t w = 0; w < work; ++w) {
    const int i = (int)(w / num_q_heads);
    const int h = (int)(w % num_q_heads);
    const int g = h / group; /* KV head read by query head h */
    const int L = seq_lens[i];
    const int ql = query_lens[i];
    if (ql == 0) continue;
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    char* vis = (char*)malloc((size_t)L + 1);
    for (int j = 0; j < ql; ++j) {
      const int pos = L - ql + j; /* absolute position of this query token */
      const int64_t row = row0[i] + j;
      const size_t qbase = ((size_t)row * num_q_heads + h) * head_dim;
      /* visible positions */
      for (int t = 0; t <= pos; ++t) vis[t] = !parents || t < L - ql;
      if (parents)
        for (int a = j; a >= 0; a = parents[row0[i] + a]) vis[L - ql + a] = 1;
      double m = -INFINITY;
      for (int t = 0; t <= pos; ++t) {
        if (!vis[t]) continue;
        const int32_t page = block_table[(size_t)i * max_pages_per_seq + t / page_size];
        const int slot = t % page_size;
        const size_t kbase =
            (((size_t)page * page_size + slot) * num_kv_heads + g) * head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
          dot += load_elem(q, dtype, qbase + d) * load_elem(k_pages, dtype, kbase + d);
        s[t] = scale * dot;
        if (s[t] > m) m = s[t];
      }
      double sum = 0.0;
      for (int t = 0; t <= pos; ++t)
        if (vis[t]) sum += exp(s[t] - m);
      const double row_lse = m + log(sum);
      lse[(size_t)row * num_q_heads + h] = row_lse;
      double* o = out + qbase;
      for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
      for (int t = 0; t <= pos; ++t) {
        if (!vis[t]) continue;
        const double wt = exp(s[t] - row_lse);
        const int32_t page = block_table[(size_t)i * max_pages_per_seq + t / page_size];
        const int slot = t % page_size;
        const size_t vbase =
            (((size_t)page * page_size + slot) * num_kv_heads + g) * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] += wt * load_elem(v_pages, dtype, vbase + d);
      }
    }
    free(vis);
    free(s);
  }
  free(row0);
  return ORC_OK;
}

int oracle_paged_attn(const void* q, const void* k_pages, const void* v_pages, int dtype,
                      const int32_t* block_table, const int32_t* seq_lens,
                      const int32_t* query_lens, int num_seqs, int num_q_heads,
                      int num_kv_heads, int head_dim, int page_size, int num_pages,
                      int max_pages_per_seq, double scale, double* out, double* lse) {
  return paged_attn_impl(q, k_pages, v_pages, dtype, block_table, seq_lens, query_lens, NULL,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                         max_pages_per_seq, scale, out, lse);
}

/* The same with a draft tree: parents[total_q_tokens] as described above. */
int oracle_paged_attn_tree(const void* q, const void* k_pages, const void* v_pages, int dtype,
                           const int32_t* block_table, const int32_t* seq_lens,
                           const int32_t* query_lens, const int32_t* parents, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                           int num_pages, int max_pages_per_seq, double scale, double* out,
                           double* lse) {
  if (!parents) return ORC_E_ARG;
  return paged_attn_impl(q, k_pages, v_pages, dtype, block_table, seq_lens, query_lens, parents,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                         max_pages_per_seq, scale, out, lse);
}

/* ------------------------------------------------------------------------------
 * Quantised KV pages ("llm-inference-optimization-batching", tempatgunting.com,
 * section "Quantization and Precision Choices for KV": INT8 or FP8 KV with per-head
 * or per-token scaling factors, separate scales for K and V, dequantised inside the
 * attention).  Reading: one scale per (page, KV head, slot), i.e. per token and head,
 * symmetric (no zero point); value = scale * decode(code).
 *
 * codes  [num_pages, page_size, num_kv_heads, head_dim] bytes (the pool layout);
 * scales [num_pages, num_kv_heads, page_size] fp32;
 * out    [num_pages, page_size, num_kv_heads, head_dim] double.
 * fmt ORC_Q_E4M3: OCP FP8 E4M3 ("fn": no infinities) -- sign bit, 4 exponent bits with
 *   bias 7, 3 mantissa bits; exponent 0 is subnormal (m * 2^-9); the pattern with all
 *   exponent and mantissa bits set is NaN; largest finite 448.
 * fmt ORC_Q_INT8: the byte as a two's-complement integer.
 * The decoded pool then goes through the float64 attention above unchanged.
 * ---------------------------------------------------------------------------- */
#define ORC_Q_E4M3 0
#define ORC_Q_INT8 1

static double decode_e4m3(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

int oracle_dequant_kv(const uint8_t* codes, const float* scales, int fmt, int64_t num_pages,
                      int page_size, int num_kv_heads, int head_dim, double* out) {
  if (num_pages < 0 || page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return ORC_E_ARG;
  if (fmt != ORC_Q_E4M3 && fmt != ORC_Q_INT8) return ORC_E_ARG;
  for (int64_t pg = 0; pg < num_pages; ++pg)
    for (int t = 0; t < page_size; ++t)
      for (int h = 0; h < num_kv_heads; ++h) {
        const double sc = (double)scales[((size_t)pg * num_kv_heads + h) * page_size + t];
        const size_t base = (((size_t)pg * page_size + t) * num_kv_heads + h) * head_dim;
        for (int d = 0; d < head_dim; ++d) {
          const uint8_t c = codes[base + d];
          const double x = fmt == ORC_Q_E4M3 ? decode_e4m3(c) : (double)(int8_t)c;
          out[base + d] = sc * x;
        }
      }
  return ORC_OK;
}

/* ------------------------------------------------------------------------------
 * Philox4x32-10 (Salmon et al., SC'11): ten rounds of the 4x32 Philox S-box on a
 * 128-bit counter under a 64-bit key, the key advanced by the two Weyl constants
 * between rounds.
 * ---------------------------------------------------------------------------- */
static void philox_sbox(uint32_t c[4], const uint32_t k[2]) {
  const uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
  const uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
  const uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
  const uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
  const uint32_t n0 = hi1 ^ c[1] ^ k[0];
  const uint32_t n2 = hi0 ^ c[3] ^ k[1];
  c[0] = n0;
  c[1] = lo1;
  c[2] = n2;
  c[3] = lo0;
}

void oracle_philox4x32_10(const uint32_t counter[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c[4] = {counter[0], counter[1], counter[2], counter[3]};
  uint32_t k[2] = {key[0], key[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += 0x9E3779B9u;
      k[1] += 0xBB67AE85u;
    }
    philox_sbox(c, k);
  }
  out[0] = c[0];
  out[1] = c[1];
  out[2] = c[2];
  out[3] = c[3];
}

/* Batched Philox for tests: out[n][4] for counters ctr[n][4] under one key. */
void oracle_philox4x32_10_many(const uint32_t* ctr, int64_t n, const uint32_t key[2],
                               uint32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) oracle_philox4x32_10(ctr + 4 * i, key, out + 4 * i);
}

/* The uniforms the method consumes.  r[b][i] (ratio test at position i) and
 * s[b][j] (resample or bonus draw at position j) for j = 0..k, all in (0, 1):
 * (word + 0.5) * 2^-32 of Philox4x32-10 at counter (position, b, 0, 0). */
void oracle_uniforms(uint64_t seed, int B, int k, double* r, double* s) {
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  for (int b = 0; b < B; ++b) {
    for (int pos = 0; pos <= k; ++pos) {
      const uint32_t ctr[4] = {(uint32_t)pos, (uint32_t)b, 0u, 0u};
      uint32_t w[4];
      oracle_philox4x32_10(ctr, key, w);
      if (pos < k) r[(size_t)b * k + pos] = ((double)w[0] + 0.5) * 0x1p-32;
      s[(size_t)b * (k + 1) + pos] = ((double)w[1] + 0.5) * 0x1p-32;
    }
  }
}

/* ------------------------------------------------------------------------------
 * Modified rejection sampling with the uniforms given explicitly.
 *
 * p: [B, k+1, V] target probabilities (row i scores position i; row k is the bonus
 *    row); q: [B, k, V] draft probabilities; draft: [B, k] proposed tokens.
 * r: [B, k] and s: [B, k+1] uniforms in (0, 1).
 *
 * For each sequence, following the neuralmasteryai page's four steps and the
 * syslabs.in loop:
 *   for i = 0 .. k-1: accept x_i iff r_i <= min(1, p_i(x_i) / q_i(x_i)), tested as
 *                     r_i * q_i(x_i) <= p_i(x_i); stop at the first rejection j.
 *   if a rejection happened at j: draw from max(0, p_j - q_j) / sum (residual);
 *   otherwise (j = k):            draw the bonus token from p_k.
 *   The draw emits the smallest x with sum_{y<=x} w(y) > s_j * sum_y w(y).
 * Outputs: accepted_len[b] = j; out_tokens[b] = x_0..x_{j-1}, drawn, then -1.
 *
 * margin[b] (optional) is the smallest distance, in uniform space, between a
 * uniform that decided this sequence's outcome and the threshold it was compared
 * with; flag_pos[b] (optional) is the first position whose decision lay within
 * `flag_window` of its threshold, or -1.
 * fallback[b] (optional) is 1 when a zero residual forced the draw from p_j.
 * Returns ORC_OK, ORC_E_TOKEN for a draft outside [0, V), ORC_E_DIST when the row
 * to draw from has no positive weight (that sequence then emits -1 at position j).
 * ---------------------------------------------------------------------------- */
/* One sequence of the rule above; w is a scratch row of V doubles. */
static int verify_one(const float* pb, const float* qb, const int32_t* xb, const double* rb,
                      const double* sb, int k, int V, double flag_window, double* w,
                      int32_t* acc_out, int32_t* ob, double* margin_out, int32_t* flag_out,
                      int32_t* fallback_out) {
  for (int t = 0; t <= k; ++t) ob[t] = -1;
  double mg = INFINITY;
  int first_flag = -1;
  int used_fallback = 0;
  for (int i = 0; i < k; ++i) {
    if (xb[i] < 0 || xb[i] >= V) {
      *acc_out = -1;
      *margin_out = 0.0;
      *flag_out = -1;
      *fallback_out = 0;
      return ORC_E_TOKEN;
    }
  }

  /* 1. Ratio tests, left to right, halting at the first rejection. */
  int j = k;
  for (int i = 0; i < k; ++i) {
    const int x = xb[i];
    const double pi = (double)pb[(size_t)i * V + x];
    const double qi = (double)qb[(size_t)i * V + x];
    const double ri = rb[i];
    if (qi > 0.0) {
      const double d = fabs(ri - pi / qi);
      if (d < mg) mg = d;
      if (d < flag_window && first_flag < 0) first_flag = i;
    }
    if (ri * qi <= pi) {
      ob[i] = x; /* accepted */
    } else {
      j = i; /* rejected: halt */
      break;
    }
  }

  /* 2. The row to draw from: residual max(0, p_j - q_j) or the bonus row p_k. */
  double S = 0.0;
  for (int x = 0; x < V; ++x) {
    if (j < k) {
      const double diff = (double)pb[(size_t)j * V + x] - (double)qb[(size_t)j * V + x];
      w[x] = diff > 0.0 ? diff : 0.0;
    } else {
      w[x] = (double)pb[(size_t)k * V + x];
    }
    S += w[x];
  }
  if (S == 0.0 && j < k) {
    /* Zero residual after a rejection: draw from p_j instead. */
    used_fallback = 1;
    for (int x = 0; x < V; ++x) {
      w[x] = (double)pb[(size_t)j * V + x];
      S += w[x];
    }
  }

  /* 3. Inverse-CDF draw: smallest x with prefix(x) > s_j * S. */
  int status = ORC_OK;
  const double sj = sb[j];
  const double target = sj * S;
  int drawn = -1;
  if (S > 0.0) {
    double c = 0.0;
    for (int x = 0; x < V; ++x) {
      const double before = c;
      c += w[x];
      if (w[x] > 0.0 && c > target) {
        drawn = x;
        const double d = fmin(sj - before / S, c / S - sj);
        if (d < mg) mg = d;
        if (d < flag_window && first_flag < 0) first_flag = j;
        break;
      }
    }
    if (drawn < 0) {
      /* Rounding left the target at or beyond the total: last token with mass. */
      for (int x = V - 1; x >= 0; --x)
        if (w[x] > 0.0) {
          drawn = x;
          break;
        }
      mg = 0.0;
      if (first_flag < 0) first_flag = j;
    }
  } else {
    status = ORC_E_DIST;
  }
  ob[j] = drawn;
  *acc_out = j;
  *margin_out = mg;
  *flag_out = first_flag;
  *fallback_out = used_fallback;
  return status;
}

int oracle_spec_verify_given_uniforms(const float* p, const float* q, const int32_t* draft,
                                      const double* r, const double* s, int B, int k, int V,
                                      double flag_window, int32_t* accepted_len,
                                      int32_t* out_tokens, double* margin, int32_t* flag_pos,
                                      int32_t* fallback) {
  if (B < 0 || k < 0 || V <= 0) return ORC_E_ARG;
  int worst = ORC_OK;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    int local = w ? ORC_OK : ORC_E_ARG;
#pragma omp for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
      if (!w) continue;
      double mg;
      int32_t fp, fb;
      const int rc = verify_one(p + (size_t)b * (k + 1) * V, q + (size_t)b * k * V,
                                draft + (size_t)b * k, r + (size_t)b * k,
                                s + (size_t)b * (k + 1), k, V, flag_window, w,
                                accepted_len + b, out_tokens + (size_t)b * (k + 1), &mg, &fp,
                                &fb);
      if (margin) margin[b] = mg;
      if (flag_pos) flag_pos[b] = fp;
      if (fallback) fallback[b] = fb;
      if (rc != ORC_OK && local == ORC_OK) local = rc;
    }
    free(w);
#pragma omp critical
    {
      if (local != ORC_OK && (worst == ORC_OK || local < worst)) worst = local;
    }
  }
  return worst;
}

/* ------------------------------------------------------------------------------
 * Verification of a draft tree (neuralmasteryai.com, "4. Tree Attention & Medusa
 * Heads": several candidate paths verified in one pass; tempatgunting.com, "Draft
 * Model Selection and Tree-Style Variants").  The pages stop at the mask; the walk is
 * this reading of the modified rejection rule ("The Modified Rejection Sampling
 * Algorithm"), applied to one candidate after another:
 *  - nodes 1..n are the draft tokens, node 0 the root (the last context token);
 *    parents[i] is the parent of node i + 1, in 0..i; draft[i] its token;
 *  - p row u (of n + 1) is the target's distribution after node u; q row u (of n) the
 *    distribution node u's children were drawn from, each independently;
 *  - at node u the children are tried in increasing node order against a residual
 *    that starts as p_u: child c (token x) is accepted iff r_c * S * q_u(x) <= R(x),
 *    where R is the residual and S its total (taken as 1 for p_u itself); on a
 *    rejection R becomes max(0, R - S * q_u) (the residual of the normalised R / S
 *    against q_u, scaled back by S) and S its sum;
 *  - an accepted child becomes u; when a node's children are all rejected, or it has
 *    none, one token is drawn from R by inverse CDF (R = p_u when nothing was
 *    rejected), and the walk ends.
 * For a chain (parents[i] = i) this is exactly the rule of verify_one above, with the
 * same uniforms: r_c = r[c - 1] (word 0 of counter (c - 1, b)), the draw at node u
 * uses s[u] (word 1 of counter (u, b)).  A rejection that leaves a zero residual
 * (impossible in exact arithmetic) falls back to drawing from p_u.
 * Outputs per sequence: accepted_len (accepted draft tokens), out_tokens [n + 1] (the
 * accepted path's tokens, the drawn token, then -1), path [n] (the accepted nodes,
 * then -1), and the margin / flag of verify_one, the flag at the output position of
 * the first decision whose uniform lies within flag_window of its threshold.
 * ---------------------------------------------------------------------------- */
static double residual_at(double p, double q, const double* S, int k) {
  double r = p; /* R_0 = p, R_{i+1} = max(0, R_i - S_i q), S_0 = 1 */
  for (int i = 0; i < k; ++i) {
    const double d = r - S[i] * q;
    r = d > 0.0 ? d : 0.0;
  }
  return r;
}

static int verify_tree_one(const float* pb, const float* qb, const int32_t* xb,
                           const int32_t* par, const double* rb, const double* sb, int n, int V,
                           double flag_window, double* w, double* S, int32_t* acc_out,
                           int32_t* ob, int32_t* path, double* margin_out, int32_t* flag_out,
                           int32_t* fallback_out) {
  for (int t = 0; t <= n; ++t) ob[t] = -1;
  for (int t = 0; t < n; ++t) path[t] = -1;
  *acc_out = -1;
  *margin_out = 0.0;
  *flag_out = -1;
  *fallback_out = 0;
  for (int i = 0; i < n; ++i) {
    if (par[i] < 0 || par[i] > i) return ORC_E_ARG;
    if (xb[i] < 0 || xb[i] >= V) return ORC_E_TOKEN;
  }
  double mg = INFINITY;
  int first_flag = -1, depth = 0, u = 0, fb = 0;
  for (;;) {
    const float* pu = pb + (size_t)u * V;
    const float* qu = qb + (size_t)(u < n ? u : 0) * V;
    int k = 0, next = -1;
    S[0] = 1.0;
    for (int c = u + 1; c <= n; ++c) {
      if (par[c - 1] != u) continue;
      const int x = xb[c - 1];
      const double qx = (double)qu[x];
      const double Rx = residual_at((double)pu[x], qx, S, k);
      const double rc = rb[c - 1];
      if (qx > 0.0) {
        const double d = fabs(rc - Rx / (S[k] * qx));
        if (d < mg) mg = d;
        if (d < flag_window && first_flag < 0) first_flag = depth;
      }
      if (rc * S[k] * qx <= Rx) {
        next = c;
        break;
      }
      double sum = 0.0; /* the rejection's new residual and its total */
      for (int y = 0; y < V; ++y) {
        const double d = residual_at((double)pu[y], (double)qu[y], S, k) - S[k] * (double)qu[y];
        sum += d > 0.0 ? d : 0.0;
      }
      S[++k] = sum;
      if (sum == 0.0) {
        fb = 1;
        break;
      }
    }
    if (next >= 0) {
      ob[depth] = xb[next - 1];
      path[depth] = next;
      ++depth;
      u = next;
      continue;
    }
    /* Draw at node u from the residual (p_u after no rejection, or on the fallback). */
    double tot = 0.0;
    for (int y = 0; y < V; ++y) {
      w[y] = (k == 0 || fb) ? (double)pu[y]
                            : residual_at((double)pu[y], (double)qu[y], S, k);
      tot += w[y];
    }
    if (!(tot > 0.0)) {
      *acc_out = depth;
      return ORC_E_DIST;
    }
    const double su = sb[u];
    const double target = su * tot;
    int drawn = -1;
    double c = 0.0;
    for (int y = 0; y < V; ++y) {
      const double before = c;
      c += w[y];
      if (w[y] > 0.0 && c > target) {
        drawn = y;
        const double d = fmin(su - before / tot, c / tot - su);
        if (d < mg) mg = d;
        if (d < flag_window && first_flag < 0) first_flag = depth;
        break;
      }
    }
    if (drawn < 0) {
      for (int y = V - 1; y >= 0; --y)
        if (w[y] > 0.0) {
          drawn = y;
          break;
        }
      mg = 0.0;
      if (first_flag < 0) first_flag = depth;
    }
    ob[depth] = drawn;
    *acc_out = depth;
    *margin_out = mg;
    *flag_out = first_flag;
    *fallback_out = fb;
    return ORC_OK;
  }
}

int oracle_spec_verify_tree_given_uniforms(const float* p, const float* q, const int32_t* draft,
                                           const int32_t* parents, const double* r,
                                           const double* s, int B, int n, int V,
                                           double flag_window, int32_t* accepted_len,
                                           int32_t* out_tokens, int32_t* path, double* margin,
                                           int32_t* flag_pos, int32_t* fallback) {
  if (B < 0 || n < 1 || V <= 0) return ORC_E_ARG;
  int worst = ORC_OK;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    double* S = (double*)malloc(sizeof(double) * (size_t)(n + 2));
    int local = (w && S) ? ORC_OK : ORC_E_ARG;
#pragma omp for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
      if (!w || !S) continue;
      double mg;
      int32_t fp, fbk;
      const int rc = verify_tree_one(
          p + (size_t)b * (n + 1) * V, q + (size_t)b * n * V, draft + (size_t)b * n,
          parents + (size_t)b * n, r + (size_t)b * n, s + (size_t)b * (n + 1), n, V,
          flag_window, w, S, accepted_len + b, out_tokens + (size_t)b * (n + 1),
          path + (size_t)b * n, &mg, &fp, &fbk);
      if (margin) margin[b] = mg;
      if (flag_pos) flag_pos[b] = fp;
      if (fallback) fallback[b] = fbk;
      if (rc != ORC_OK && local == ORC_OK) local = rc;
    }
    free(w);
    free(S);
#pragma omp critical
    {
      if (local != ORC_OK && (worst == ORC_OK || local < worst)) worst = local;
    }
  }
  return worst;
}

/* Full oracle: Philox uniforms followed by the rejection rule above. */
int oracle_spec_verify(const float* p, const float* q, const int32_t* draft, uint64_t seed,
                       int B, int k, int V, double flag_window, int32_t* accepted_len,
                       int32_t* out_tokens, double* margin, int32_t* flag_pos,
                       int32_t* fallback) {
  if (B < 0 || k < 0 || V <= 0) return ORC_E_ARG;
  double* r = (double*)malloc(sizeof(double) * ((size_t)B * k + 1));
  double* s = (double*)malloc(sizeof(double) * ((size_t)B * (k + 1) + 1));
  if (!r || !s) {
    free(r);
    free(s);
    return ORC_E_ARG;
  }
  oracle_uniforms(seed, B, k, r, s);
  const int rc = oracle_spec_verify_given_uniforms(p, q, draft, r, s, B, k, V, flag_window,
                                                   accepted_len, out_tokens, margin, flag_pos,
                                                   fallback);
  free(r);
  free(s);
  return rc;
}

/* Full tree oracle: Philox uniforms (r[b][i] for node i + 1, s[b][u] for the draw at
 * node u, as oracle_uniforms with k = n) followed by the walk above. */
int oracle_spec_verify_tree(const float* p, const float* q, const int32_t* draft,
                            const int32_t* parents, uint64_t seed, int B, int n, int V,
                            double flag_window, int32_t* accepted_len, int32_t* out_tokens,
                            int32_t* path, double* margin, int32_t* flag_pos,
                            int32_t* fallback) {
  if (B < 0 || n < 1 || V <= 0) return ORC_E_ARG;
  double* r = (double*)malloc(sizeof(double) * ((size_t)B * n + 1));
  double* s = (double*)malloc(sizeof(double) * ((size_t)B * (n + 1) + 1));
  if (!r || !s) {
    free(r);
    free(s);
    return ORC_E_ARG;
  }
  oracle_uniforms(seed, B, n, r, s);
  const int rc = oracle_spec_verify_tree_given_uniforms(p, q, draft, parents, r, s, B, n, V,
                                                        flag_window, accepted_len, out_tokens,
                                                        path, margin, flag_pos, fallback);
  free(r);
  free(s);
  return rc;
}
