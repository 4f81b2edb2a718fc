/*
 * oracle.c -- plain, slow, obviously-correct fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It shares no
 * code with the CUDA library.  Single-threaded, no vectorisation tricks,
 * no blocking or reordering beyond what the definitions below state.
 *
 * Sources (web pages; quoted by title and section):
 *  [SD]  "How speculative decoding doubles LLM speed without quality loss"
 *        (dothoosh.com): sections "The speculative execution cycle"
 *        (step 2 verification, step 3 sampling), "Absolute mathematical
 *        exactness" and "Modern architecture variants" (SpecInfer's draft
 *        tree).
 *  [KV]  "KV cache & Flash Attention" lesson (nextadmin.net): sections
 *        "KV-cache math", "FlashAttention -- the tiling trick",
 *        "PagedAttention -- the KV cache as virtual memory",
 *        "Implementation, step 2: tiled softmax".
 *  [SL]  "How StreamingLLM stabilizes million-token streams via attention
 *        sinks" (dothoosh.com): sections "The softmax problem",
 *        "Why sliding windows fail", "The StreamingLLM solution".
 *  [MD]  "How Moondream cut VLM inference latency by 35% via pipelined
 *        decoding" (dothoosh.com): section "Mechanism one: ping-pong slots"
 *        and "Mechanism two: forward first, then sample" (constrained
 *        decoding sets disallowed tokens' logits to -inf before sampling).
 *  [SP]  "Speculative decoding: how AI models get faster without getting
 *        bigger" (aioapex.com): sections "What speculative decoding does" and
 *        "Real-world adoption" (tree speculation, longest accepted path).
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): query i of a q_len-row verify block sits at absolute position
 * t_i = seq_len - q_len + i and sees keys j <= t_i (causal inside the draft,
 * [SD] step 2); with window > 0 a key is visible iff j < n_sink or
 * j > t_i - window (sinks plus the last `window` keys, the query's own key
 * included, [SL] "The StreamingLLM solution"); window == 0 disables both;
 * GQA maps query head h to kv head floor(h / (Hq/Hkv)); lse is the natural
 * log-sum-exp of the scaled scores over the visible set.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- element access: the stored bits widened to fp64 ------------------ */

/* ---- FP8 E4M3 (the OCP 8-bit float: 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 = NaN), the format behind the
 * "--kv-cache-dtype fp8" option the KV-cache lesson names ([KV] "Practical
 * use") and the KV quantisation [SL] lists ("The KV cache memory
 * bottleneck").  Decoding follows the definition; encoding takes the
 * nearest finite value, ties to the even code, saturating at +-448. ---- */

static double e4m3_value(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);        /* subnormal */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

static uint8_t e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
  const double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E;       /* saturate */
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {         /* every finite magnitude */
    const double d = fabs(e4m3_value((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_d = d;
    }
  }
  return sign | (uint8_t)best;
}

int oracle_e4m3_decode(const uint8_t *codes, long n, double *out) {
  for (long i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
  return 0;
}

int oracle_e4m3_encode(const float *x, long n, float scale, uint8_t *out) {
  if (!(scale > 0.0f)) return -1;
  for (long i = 0; i < n; ++i) out[i] = e4m3_encode((double)(x[i] / scale));
  return 0;
}

static double widen(const void *base, size_t idx, int dtype) {
  if (dtype == 0) return (double)((const float *)base)[idx];
  if (dtype == 2) return e4m3_value(((const uint8_t *)base)[idx]);
  /* bfloat16: the upper 16 bits of an IEEE fp32 pattern. */
  uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ---- mask: [SD] step 2 (causal) and [SL] (sinks + sliding window) ------ */

static int key_visible(long j, long t, int n_sink, int window) {
  if (j < 0 || j > t) return 0;
  if (window == 0) return 1;
  return (j < n_sink) || (j > t - window);
}

/* The draft-tree mask ([SD] "Modern architecture variants": SpecInfer checks
 * every branch of a draft tree in one pass with a two-dimensional attention
 * mask).  The q_len new rows of a sequence are the tree's nodes, node k at
 * position base + k; query node i sees every key before base and the node
 * keys whose bit is set in its mask word (its ancestors and itself). */
static int key_visible_tree(long j, long t, long base, uint32_t mask) {
  if (j < 0 || j > t) return 0;
  if (j < base) return 1;
  return (int)((mask >> (j - base)) & 1u);
}

/* Flat element offset of row `pos` of the logical sequence b, kv head g.
 * [KV] "PagedAttention": logical position -> (block_table[b][pos/bs], pos%bs).
 * Returns -1 if the physical block id is out of range. */
static long kv_offset(const int32_t *block_table, int max_blocks, int b,
                      long pos, int block_size, int num_kv_heads, int g,
                      int head_dim, int num_blocks) {
  long lb = pos / block_size;
  if (lb >= max_blocks) return -1;
  int32_t phys = block_table[(long)b * max_blocks + lb];
  if (phys < 0 || phys >= num_blocks) return -1;
  long row = pos % block_size;
  return (((long)phys * num_kv_heads + g) * block_size + row) * head_dim;
}

static int check_sizes(int batch, int num_q_heads, int num_kv_heads,
                       int head_dim, int block_size, int max_blocks,
                       int num_blocks, int dtype, int q_len, int n_sink,
                       int window) {
  if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 ||
      block_size < 1 || max_blocks < 0 || num_blocks < 0 || q_len < 1 ||
      n_sink < 0 || window < 0 || dtype < 0 || dtype > 2)
    return -1;
  if (num_q_heads % num_kv_heads != 0) return -1;
  return 0;
}

/* ---- exact attention: [KV] "FlashAttention" (S = QK^T, P = softmax(S),
 * O = PV) and [SL] "The softmax problem" (softmax(QK^T/sqrt(d))V) -------- */

/* q in `dtype` (fp32 or bf16); the caches in kv_dtype (the same, or 2 = FP8
 * E4M3 codes whose values are scaled by k_scale / v_scale). */
static int attention_rows(int batch, int num_q_heads, int num_kv_heads,
                          int head_dim, int block_size, int max_blocks_per_seq,
                          int num_blocks, int dtype, int kv_dtype,
                          double k_scale, double v_scale, const void *q,
                          const void *k_cache, const void *v_cache,
                          const int32_t *block_table, const int32_t *seq_lens,
                          int q_len, int n_sink, int window,
                          const uint32_t *tree_mask, float scale,
                          const int64_t *rows, int64_t n_rows, double *out,
                          double *lse) {
  if (check_sizes(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                  max_blocks_per_seq, num_blocks, dtype, q_len, n_sink,
                  window))
    return -1;
  if (tree_mask && (window != 0 || q_len > 32)) return -1;
  const int64_t total_rows = (int64_t)batch * q_len * num_q_heads;
  if (rows == NULL) n_rows = total_rows;
  const int group = num_q_heads / num_kv_heads;
  const double sc = (double)scale;

  long max_len = 0;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  double *s = (double *)malloc(sizeof(double) * (size_t)(max_len + 1));
  long *koff = (long *)malloc(sizeof(long) * (size_t)(max_len + 1));
  if (!s || !koff) {
    free(s);
    free(koff);
    return -1;
  }
  int status = 0;

  for (int64_t n = 0; n < n_rows && status == 0; ++n) {
    const int64_t row = rows ? rows[n] : n;
    if (row < 0 || row >= total_rows) {
      status = -1;
      break;
    }
    const int h = (int)(row % num_q_heads);
    const int i = (int)((row / num_q_heads) % q_len);
    const int b = (int)(row / ((int64_t)num_q_heads * q_len));
    const int g = h / group; /* GQA: contiguous head groups */
    const long L = seq_lens[b];
    if (L < q_len) {
      status = -3;
      break;
    }
    const long t = L - q_len + i; /* absolute position of query i */

    /* 1. gather the visible keys and their scores */
    long nv = 0;
    for (long j = 0; j <= t; ++j) {
      if (tree_mask ? !key_visible_tree(j, t, L - q_len,
                                        tree_mask[(size_t)b * q_len + i])
                    : !key_visible(j, t, n_sink, window))
        continue;
      long off = kv_offset(block_table, max_blocks_per_seq, b, j, block_size,
                           num_kv_heads, g, head_dim, num_blocks);
      if (off < 0) {
        status = -2;
        break;
      }
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d)
        dot += widen(q, (size_t)row * head_dim + d, dtype) *
               (k_scale * widen(k_cache, (size_t)off + d, kv_dtype));
      s[nv] = sc * dot;
      koff[nv] = off;
      ++nv;
    }
    if (status) break;

    /* 2. softmax over the visible set, max-subtracted */
    double m = -INFINITY;
    for (long k = 0; k < nv; ++k)
      if (s[k] > m) m = s[k];
    double z = 0.0;
    for (long k = 0; k < nv; ++k) z += exp(s[k] - m);

    /* 3. O = P V */
    double *o = out + (size_t)n * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    for (long k = 0; k < nv; ++k) {
      double p = exp(s[k] - m) / z;
      for (int d = 0; d < head_dim; ++d)
        o[d] += p * (v_scale * widen(v_cache, (size_t)koff[k] + d, kv_dtype));
    }
    lse[n] = m + log(z);
  }
  free(s);
  free(koff);
  return status;
}

int oracle_paged_attention(int batch, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, int max_blocks_per_seq,
                           int num_blocks, int dtype, const void *q,
                           const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int q_len, int n_sink, int window, float scale,
                           const int64_t *rows, int64_t n_rows, double *out,
                           double *lse) {
  if (dtype == 2) return -1; /* q is fp32 or bf16 */
  return attention_rows(batch, num_q_heads, num_kv_heads, head_dim,
                        block_size, max_blocks_per_seq, num_blocks, dtype,
                        dtype, 1.0, 1.0, q, k_cache, v_cache, block_table,
                        seq_lens, q_len, n_sink, window, NULL, scale, rows,
                        n_rows, out, lse);
}

int oracle_paged_attention_fp8(int batch, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size,
                               int max_blocks_per_seq, int num_blocks,
                               const void *q, const void *k_cache,
                               const void *v_cache, double k_scale,
                               double v_scale, const int32_t *block_table,
                               const int32_t *seq_lens, int q_len, int n_sink,
                               int window, float scale, const int64_t *rows,
                               int64_t n_rows, double *out, double *lse) {
  return attention_rows(batch, num_q_heads, num_kv_heads, head_dim,
                        block_size, max_blocks_per_seq, num_blocks, 1, 2,
                        k_scale, v_scale, q, k_cache, v_cache, block_table,
                        seq_lens, q_len, n_sink, window, NULL, scale, rows,
                        n_rows, out, lse);
}

int oracle_paged_tree_attention(int batch, int num_q_heads, int num_kv_heads,
                                int head_dim, int block_size,
                                int max_blocks_per_seq, int num_blocks,
                                int dtype, const void *q, const void *k_cache,
                                const void *v_cache,
                                const int32_t *block_table,
                                const int32_t *seq_lens, int q_len,
                                const uint32_t *tree_mask, float scale,
                                const int64_t *rows, int64_t n_rows,
                                double *out, double *lse) {
  if (!tree_mask || dtype == 2) return -1;
  return attention_rows(batch, num_q_heads, num_kv_heads, head_dim,
                        block_size, max_blocks_per_seq, num_blocks, dtype,
                        dtype, 1.0, 1.0, q, k_cache, v_cache, block_table,
                        seq_lens, q_len, 0, 0, tree_mask, scale, rows, n_rows,
                        out, lse);
}

/* ---- tiled variant: [KV] "FlashAttention -- the tiling trick" and
 * "Implementation, step 2": a running (max, sum, accumulator) folded over
 * blocks of keys, rescaled by exp(m_old - m_new); parts merged by LSE. ---- */

int oracle_paged_attention_tiled(int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, int block_size,
                                 int max_blocks_per_seq, int num_blocks,
                                 int dtype, const void *q, const void *k_cache,
                                 const void *v_cache,
                                 const int32_t *block_table,
                                 const int32_t *seq_lens, int q_len, int n_sink,
                                 int window, float scale, int tile,
                                 int n_splits, double *out, double *lse) {
  if (check_sizes(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                  max_blocks_per_seq, num_blocks, dtype, q_len, n_sink,
                  window) ||
      tile < 1 || n_splits < 1)
    return -1;
  const int group = num_q_heads / num_kv_heads;
  const double sc = (double)scale;
  long max_len = 0;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  long *keys = (long *)malloc(sizeof(long) * (size_t)(max_len + 1));
  double *part_o = (double *)malloc(sizeof(double) * (size_t)n_splits * head_dim);
  double *part_lse = (double *)malloc(sizeof(double) * (size_t)n_splits);
  double *acc = (double *)malloc(sizeof(double) * (size_t)head_dim);
  double *sblk = (double *)malloc(sizeof(double) * (size_t)tile);
  if (!keys || !part_o || !part_lse || !acc || !sblk) {
    free(keys); free(part_o); free(part_lse); free(acc); free(sblk);
    return -1;
  }
  int status = 0;
  const int64_t total_rows = (int64_t)batch * q_len * num_q_heads;
  for (int64_t row = 0; row < total_rows && status == 0; ++row) {
    const int h = (int)(row % num_q_heads);
    const int i = (int)((row / num_q_heads) % q_len);
    const int b = (int)(row / ((int64_t)num_q_heads * q_len));
    const int g = h / group;
    const long L = seq_lens[b];
    if (L < q_len) { status = -3; break; }
    const long t = L - q_len + i;
    long nv = 0;
    for (long j = 0; j <= t; ++j) {
      if (!key_visible(j, t, n_sink, window)) continue;
      long off = kv_offset(block_table, max_blocks_per_seq, b, j, block_size,
                           num_kv_heads, g, head_dim, num_blocks);
      if (off < 0) { status = -2; break; }
      keys[nv++] = off;
    }
    if (status) break;

    for (int part = 0; part < n_splits; ++part) {
      long lo = nv * part / n_splits, hi = nv * (part + 1) / n_splits;
      double m = -INFINITY, ssum = 0.0;
      for (int d = 0; d < head_dim; ++d) acc[d] = 0.0;
      for (long start = lo; start < hi; start += tile) {
        long cnt = (hi - start < tile) ? hi - start : tile;
        double new_m = m;
        for (long k = 0; k < cnt; ++k) {
          double dot = 0.0;
          for (int d = 0; d < head_dim; ++d)
            dot += widen(q, (size_t)row * head_dim + d, dtype) *
                   widen(k_cache, (size_t)keys[start + k] + d, dtype);
          sblk[k] = sc * dot;
          if (sblk[k] > new_m) new_m = sblk[k];
        }
        double exp_old = (m == -INFINITY) ? 0.0 : exp(m - new_m);
        ssum *= exp_old;
        for (int d = 0; d < head_dim; ++d) acc[d] *= exp_old;
        for (long k = 0; k < cnt; ++k) {
          double e = exp(sblk[k] - new_m);
          ssum += e;
          for (int d = 0; d < head_dim; ++d)
            acc[d] += e * widen(v_cache, (size_t)keys[start + k] + d, dtype);
        }
        m = new_m;
      }
      if (hi > lo) {
        for (int d = 0; d < head_dim; ++d)
          part_o[(size_t)part * head_dim + d] = acc[d] / ssum;
        part_lse[part] = m + log(ssum);
      } else { /* an empty part carries zero weight */
        for (int d = 0; d < head_dim; ++d) part_o[(size_t)part * head_dim + d] = 0.0;
        part_lse[part] = -INFINITY;
      }
    }
    /* merge the parts: weights exp(lse_part - lse_total) */
    double mx = -INFINITY;
    for (int part = 0; part < n_splits; ++part)
      if (part_lse[part] > mx) mx = part_lse[part];
    double wsum = 0.0;
    for (int part = 0; part < n_splits; ++part)
      if (part_lse[part] != -INFINITY) wsum += exp(part_lse[part] - mx);
    double total = mx + log(wsum);
    double *o = out + (size_t)row * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    for (int part = 0; part < n_splits; ++part) {
      if (part_lse[part] == -INFINITY) continue;
      double w = exp(part_lse[part] - total);
      for (int d = 0; d < head_dim; ++d) o[d] += w * part_o[(size_t)part * head_dim + d];
    }
    lse[row] = total;
  }
  free(keys); free(part_o); free(part_lse); free(acc); free(sblk);
  return status;
}

/* ---- KV append: [KV] "KV cache" (store K and V of every new token) and
 * "PagedAttention" (logical position -> physical block, row) ------------ */

int oracle_kv_append(int batch, int num_kv_heads, int head_dim, int block_size,
                     int max_blocks_per_seq, int num_blocks, int elem_bytes,
                     const void *k_new, const void *v_new, void *k_cache,
                     void *v_cache, const int32_t *block_table,
                     const int32_t *seq_lens, int n_new) {
  if (batch < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
      n_new < 0 || (elem_bytes != 2 && elem_bytes != 4))
    return -1;
  const size_t row_bytes = (size_t)head_dim * elem_bytes;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < n_new) return -1;
    for (int k = 0; k < n_new; ++k) {
      long pos = (long)seq_lens[b] - n_new + k;
      for (int g = 0; g < num_kv_heads; ++g) {
        long off = kv_offset(block_table, max_blocks_per_seq, b, pos,
                             block_size, num_kv_heads, g, head_dim, num_blocks);
        if (off < 0) return -2;
        size_t src = ((((size_t)b * n_new + k) * num_kv_heads) + g) * row_bytes;
        memcpy((char *)k_cache + (size_t)off * elem_bytes,
               (const char *)k_new + src, row_bytes);
        memcpy((char *)v_cache + (size_t)off * elem_bytes,
               (const char *)v_new + src, row_bytes);
      }
    }
  }
  return 0;
}

/* FP8 append: the new rows arrive in bf16; each value x is stored as the
 * E4M3 code of the fp32 quotient x / scale (k_scale for K, v_scale for V),
 * nearest, ties to even, saturated at +-448. */
int oracle_kv_append_fp8(int batch, int num_kv_heads, int head_dim,
                         int block_size, int max_blocks_per_seq,
                         int num_blocks, const uint16_t *k_new,
                         const uint16_t *v_new, uint8_t *k_cache,
                         uint8_t *v_cache, float k_scale, float v_scale,
                         const int32_t *block_table, const int32_t *seq_lens,
                         int n_new) {
  if (batch < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
      n_new < 0 || !(k_scale > 0.0f) || !(v_scale > 0.0f))
    return -1;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < n_new) return -1;
    for (int k = 0; k < n_new; ++k) {
      long pos = (long)seq_lens[b] - n_new + k;
      for (int g = 0; g < num_kv_heads; ++g) {
        long off = kv_offset(block_table, max_blocks_per_seq, b, pos,
                             block_size, num_kv_heads, g, head_dim, num_blocks);
        if (off < 0) return -2;
        size_t src = ((((size_t)b * n_new + k) * num_kv_heads) + g) * head_dim;
        for (int d = 0; d < head_dim; ++d) {
          const float kx = (float)widen(k_new, src + d, 1);
          const float vx = (float)widen(v_new, src + d, 1);
          k_cache[off + d] = e4m3_encode((double)(kx / k_scale));
          v_cache[off + d] = e4m3_encode((double)(vx / v_scale));
        }
      }
    }
  }
  return 0;
}

/* ---- speculative acceptance: [SD] "The speculative execution cycle",
 * step 3, and [SP] "What speculative decoding does" ---------------------- */

/* softmax of one logit row in fp64, max-subtracted */
static void softmax_row(const float *logits, int vocab, double *p) {
  double m = -INFINITY;
  for (int x = 0; x < vocab; ++x)
    if ((double)logits[x] > m) m = (double)logits[x];
  double z = 0.0;
  for (int x = 0; x < vocab; ++x) {
    p[x] = exp((double)logits[x] - m);
    z += p[x];
  }
  for (int x = 0; x < vocab; ++x) p[x] /= z;
}

/* Inverse-CDF draw in token-index order: the smallest x whose running sum of
 * w exceeds u * sum(w); if rounding leaves none, the last x with w_x > 0.
 * Sets *near when u*W lies within eps*W of the running sum at the chosen x or
 * at the one before it. */
static int inverse_cdf(const double *w, int vocab, double u, double eps,
                       int *near) {
  double total = 0.0;
  for (int x = 0; x < vocab; ++x) total += w[x];
  const double target = u * total;
  double c = 0.0;
  for (int x = 0; x < vocab; ++x) {
    double prev = c;
    c += w[x];
    if (c > target) {
      if (fabs(c - target) < eps * total || fabs(prev - target) < eps * total)
        *near = 1;
      return x;
    }
  }
  *near = 1; /* the draw fell off the end by rounding */
  for (int x = vocab - 1; x >= 0; --x)
    if (w[x] > 0.0) return x;
  return vocab - 1;
}

int oracle_spec_accept(int batch, int num_draft, int vocab,
                       const float *target_logits, const float *draft_logits,
                       const int32_t *draft_tokens, const float *uniforms,
                       int32_t *out_tokens, int32_t *n_accepted,
                       int32_t *near_boundary, int32_t *residual_fallback,
                       double eps) {
  if (batch < 0 || num_draft < 1 || vocab < 2) return -1;
  const int K = num_draft;
  double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *qd = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *w = (double *)malloc(sizeof(double) * (size_t)vocab);
  if (!p || !qd || !w) { free(p); free(qd); free(w); return -1; }
  int status = 0;
  for (int b = 0; b < batch && status == 0; ++b) {
    int32_t *emit = out_tokens + (size_t)b * (K + 1);
    const float *u = uniforms + (size_t)b * (K + 1);
    int near = 0, fallback = 0, n_out = 0, accepted_all = 1;
    for (int k = 0; k <= K; ++k) emit[k] = -1;
    for (int i = 0; i < K; ++i) { /* every draft token must be a token id */
      const int x = draft_tokens[(size_t)b * K + i];
      if (x < 0 || x >= vocab) status = -4;
    }
    if (status) break;
    for (int i = 0; i < K; ++i) {
      const int x = draft_tokens[(size_t)b * K + i];
      softmax_row(target_logits + ((size_t)b * (K + 1) + i) * vocab, vocab, p);
      softmax_row(draft_logits + ((size_t)b * K + i) * vocab, vocab, qd);
      /* accept iff r <= min(1, p(x)/q(x)); q(x) = 0 reads as ratio +inf */
      const double r = (double)u[i];
      const double ratio = (qd[x] > 0.0) ? p[x] / qd[x] : INFINITY;
      if (fabs(r - ratio) < eps) near = 1;
      if (r <= ratio) {
        emit[n_out++] = x;
        continue;
      }
      /* rejected at position i: resample from max(0, p - q) normalised */
      double mass = 0.0;
      for (int y = 0; y < vocab; ++y) {
        w[y] = (p[y] - qd[y] > 0.0) ? p[y] - qd[y] : 0.0;
        mass += w[y];
      }
      if (mass == 0.0) { /* impossible in exact arithmetic: sample p */
        fallback = 1;
        for (int y = 0; y < vocab; ++y) w[y] = p[y];
      }
      emit[n_out++] = inverse_cdf(w, vocab, (double)u[K], eps, &near);
      n_accepted[b] = i;
      accepted_all = 0;
      break;
    }
    if (status) break;
    if (accepted_all) {
      /* every draft accepted: the bonus token from the last target row */
      softmax_row(target_logits + ((size_t)b * (K + 1) + K) * vocab, vocab, p);
      emit[n_out++] = inverse_cdf(p, vocab, (double)u[K], eps, &near);
      n_accepted[b] = K;
    }
    if (near_boundary) near_boundary[b] = near;
    if (residual_fallback) residual_fallback[b] = fallback;
  }
  free(p); free(qd); free(w);
  return status;
}

/* ---- tree acceptance: [SD] "Modern architecture variants" (SpecInfer: a
 * tree of speculative branches checked in one pass) and [SP] "Real-world
 * adoption" (the verifier keeps the longest accepted path).  Reading: the
 * walk starts at the root; a node's children are tried in index order with
 * the linear rule of [SD] step 3, u_c <= r(x_c)/q(x_c), where r starts as
 * the target distribution after the node and, after each rejected child,
 * becomes the normalised residual max(0, r - q) -- the distribution the
 * linear rule resamples from; an accepted child becomes the next node; when
 * every child is rejected (or the node is a leaf) one token is drawn from r
 * with u_0.  On a chain this is exactly the linear rule. ---------------- */

int oracle_spec_accept_tree(int batch, int num_nodes, int vocab,
                            const float *target_logits,
                            const float *draft_logits, const int32_t *parents,
                            const int32_t *node_tokens, const float *uniforms,
                            int32_t *out_tokens, int32_t *out_nodes,
                            int32_t *n_accepted, int32_t *near_boundary,
                            int32_t *residual_fallback, double eps) {
  if (batch < 0 || num_nodes < 1 || vocab < 2) return -1;
  const int N = num_nodes;
  double *r = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *qd = (double *)malloc(sizeof(double) * (size_t)vocab);
  if (!r || !qd) { free(r); free(qd); return -1; }
  int status = 0;
  for (int b = 0; b < batch && status == 0; ++b) {
    const int32_t *par = parents + (size_t)b * N;
    const int32_t *tok = node_tokens + (size_t)b * N;
    const float *u = uniforms + (size_t)b * N;
    int32_t *emit = out_tokens + (size_t)b * N;
    int32_t *nodes = out_nodes + (size_t)b * N;
    for (int k = 0; k < N; ++k) { emit[k] = -1; nodes[k] = -1; }
    /* a tree: node 0 is the root, every other node's parent comes first */
    if (par[0] != -1) status = -1;
    for (int c = 1; c < N; ++c) {
      if (par[c] < 0 || par[c] >= c) status = -1;
      if (tok[c] < 0 || tok[c] >= vocab) status = status ? status : -4;
    }
    if (status) break;
    int near = 0, fallback = 0, n_out = 0, cur = 0;
    for (;;) {
      softmax_row(target_logits + ((size_t)b * N + cur) * vocab, vocab, r);
      softmax_row(draft_logits + ((size_t)b * N + cur) * vocab, vocab, qd);
      int next = -1;
      for (int c = cur + 1; c < N && next < 0; ++c) {
        if (par[c] != cur) continue;
        const int x = tok[c];
        const double ur = (double)u[c];
        const double ratio = (qd[x] > 0.0) ? r[x] / qd[x] : INFINITY;
        if (fabs(ur - ratio) < eps) near = 1;
        if (ur <= ratio) {
          next = c;
          break;
        }
        /* child rejected: continue with the normalised residual */
        double mass = 0.0;
        for (int y = 0; y < vocab; ++y)
          mass += (r[y] - qd[y] > 0.0) ? r[y] - qd[y] : 0.0;
        if (mass == 0.0) { /* impossible in exact arithmetic: keep r */
          fallback = 1;
          continue;
        }
        for (int y = 0; y < vocab; ++y)
          r[y] = ((r[y] - qd[y] > 0.0) ? r[y] - qd[y] : 0.0) / mass;
      }
      if (next < 0) {
        emit[n_out] = inverse_cdf(r, vocab, (double)u[0], eps, &near);
        break;
      }
      emit[n_out] = tok[next];
      nodes[n_out] = next;
      ++n_out;
      cur = next;
    }
    n_accepted[b] = n_out;
    if (near_boundary) near_boundary[b] = near;
    if (residual_fallback) residual_fallback[b] = fallback;
  }
  free(r); free(qd);
  return status;
}

/* ---- the verify epilogue: temperature, constrained decoding, greedy ----
 * [SD] "Deployment limits": sampling temperature T (the distributions are
 * softmax(logits / T) for both models); [MD] section "Mechanism two:
 * forward first, then sample" (constrained decoding): tokens the grammar
 * does not allow get logit -inf
 * before sampling; greedy verification accepts a draft iff it is the
 * target's most likely token.  Readings: mask row i applies to target row
 * i and draft row i; a draft token the mask excludes has p(x) = 0 and is
 * rejected; greedy ties go to the smallest token index. */

/* softmax of one logit row at temperature T over the allowed tokens
 * (allowed == NULL: all); excluded tokens get probability 0. */
static void softmax_row_ex(const float *logits, int vocab, double inv_t,
                           const uint32_t *allowed, double *p) {
  double m = -INFINITY;
  for (int x = 0; x < vocab; ++x) {
    if (allowed && !((allowed[x >> 5] >> (x & 31)) & 1u)) continue;
    const double v = (double)logits[x] * inv_t;
    if (v > m) m = v;
  }
  double z = 0.0;
  for (int x = 0; x < vocab; ++x) {
    if (allowed && !((allowed[x >> 5] >> (x & 31)) & 1u)) {
      p[x] = 0.0;
      continue;
    }
    p[x] = exp((double)logits[x] * inv_t - m);
    z += p[x];
  }
  for (int x = 0; x < vocab; ++x) p[x] /= z;
}

/* most likely allowed token of a logit row, smallest index on ties */
static int argmax_row(const float *logits, int vocab, const uint32_t *allowed) {
  int best = -1;
  for (int x = 0; x < vocab; ++x) {
    if (allowed && !((allowed[x >> 5] >> (x & 31)) & 1u)) continue;
    if (best < 0 || logits[x] > logits[best]) best = x;
  }
  return best;
}

int oracle_spec_accept_ex(int batch, int num_draft, int vocab,
                          const float *target_logits,
                          const float *draft_logits,
                          const int32_t *draft_tokens, const float *uniforms,
                          double temperature, const uint32_t *allowed,
                          int greedy, int32_t *out_tokens,
                          int32_t *n_accepted, int32_t *near_boundary,
                          double eps) {
  if (batch < 0 || num_draft < 1 || vocab < 2) return -1;
  if (!greedy && !(temperature > 0.0)) return -1;
  const int K = num_draft;
  const int words = (vocab + 31) / 32;
  const double inv_t = greedy ? 1.0 : 1.0 / temperature;
  double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *qd = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *w = (double *)malloc(sizeof(double) * (size_t)vocab);
  if (!p || !qd || !w) { free(p); free(qd); free(w); return -1; }
  int status = 0;
  for (int b = 0; b < batch && status == 0; ++b) {
    int32_t *emit = out_tokens + (size_t)b * (K + 1);
    const float *u = uniforms + (size_t)b * (K + 1);
    int near = 0, n_out = 0, j = K;
    for (int k = 0; k <= K; ++k) emit[k] = -1;
    for (int i = 0; i < K; ++i) {
      const int x = draft_tokens[(size_t)b * K + i];
      if (x < 0 || x >= vocab) status = -4;
    }
    if (status) break;
    for (int i = 0; i < K; ++i) {
      const int x = draft_tokens[(size_t)b * K + i];
      const float *tl = target_logits + ((size_t)b * (K + 1) + i) * vocab;
      const float *dl = draft_logits + ((size_t)b * K + i) * vocab;
      const uint32_t *al =
          allowed ? allowed + ((size_t)b * (K + 1) + i) * words : NULL;
      const int ok_x = !al || ((al[x >> 5] >> (x & 31)) & 1u);
      if (greedy) {
        if (ok_x && x == argmax_row(tl, vocab, al)) {
          emit[n_out++] = x;
          continue;
        }
        emit[n_out++] = argmax_row(tl, vocab, al);
        j = i;
        break;
      }
      softmax_row_ex(tl, vocab, inv_t, al, p);
      softmax_row_ex(dl, vocab, inv_t, al, qd);
      const double r = (double)u[i];
      const double ratio = !ok_x ? 0.0 : (qd[x] > 0.0) ? p[x] / qd[x] : INFINITY;
      if (ok_x && fabs(r - ratio) < eps) near = 1;
      if (ok_x && r <= ratio) {
        emit[n_out++] = x;
        continue;
      }
      double mass = 0.0;
      for (int y = 0; y < vocab; ++y) {
        w[y] = (p[y] - qd[y] > 0.0) ? p[y] - qd[y] : 0.0;
        mass += w[y];
      }
      if (mass == 0.0)
        for (int y = 0; y < vocab; ++y) w[y] = p[y];
      emit[n_out++] = inverse_cdf(w, vocab, (double)u[K], eps, &near);
      j = i;
      break;
    }
    if (j == K) { /* every draft accepted: the bonus from the last row */
      const float *tl = target_logits + ((size_t)b * (K + 1) + K) * vocab;
      const uint32_t *al =
          allowed ? allowed + ((size_t)b * (K + 1) + K) * words : NULL;
      if (greedy) {
        emit[n_out++] = argmax_row(tl, vocab, al);
      } else {
        softmax_row_ex(tl, vocab, inv_t, al, p);
        emit[n_out++] = inverse_cdf(p, vocab, (double)u[K], eps, &near);
      }
    }
    n_accepted[b] = j;
    if (near_boundary) near_boundary[b] = near;
  }
  free(p); free(qd); free(w);
  return status;
}

/* ---- outcomes that are valid near a decision boundary ----------------
 * The acceptance rule ([SD] step 3) is a chain of comparisons: u_i against
 * p(x)/q(x), and u*W against running sums of the draw's weights.  In exact
 * arithmetic each has one answer; an implementation in another precision
 * may take the other side of a comparison that lies within eps of its
 * boundary (the band within which decisions are not compared exactly).
 * The functions below list every outcome the literal rule can reach when
 * each comparison within eps of its boundary may go either way, and every
 * other comparison goes as in exact arithmetic.  With eps = 0 the set is
 * the single outcome of the rule. */

/* Tokens a draw from weights w with uniform u may return when the running
 * sums within eps*W of u*W may compare either way: every x of positive
 * weight whose interval [C(x-1), C(x)) meets the band [u*W - eps*W,
 * u*W + eps*W], plus the last token of positive weight when u*W is at or
 * past the total (the rule's fallback).  Writes at most max_cand tokens to
 * cand (in token order) and returns how many there are (which may exceed
 * max_cand). */
static int draw_candidates(const double *w, int vocab, double u, double eps,
                           int32_t *cand, int max_cand) {
  double total = 0.0;
  for (int x = 0; x < vocab; ++x) total += w[x];
  const double target = u * total;
  const double lo = target - eps * total, hi = target + eps * total;
  int n = 0, last_pos = -1, last_added = -1, reached = 0;
  double c = 0.0;
  for (int x = 0; x < vocab; ++x) {
    const double prev = c;
    c += w[x];
    if (c > target) reached = 1;
    if (!(w[x] > 0.0)) continue;
    last_pos = x;
    if (prev <= hi && c > lo) {
      if (n < max_cand) cand[n] = x;
      ++n;
      last_added = x;
    }
  }
  if (!reached && last_pos >= 0 && last_added != last_pos) {
    if (n < max_cand) cand[n] = last_pos;
    ++n;
  }
  return n;
}

int oracle_spec_accept_valid(int batch, int num_draft, int vocab,
                             const float *target_logits,
                             const float *draft_logits,
                             const int32_t *draft_tokens,
                             const float *uniforms, double temperature,
                             const uint32_t *allowed, int32_t *path_valid,
                             int32_t *cand, int32_t *n_cand, int max_cand,
                             double eps) {
  if (batch < 0 || num_draft < 1 || vocab < 2 || max_cand < 1) return -1;
  if (!(temperature > 0.0) || eps < 0.0) return -1;
  const int K = num_draft;
  const int words = (vocab + 31) / 32;
  const double inv_t = 1.0 / temperature;
  double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *qd = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *w = (double *)malloc(sizeof(double) * (size_t)vocab);
  if (!p || !qd || !w) { free(p); free(qd); free(w); return -1; }
  int status = 0;
  for (int b = 0; b < batch && status == 0; ++b) {
    const float *u = uniforms + (size_t)b * (K + 1);
    int32_t *pv = path_valid + (size_t)b * (K + 1);
    for (int j = 0; j <= K; ++j) {
      pv[j] = 0;
      n_cand[(size_t)b * (K + 1) + j] = 0;
      for (int c = 0; c < max_cand; ++c)
        cand[((size_t)b * (K + 1) + j) * max_cand + c] = -1;
    }
    for (int i = 0; i < K; ++i) {
      const int x = draft_tokens[(size_t)b * K + i];
      if (x < 0 || x >= vocab) status = -4;
    }
    if (status) break;
    /* path j < K: drafts 0..j-1 accepted, draft j rejected, one draw from
     * the residual of row j; path K: all accepted, the bonus draw from
     * row K.  Walk the drafts while "accepted" stays a valid answer. */
    for (int j = 0; j <= K; ++j) {
      const float *tl = target_logits + ((size_t)b * (K + 1) + j) * vocab;
      const uint32_t *al =
          allowed ? allowed + ((size_t)b * (K + 1) + j) * words : NULL;
      const size_t slot = (size_t)b * (K + 1) + j;
      softmax_row_ex(tl, vocab, inv_t, al, p);
      if (j == K) { /* every draft accepted */
        pv[j] = 1;
        n_cand[slot] = draw_candidates(p, vocab, (double)u[K], eps,
                                       cand + slot * max_cand, max_cand);
        break;
      }
      const int x = draft_tokens[(size_t)b * K + j];
      const float *dl = draft_logits + ((size_t)b * K + j) * vocab;
      softmax_row_ex(dl, vocab, inv_t, al, qd);
      const int ok_x = !al || ((al[x >> 5] >> (x & 31)) & 1u);
      const double r = (double)u[j];
      const double ratio = !ok_x ? 0.0 : (qd[x] > 0.0) ? p[x] / qd[x] : INFINITY;
      const int near = ok_x && fabs(r - ratio) < eps;
      const int can_accept = ok_x && (r <= ratio || near);
      const int can_reject = !ok_x || r > ratio || near;
      if (can_reject) {
        double mass = 0.0;
        for (int y = 0; y < vocab; ++y) {
          w[y] = (p[y] - qd[y] > 0.0) ? p[y] - qd[y] : 0.0;
          mass += w[y];
        }
        if (mass == 0.0)
          for (int y = 0; y < vocab; ++y) w[y] = p[y];
        pv[j] = 1;
        n_cand[slot] = draw_candidates(w, vocab, (double)u[K], eps,
                                       cand + slot * max_cand, max_cand);
      }
      if (!can_accept) break;
    }
  }
  free(p); free(qd); free(w);
  return status;
}

/* Tree walk with both answers at every accept test within eps of its
 * boundary: a depth-first enumeration of the literal walk of
 * oracle_spec_accept_tree.  Each outcome is one row of `outcomes`:
 * [N entries: the accepted nodes in order, -1 padded] [n_accepted]
 * [n_cand] [max_cand candidate tokens of the final draw, -1 padded]. */
typedef struct {
  int N, vocab, max_out, max_cand, n_out;
  double eps;
  const float *tl, *dl, *u;
  const int32_t *par, *tok;
  double *scratch; /* 2 * vocab doubles per depth */
  int32_t *rows;
  int32_t path[64];
} tree_enum;

static void tree_enum_emit(tree_enum *e, int depth, const double *r) {
  const int stride = e->N + 2 + e->max_cand;
  int32_t tmp[1];
  if (e->n_out < e->max_out) {
    int32_t *row = e->rows + (size_t)e->n_out * stride;
    for (int k = 0; k < e->N; ++k) row[k] = k < depth ? e->path[k] : -1;
    row[e->N] = depth;
    for (int c = 0; c < e->max_cand; ++c) row[e->N + 2 + c] = -1;
    row[e->N + 1] = draw_candidates(r, e->vocab, (double)e->u[0], e->eps,
                                    row + e->N + 2, e->max_cand);
  } else {
    (void)draw_candidates(r, e->vocab, (double)e->u[0], e->eps, tmp, 1);
  }
  ++e->n_out;
}

static void tree_enum_node(tree_enum *e, int cur, int depth) {
  const int V = e->vocab;
  double *r = e->scratch + (size_t)2 * depth * V;
  double *qd = r + V;
  softmax_row(e->tl + (size_t)cur * V, V, r);
  softmax_row(e->dl + (size_t)cur * V, V, qd);
  for (int c = cur + 1; c < e->N; ++c) {
    if (e->par[c] != cur) continue;
    const int x = e->tok[c];
    const double ur = (double)e->u[c];
    const double ratio = (qd[x] > 0.0) ? r[x] / qd[x] : INFINITY;
    const int near = fabs(ur - ratio) < e->eps;
    if (ur <= ratio || near) { /* accepting child c is a valid answer */
      e->path[depth] = c;
      tree_enum_node(e, c, depth + 1);
    }
    if (!(ur > ratio || near)) return; /* rejecting it is not */
    double mass = 0.0;
    for (int y = 0; y < V; ++y)
      mass += (r[y] - qd[y] > 0.0) ? r[y] - qd[y] : 0.0;
    if (mass == 0.0) continue; /* the walk keeps r (see above) */
    for (int y = 0; y < V; ++y)
      r[y] = ((r[y] - qd[y] > 0.0) ? r[y] - qd[y] : 0.0) / mass;
  }
  tree_enum_emit(e, depth, r); /* no child accepted: draw from r */
}

int oracle_spec_accept_tree_valid(int batch, int num_nodes, int vocab,
                                  const float *target_logits,
                                  const float *draft_logits,
                                  const int32_t *parents,
                                  const int32_t *node_tokens,
                                  const float *uniforms, int32_t *outcomes,
                                  int32_t *n_outcomes, int max_out,
                                  int max_cand, double eps) {
  if (batch < 0 || num_nodes < 1 || num_nodes > 64 || vocab < 2 ||
      max_out < 1 || max_cand < 1 || eps < 0.0)
    return -1;
  const int N = num_nodes;
  double *scratch =
      (double *)malloc(sizeof(double) * 2 * (size_t)vocab * (size_t)(N + 1));
  if (!scratch) return -1;
  int status = 0;
  const int stride = N + 2 + max_cand;
  for (int b = 0; b < batch && status == 0; ++b) {
    const int32_t *par = parents + (size_t)b * N;
    const int32_t *tok = node_tokens + (size_t)b * N;
    if (par[0] != -1) status = -1;
    for (int c = 1; c < N; ++c) {
      if (par[c] < 0 || par[c] >= c) status = -1;
      if (tok[c] < 0 || tok[c] >= vocab) status = status ? status : -4;
    }
    if (status) break;
    tree_enum e;
    e.N = N; e.vocab = vocab; e.max_out = max_out; e.max_cand = max_cand;
    e.n_out = 0; e.eps = eps;
    e.tl = target_logits + (size_t)b * N * vocab;
    e.dl = draft_logits + (size_t)b * N * vocab;
    e.u = uniforms + (size_t)b * N;
    e.par = par; e.tok = tok; e.scratch = scratch;
    e.rows = outcomes + (size_t)b * max_out * stride;
    for (int k = 0; k < max_out * stride; ++k) e.rows[k] = -1;
    tree_enum_node(&e, 0, 0);
    n_outcomes[b] = e.n_out;
  }
  free(scratch);
  return status;
}
