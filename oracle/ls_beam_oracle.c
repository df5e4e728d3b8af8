/*
 * Oracle for the hierarchical beam-search step and the beam-cache refresh.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library and never includes anything from it.
 *
 * Source: the LightSeq inference article (31duo.com, itemid-283120),
 * section on the hierarchical rewrite of decoding ("层级式改写"):
 *   - naive decoding: softmax over the [batch_size, beam_size, vocab_size]
 *     logits followed by batch_size sorts; the hierarchical method is said to
 *     reach the same, exact top-k per sequence.  This oracle therefore IS the
 *     naive definition: full log-softmax in double precision and one full
 *     sort of every (beam, token) pair of a batch.
 *   - first traversal: the R-top-k bound (k groups, the min of the k group
 *     maxima, never above the true k-th largest) and the per-beam
 *     log_sum_exp; oracle_rtopk_stats() restates it as a diagnostic.
 *   - "update the cache" after selection: oracle_cache_reorder() is the
 *     plain gather of the cache rows by parent beam.
 *
 * Readings where the article is silent:
 *   - x = logit + bias[v] (bias optional) is the value used everywhere.
 *   - candidate score s = beam_score + x - lse, lse = log sum_v exp(x_v).
 *   - a finished beam contributes exactly one candidate (eos_id, its score
 *     unchanged); out_finished = finished[parent] || token == eos_id.
 *   - the top-k is taken over all k*vocab pairs of a batch; order is score
 *     descending, then smaller flattened index j*vocab+v first.
 *   - a live beam whose logits are all -inf, or whose beam score is -inf,
 *     gives every one of its tokens the score -inf.
 *
 * Precision: every sum, exp and log is in double.  fp16 and bf16 logits are
 * decoded exactly to double from their IEEE bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2
#define ORC_F64 3 /* logits already in double (the output projection below) */

/* IEEE 754 binary16: sign, 5-bit biased exponent, 10-bit fraction. */
static double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16 is the top half of an IEEE binary32. */
static double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double orc_logit(const void* logits, int dtype, size_t idx) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)logits)[idx];
    case ORC_F16: return orc_half_to_double(((const uint16_t*)logits)[idx]);
    case ORC_F64: return ((const double*)logits)[idx];
    default: return orc_bf16_to_double(((const uint16_t*)logits)[idx]);
  }
}

/* x[b,j,v] = logit + bias[v], exact in double. */
static void orc_row_values(const void* logits, int dtype, const float* bias, size_t row, int vocab,
                           double* x) {
  for (int v = 0; v < vocab; ++v) {
    double xv = orc_logit(logits, dtype, row * (size_t)vocab + (size_t)v);
    if (bias) xv += (double)bias[v];
    x[v] = xv;
  }
}

/* lse = m + log(sum exp(x - m)), m = max x.  Returns -inf for an all -inf row. */
static double orc_log_sum_exp(const double* x, int n) {
  double m = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (x[i] > m) m = x[i];
  if (m == -INFINITY) return -INFINITY;
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += exp(x[i] - m);
  return m + log(s);
}

typedef struct {
  double s;
  int64_t flat; /* j * vocab + v */
} orc_cand;

/* score descending, then flattened index ascending */
static int orc_cmp_cand(const void* pa, const void* pb) {
  const orc_cand* a = (const orc_cand*)pa;
  const orc_cand* b = (const orc_cand*)pb;
  if (a->s > b->s) return -1;
  if (a->s < b->s) return 1;
  return (a->flat < b->flat) ? -1 : (a->flat > b->flat);
}

/*
 * One beam-search step by the naive definition.
 * logits [batch, k, vocab] (dtype 0 f32, 1 f16 bits, 2 bf16 bits); bias [vocab] or NULL;
 * beam_scores [batch, k]; finished [batch, k] (0/1) or NULL.
 * Writes, per batch, the first m_out entries of the fully sorted candidate list:
 * token, parent, score (double), finished flag.  Entries past the candidate
 * count get token = parent = -1 and score NaN.  out_lse [batch*k] (optional)
 * receives each beam's log-sum-exp (NaN for finished beams).
 * Returns 0, or -1 on bad arguments, -2 on allocation failure.
 */
int oracle_beam_step(const void* logits, int dtype, const float* bias, const float* beam_scores,
                     const uint8_t* finished, int batch, int k, int vocab, int eos_id, int m_out,
                     int32_t* out_token, int32_t* out_parent, double* out_score,
                     uint8_t* out_finished, double* out_lse) {
  if (!logits || !beam_scores || !out_token || !out_parent || !out_score || !out_finished)
    return -1;
  if (batch < 0 || k < 1 || vocab < 1 || m_out < 1 || eos_id < 0 || eos_id >= vocab) return -1;
  if (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16 && dtype != ORC_F64) return -1;
  size_t ncap = (size_t)k * (size_t)vocab;
  orc_cand* cand = (orc_cand*)malloc(ncap * sizeof(orc_cand));
  double* x = (double*)malloc((size_t)vocab * sizeof(double));
  if (!cand || !x) {
    free(cand);
    free(x);
    return -2;
  }
  for (int b = 0; b < batch; ++b) {
    size_t n = 0;
    for (int j = 0; j < k; ++j) {
      size_t row = (size_t)b * k + j;
      double beam = (double)beam_scores[row];
      if (finished && finished[row]) {
        cand[n].s = beam;
        cand[n].flat = (int64_t)j * vocab + eos_id;
        ++n;
        if (out_lse) out_lse[row] = NAN;
        continue;
      }
      orc_row_values(logits, dtype, bias, row, vocab, x);
      double lse = orc_log_sum_exp(x, vocab);
      if (out_lse) out_lse[row] = lse;
      int dead = (lse == -INFINITY) || (beam == -INFINITY);
      for (int v = 0; v < vocab; ++v) {
        cand[n].s = dead ? -INFINITY : (beam + x[v]) - lse;
        cand[n].flat = (int64_t)j * vocab + v;
        ++n;
      }
    }
    qsort(cand, n, sizeof(orc_cand), orc_cmp_cand);
    for (int r = 0; r < m_out; ++r) {
      size_t o = (size_t)b * m_out + r;
      if ((size_t)r < n) {
        int parent = (int)(cand[r].flat / vocab);
        int token = (int)(cand[r].flat % vocab);
        out_token[o] = token;
        out_parent[o] = parent;
        out_score[o] = cand[r].s;
        int fin = finished ? (finished[(size_t)b * k + parent] != 0) : 0;
        out_finished[o] = (uint8_t)(fin || token == eos_id);
      } else {
        out_token[o] = -1;
        out_parent[o] = -1;
        out_score[o] = NAN;
        out_finished[o] = 0;
      }
    }
  }
  free(cand);
  free(x);
  return 0;
}

/*
 * The step before the beam step: the decoder's output projection, whose result is
 * the logit tensor the article's first traversal reads.  logits = hidden . weight^T:
 *   x[r, v] = sum_d hidden[r, d] * weight[v, d]
 * hidden [rows, dim] and weight [vocab, dim] (the projection matrix, one row per token)
 * hold dtype 0 f32, 1 f16 bits or 2 bf16 bits; out [rows, vocab] is double.  The
 * inputs decode exactly to double, their products are exact in double (at most 48
 * significant bits), and the dim products are summed in order d = 0, 1, ...
 * Returns 0, or -1 on bad arguments.
 */
int oracle_logits(const void* hidden, const void* weight, int dtype, int rows, int vocab, int dim,
                  double* out) {
  if (!hidden || !weight || !out || rows < 0 || vocab < 0 || dim < 0) return -1;
  if (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16) return -1;
  double* h = (double*)malloc(((size_t)dim + 1) * sizeof(double));
  if (!h) return -2;
  for (int r = 0; r < rows; ++r) {
    for (int d = 0; d < dim; ++d) h[d] = orc_logit(hidden, dtype, (size_t)r * dim + d);
    for (int v = 0; v < vocab; ++v) {
      double acc = 0.0;
      for (int d = 0; d < dim; ++d) acc += h[d] * orc_logit(weight, dtype, (size_t)v * dim + d);
      out[(size_t)r * vocab + v] = acc;
    }
  }
  free(h);
  return 0;
}

/* k-th largest (1-based k) of n doubles by selection on a copy. */
static int orc_cmp_desc(const void* pa, const void* pb) {
  double a = *(const double*)pa, b = *(const double*)pb;
  return (a > b) ? -1 : (a < b);
}

/*
 * Diagnostic restatement of the first traversal (not an output of the step).
 * For every row: split the vocab into `groups` groups, group g = {v : v mod groups == g}
 * (the article's k groups when groups == k), take each group's max, and let
 * R = the k-th largest of those group maxima (= their min when groups == k).
 * kth = the true k-th largest x of the row; ncand = #{v : x_v >= R}.
 * R is -inf when fewer than k groups are non-empty.
 */
int oracle_rtopk_stats(const void* logits, int dtype, const float* bias, int rows, int k, int vocab,
                       int groups, double* out_R, double* out_kth, int64_t* out_ncand) {
  if (!logits || !out_R || !out_kth || !out_ncand) return -1;
  if (rows < 0 || k < 1 || vocab < k || groups < k) return -1;
  double* x = (double*)malloc((size_t)vocab * sizeof(double));
  double* srt = (double*)malloc((size_t)vocab * sizeof(double));
  double* gm = (double*)malloc((size_t)groups * sizeof(double));
  if (!x || !srt || !gm) {
    free(x);
    free(srt);
    free(gm);
    return -2;
  }
  for (int r = 0; r < rows; ++r) {
    orc_row_values(logits, dtype, bias, (size_t)r, vocab, x);
    for (int g = 0; g < groups; ++g) gm[g] = -INFINITY;
    for (int v = 0; v < vocab; ++v) {
      int g = v % groups;
      if (x[v] > gm[g]) gm[g] = x[v];
    }
    qsort(gm, (size_t)groups, sizeof(double), orc_cmp_desc);
    double R = gm[k - 1];
    memcpy(srt, x, (size_t)vocab * sizeof(double));
    qsort(srt, (size_t)vocab, sizeof(double), orc_cmp_desc);
    int64_t c = 0;
    for (int v = 0; v < vocab; ++v) c += (x[v] >= R);
    out_R[r] = R;
    out_kth[r] = srt[k - 1];
    out_ncand[r] = c;
  }
  free(x);
  free(srt);
  free(gm);
  return 0;
}

/*
 * Beam-cache refresh: dst[l, b*k+j, h, p, :] = src[l, b*k+parent[b,j], h, p, :]
 * for p < len; positions p >= len of dst are not written.
 * Layout [layers, batch*k, heads, max_len, head_dim], elem_bytes per element.
 * Returns -1 on bad arguments (including a parent outside [0, k)).
 */
int oracle_cache_reorder(const void* src, void* dst, int elem_bytes, const int32_t* parent,
                         int layers, int batch, int k, int heads, int max_len, int len,
                         int head_dim) {
  if (!src || !dst || !parent || elem_bytes < 1) return -1;
  if (layers < 0 || batch < 0 || k < 1 || heads < 0 || max_len < 0 || len < 0 || len > max_len ||
      head_dim < 0)
    return -1;
  for (int r = 0; r < batch * k; ++r)
    if (parent[r] < 0 || parent[r] >= k) return -1;
  const unsigned char* s = (const unsigned char*)src;
  unsigned char* d = (unsigned char*)dst;
  size_t rows = (size_t)batch * k;
  for (int l = 0; l < layers; ++l)
    for (int b = 0; b < batch; ++b)
      for (int j = 0; j < k; ++j) {
        size_t drow = (size_t)b * k + j;
        size_t srow = (size_t)b * k + parent[drow];
        for (int h = 0; h < heads; ++h)
          for (int p = 0; p < len; ++p)
            for (int e = 0; e < head_dim; ++e) {
              size_t di = ((((size_t)l * rows + drow) * heads + h) * max_len + p) * head_dim + e;
              size_t si = ((((size_t)l * rows + srow) * heads + h) * max_len + p) * head_dim + e;
              memcpy(d + di * elem_bytes, s + si * elem_bytes, (size_t)elem_bytes);
            }
      }
  return 0;
}

/*
 * End of a search: the token sequence of every final beam, read back through the
 * per-step parent pointers (the step after the decode loop; the article's decoding
 * keeps a beam's history by parent beam, which the cache refresh also follows).
 *
 * token_hist, parent_hist [steps, batch, k]: the outputs of decode steps 1..steps
 * (step t's beam j continued beam parent_hist[t, b, j] of step t-1 and appended
 * token_hist[t, b, j]).  For final beam j of batch b:
 *   c_{steps-1} = j,  seq[b, j, t] = token_hist[t, b, c_t],  c_{t-1} = parent_hist[t, b, c_t].
 * len[b, j] = 1 + the first t with seq[b, j, t] == eos_id, or steps when there is none.
 * Returns -1 on bad arguments (including a parent outside [0, k) on a walked path).
 */
int oracle_backtrack(const int32_t* token_hist, const int32_t* parent_hist, int steps, int batch, int k,
                     int eos_id, int32_t* out_seq, int32_t* out_len) {
  if (steps < 0 || batch < 0 || k < 1) return -1;
  if (steps == 0 || batch == 0) return 0;
  if (!token_hist || !parent_hist || !out_seq || !out_len) return -1;
  for (int b = 0; b < batch; ++b)
    for (int j = 0; j < k; ++j) {
      int c = j;
      for (int t = steps - 1; t >= 0; --t) {
        if (c < 0 || c >= k) return -1;
        size_t h = ((size_t)t * batch + b) * k + c;
        out_seq[((size_t)b * k + j) * steps + t] = token_hist[h];
        c = parent_hist[h];
      }
      int len = steps;
      for (int t = 0; t < steps; ++t)
        if (out_seq[((size_t)b * k + j) * steps + t] == eos_id) {
          len = t + 1;
          break;
        }
      out_len[(size_t)b * k + j] = len;
    }
  return 0;
}

/*
 * Sampling decoding (the article's other decoding mode next to beam search): one row of
 * logits per sequence, x = logit + bias.  The top_k tokens by x (ties: smaller token id
 * first) carry probabilities proportional to exp(x), renormalised over those top_k; with
 * top_p < 1 only the shortest prefix of them (in that order) whose cumulative probability
 * reaches top_p is kept and renormalised again.  The token drawn for uniform u in [0, 1)
 * is the first candidate whose cumulative probability exceeds u (inverse CDF).
 * out_logprob = x(token) - log sum_v exp(x_v) over the whole row.
 * out_margin (may be NULL) = the smaller of the distance of u from the nearest cumulative
 * boundary of the kept set and, with top_p < 1, the distance of top_p from the nearest
 * cumulative boundary of the top_k (a draw or a cut this close to a boundary may
 * legitimately round either way).
 * Returns -1 on bad arguments.
 */
int oracle_sample(const void* logits, int dtype, const float* bias, int rows, int vocab, int top_k,
                  double top_p, const double* u, int32_t* out_token, double* out_logprob,
                  double* out_margin) {
  if (!logits || !u || !out_token || !out_logprob) return -1;
  if (rows < 0 || vocab < 1 || top_k < 1 || top_k > vocab || !(top_p > 0.0) || top_p > 1.0) return -1;
  double* x = (double*)malloc(sizeof(double) * (size_t)vocab);
  orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)vocab);
  double* cum = (double*)malloc(sizeof(double) * (size_t)top_k);
  if (!x || !c || !cum) {
    free(x);
    free(c);
    free(cum);
    return -1;
  }
  for (int r = 0; r < rows; ++r) {
    orc_row_values(logits, dtype, bias, (size_t)r, vocab, x);
    const double lse = orc_log_sum_exp(x, vocab);
    for (int v = 0; v < vocab; ++v) {
      c[v].s = x[v];
      c[v].flat = v;
    }
    qsort(c, (size_t)vocab, sizeof(orc_cand), orc_cmp_cand);  /* x descending, token ascending */
    const double x0 = c[0].s;
    double acc = 0.0;
    for (int i = 0; i < top_k; ++i) {
      acc += exp(c[i].s - x0);
      cum[i] = acc;
    }
    int m = top_k;  /* kept prefix */
    if (top_p < 1.0) {
      for (int i = 0; i < top_k; ++i)
        if (cum[i] >= top_p * cum[top_k - 1]) {
          m = i + 1;
          break;
        }
    }
    const double target = u[r] * cum[m - 1];
    int pick = m - 1;
    for (int i = 0; i < m; ++i)
      if (cum[i] > target) {
        pick = i;
        break;
      }
    out_token[r] = c[pick].flat;
    out_logprob[r] = c[pick].s - lse;
    if (out_margin) {
      double mg = 1.0;
      for (int i = 0; i < m - 1; ++i) {
        const double d = fabs(cum[i] / cum[m - 1] - u[r]);
        if (d < mg) mg = d;
      }
      if (top_p < 1.0)
        for (int i = 0; i < top_k; ++i) {
          const double d = fabs(cum[i] / cum[top_k - 1] - top_p);
          if (d < mg) mg = d;
        }
      out_margin[r] = mg;
    }
  }
  free(x);
  free(c);
  free(cum);
  return 0;
}

/*
 * Beam-cache refresh in place: cache[l, b*k+j, h, p, :] becomes the old
 * cache[l, b*k+parent[b,j], h, p, :] for p < len (every row reads the state before the
 * step, whatever order rows are written in); positions p >= len keep their own content.
 * Written as the definition: a full copy of the old cache, then the gather from it.
 * Returns -1 on bad arguments (including a parent outside [0, k)), -2 on allocation failure.
 */
int oracle_cache_refresh_inplace(void* cache, int elem_bytes, const int32_t* parent, int layers, int batch, int k,
                                 int heads, int max_len, int len, int head_dim) {
  if (!cache || !parent || elem_bytes < 1) return -1;
  if (layers < 0 || batch < 0 || k < 1 || heads < 0 || max_len < 0 || len < 0 || len > max_len || head_dim < 0)
    return -1;
  const size_t total = (size_t)layers * batch * k * heads * max_len * head_dim * (size_t)elem_bytes;
  void* old = malloc(total ? total : 1);
  if (!old) return -2;
  memcpy(old, cache, total);
  const int rc = oracle_cache_reorder(old, cache, elem_bytes, parent, layers, batch, k, heads, max_len, len, head_dim);
  free(old);
  return rc;
}
