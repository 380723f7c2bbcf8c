/*
 * spec_oracle.c -- plain, slow, fp64 CPU oracle for the batched
 * speculative-decoding verify step over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may call it. It shares no code, header,
 * table or constant with the CUDA library; it reads the same seeded inputs.
 *
 * What it follows (pages on speculative decoding, cited by title/section):
 *  - "Speculative decoding and continuous batching in practice", sec. 1.2:
 *    the target scores gamma+1 positions in one pass; each draft token is
 *    accepted with probability min(1, p(x)/q(x)).
 *  - "Speculative decoding principles and a vLLM production setup", sec. 2.1
 *    and 2.2: positions are tested in order, the first rejection drops the
 *    rest of the draft, and the replacement is drawn from norm(max(0, p - q)).
 *  - "LLM serving: speculative decoding and PagedAttention memory management",
 *    PagedAttention section: each sequence's logical KV blocks map to physical
 *    blocks through its block table.
 *  - "LLM inference optimisation: speculative decoding and dynamic batching",
 *    engineering section: greedy verification keeps the drafts up to the
 *    first mismatch with the target and restarts from the mismatching position.
 *  - same vLLM page, sec. 3.2 and 5.2: tree attention; each tree node sees the
 *    prefix and its ancestors.
 *
 * Readings where the pages are silent (each repeated where it is used):
 *  - accept iff u < min(1, p/q), u in [0, 1); q(x) == 0 gives ratio +inf;
 *  - inverse CDF: the smallest index whose inclusive prefix sum strictly
 *    exceeds u * (total mass); zero-mass tokens are never chosen;
 *  - residual mass zero: draw from p at the rejected position instead;
 *  - argmax ties go to the lowest token index.
 *
 * Precision: every sum, product, exp and division is in IEEE fp64, in plain
 * left-to-right loops (compile without -ffast-math). bf16 inputs (uint16 bit
 * patterns) are widened exactly.
 *
 * Threads (OpenMP, when built with it): attention runs its (sequence, KV head)
 * pairs, the chain sampler its sequences, as independent tasks; every result is
 * computed by one task in the same order as on one thread, so the values do
 * not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SO_OK 0
#define SO_ERR_ARG (-1)
#define SO_ERR_BLOCK (-2)
#define SO_ERR_TOKEN (-3)
#define SO_ERR_NONFINITE (-4)
#define SO_ERR_NOMEM (-5)

#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads of the parallel loops below (1: one thread). Returns the count in use. */
int so_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* dtype codes: 0 = bf16 stored as uint16 bit patterns, 1 = fp32 */
static double widen(const void *base, int dtype, size_t i) {
  if (dtype == 0) {
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float *)base)[i];
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                */
/* ------------------------------------------------------------------------ */

/* Whether query row i (0-based among the sequence's n new rows) may attend to
 * key position t of a sequence with c committed tokens. Committed tokens are
 * always visible. New row j = t - c is visible when j <= i (causal) or when
 * bit j of the row's tree mask is set (tree: ancestors and itself). */
static int visible(int t, int c, int i, int mask_kind, const uint64_t *tree_mask_row) {
  if (t < c) return 1;
  int j = t - c;
  if (mask_kind == 0) return j <= i;
  if (j >= 64) return 0;
  return (int)((*tree_mask_row >> j) & 1u);
}

/*
 * Dense masked attention over one sequence's contiguous keys and values.
 *   k, v : [L, hkv, d] fp64, positions 0..L-1 (c committed + n new)
 *   q    : [n, hq, d] fp64
 *   out  : [n, hq, d] fp64
 * Query head h reads KV head h / (hq / hkv) (grouped-query attention).
 * s_t = scale * <q, k_t>; o = sum_t softmax(s)_t v_t over visible t, with the
 * maximum subtracted before exp. A row that sees no key gets o = 0.
 */
int so_dense_attention(int L, int c, int n, int hq, int hkv, int d, const double *k, const double *v,
                       const double *q, int mask_kind, const uint64_t *tree_mask, double scale,
                       double *out) {
  if (L != c + n || hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0) return SO_ERR_ARG;
  int group = hq / hkv;
  double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  char *vis = (char *)malloc((size_t)(L > 0 ? L : 1));
  if (!s || !vis) {
    free(s);
    free(vis);
    return SO_ERR_NOMEM;
  }
  for (int i = 0; i < n; ++i) {
    const uint64_t *mrow = tree_mask ? &tree_mask[i] : NULL;
    for (int h = 0; h < hq; ++h) {
      int kh = h / group;
      const double *qr = &q[((size_t)i * hq + h) * d];
      double mx = -INFINITY;
      int any = 0;
      for (int t = 0; t < L; ++t) {
        vis[t] = (char)visible(t, c, i, mask_kind, mrow);
        if (!vis[t]) continue;
        const double *kr = &k[((size_t)t * hkv + kh) * d];
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += qr[e] * kr[e];
        s[t] = dot * scale;
        if (!any || s[t] > mx) mx = s[t];
        any = 1;
      }
      double *o = &out[((size_t)i * hq + h) * d];
      for (int e = 0; e < d; ++e) o[e] = 0.0;
      if (!any) continue;
      double denom = 0.0;
      for (int t = 0; t < L; ++t) {
        if (!vis[t]) continue;
        double w = exp(s[t] - mx);
        s[t] = w;
        denom += w;
      }
      for (int t = 0; t < L; ++t) {
        if (!vis[t]) continue;
        const double *vr = &v[((size_t)t * hkv + kh) * d];
        for (int e = 0; e < d; ++e) o[e] += s[t] * vr[e];
      }
      for (int e = 0; e < d; ++e) o[e] /= denom;
    }
  }
  free(s);
  free(vis);
  return SO_OK;
}

/*
 * Paged attention: gather each selected sequence's keys and values through its
 * block table (position t lives in physical block block_table[b][t / bs], slot
 * t % bs; pools are [num_blocks, hkv, bs, d]), then run the dense definition.
 *   ctx_lens[b] = c_b committed tokens; the sequence's n_b = cu_q[b+1]-cu_q[b]
 *   new rows occupy positions c_b .. c_b+n_b-1 (already appended).
 *   q [T_q, hq, d]; out [T_q, hq, d] fp64 (rows of unselected sequences untouched).
 *   seqs: the sequences to compute (n_seqs of them), or NULL for all.
 */
int so_paged_attention(int batch, int hq, int hkv, int d, int bs, int max_blocks, int num_blocks,
                       const int32_t *ctx_lens, const int32_t *cu_q, const int32_t *block_table,
                       const void *k_pool, const void *v_pool, int kv_dtype, const void *q, int q_dtype,
                       int mask_kind, const uint64_t *tree_mask, double scale, const int32_t *seqs,
                       int n_seqs, double *out) {
  if (batch < 0 || bs <= 0 || hkv <= 0 || hq % hkv != 0) return SO_ERR_ARG;
  int count = seqs ? n_seqs : batch;
  for (int si = 0; si < count; ++si) {  /* lengths and table room first */
    int b = seqs ? seqs[si] : si;
    if (b < 0 || b >= batch) return SO_ERR_ARG;
    int c = ctx_lens[b], n = cu_q[b + 1] - cu_q[b];
    if (c < 0 || n < 0) return SO_ERR_ARG;
    if ((c + n + bs - 1) / bs > max_blocks) return SO_ERR_BLOCK;
  }
  const int group = hq / hkv;
  const long ntask = (long)count * hkv;
  int rc_all = SO_OK;
  /* one task per (sequence, KV head): its keys and values, its `group` query heads */
#pragma omp parallel for schedule(dynamic, 1)
  for (long task = 0; task < ntask; ++task) {
    int si = (int)(task / hkv), kh = (int)(task % hkv);
    int b = seqs ? seqs[si] : si;
    int c = ctx_lens[b];
    int n = cu_q[b + 1] - cu_q[b];
    int L = c + n;
    double *kd = (double *)malloc(sizeof(double) * ((size_t)L * d + 1));
    double *vd = (double *)malloc(sizeof(double) * ((size_t)L * d + 1));
    double *qd = (double *)malloc(sizeof(double) * ((size_t)n * group * d + 1));
    double *od = (double *)malloc(sizeof(double) * ((size_t)n * group * d + 1));
    int rc = (kd && vd && qd && od) ? SO_OK : SO_ERR_NOMEM;
    for (int t = 0; t < L && rc == SO_OK; ++t) {
      int blk = block_table[(size_t)b * max_blocks + t / bs];
      if (blk < 0 || blk >= num_blocks) {
        rc = SO_ERR_BLOCK;
        break;
      }
      int slot = t % bs;
      for (int e = 0; e < d; ++e) {
        size_t src = (((size_t)blk * hkv + kh) * bs + slot) * d + e;
        kd[(size_t)t * d + e] = widen(k_pool, kv_dtype, src);
        vd[(size_t)t * d + e] = widen(v_pool, kv_dtype, src);
      }
    }
    if (rc == SO_OK) {
      size_t row0 = (size_t)cu_q[b];
      for (int i = 0; i < n; ++i)
        for (int g = 0; g < group; ++g)
          for (int e = 0; e < d; ++e)
            qd[((size_t)i * group + g) * d + e] =
                widen(q, q_dtype, ((row0 + i) * hq + (size_t)kh * group + g) * d + e);
      rc = so_dense_attention(L, c, n, group, 1, d, kd, vd, qd, mask_kind, tree_mask ? &tree_mask[row0] : NULL,
                              scale, od);
      if (rc == SO_OK)
        for (int i = 0; i < n; ++i)
          memcpy(&out[((row0 + i) * hq + (size_t)kh * group) * d], &od[(size_t)i * group * d],
                 sizeof(double) * (size_t)group * d);
    }
    free(kd); free(vd); free(qd); free(od);
    if (rc != SO_OK) {
#pragma omp critical(so_rc)
      rc_all = rc;
    }
  }
  return rc_all;
}


/* ------------------------------------------------------------------------ */
/* Sampler                                                                  */
/* ------------------------------------------------------------------------ */

/* p_v = exp((l_v - max l) / T) / sum_w exp((l_w - max l) / T), fp64. */
static int softmax_row(const void *logits, int dtype, size_t row, int V, double T, double *p) {
  double mx = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = widen(logits, dtype, row * (size_t)V + v);
    if (isnan(x) || x == INFINITY) return SO_ERR_NONFINITE;
    p[v] = x;
    if (x > mx) mx = x;
  }
  if (mx == -INFINITY) return SO_ERR_NONFINITE;
  double z = 0.0;
  for (int v = 0; v < V; ++v) {
    p[v] = exp((p[v] - mx) / T);
    z += p[v];
  }
  for (int v = 0; v < V; ++v) p[v] /= z;
  return SO_OK;
}

/* argmax with the lowest index on ties */
static int argmax_row(const void *logits, int dtype, size_t row, int V, int *idx) {
  double best = 0.0;
  int bi = -1;
  for (int v = 0; v < V; ++v) {
    double x = widen(logits, dtype, row * (size_t)V + v);
    if (isnan(x)) return SO_ERR_NONFINITE;
    if (bi < 0 || x > best) {
      best = x;
      bi = v;
    }
  }
  *idx = bi;
  return SO_OK;
}

/* Inverse CDF over non-negative weights w (total mass `total`): the smallest v
 * whose inclusive prefix sum strictly exceeds `target`. `*margin` receives the
 * distance of target/total from the chosen interval's edges, on the
 * normalised CDF. If rounding leaves no crossing, the last v with w_v > 0 is
 * taken and the margin is 0. */
static int inverse_cdf(const double *w, int V, double target, double total, double *margin) {
  double cum = 0.0;
  int last_pos = -1;
  for (int v = 0; v < V; ++v) {
    double prev = cum;
    cum += w[v];
    if (w[v] > 0.0) last_pos = v;
    if (cum > target) {
      double lo = (target - prev) / total, hi = (cum - target) / total;
      *margin = lo < hi ? lo : hi;
      return v;
    }
  }
  *margin = 0.0;
  return last_pos;
}

/*
 * Lossless verification of chain drafts (temperature > 0), or greedy
 * verification (temperature == 0).
 *
 * Sequence b has n = cu_q[b+1]-cu_q[b] target rows and K = n-1 draft tokens.
 * Target row cu_q[b]+i holds the logits p_{i+1} of the position that draft
 * token x_{i+1} fills (row 0 scores x_1, row K is the bonus position). Draft
 * row / token / accept uniform of x_{i+1} sit at index cu_q[b]-b+i.
 *
 * T > 0:  p = softmax(l_t / T), q = softmax(l_d / T). For i = 0..K-1 accept
 *   x iff u_acc < min(1, p(x)/q(x)); a = the first rejected i, or K.
 *   a < K: y = inverse CDF of r = max(0, p_a - q_a) at u_res * sum(r);
 *          if sum(r) == 0, y = inverse CDF of p_a at u_res (fallback[b] = 1).
 *   a = K: y = inverse CDF of p_K at u_res.
 * T == 0: accept while x equals argmax of the target row; y = argmax row a.
 *
 * Outputs: accept_cnt[b] = a; out_tok[b][0..a] = x_1..x_a, y (rest -1);
 * num_out[b] = a + 1. margin[b] = the smallest distance, over every
 * comparison that decided b's outcome, between the uniform and the
 * threshold it was compared with (|u - min(1,p/q)|, and the CDF crossing);
 * +inf for greedy.
 */
/* One sequence of so_rejection_sample; p and qd are scratch of `vocab` doubles. */
static int rejection_one(int b, int vocab, const int32_t *cu_q, const void *tgt, const void *drf, int dtype,
                         const int32_t *draft_tok, const float *u_acc, const float *u_res, double temperature,
                         int max_q, int32_t *accept_cnt, int32_t *out_tok, int32_t *num_out, double *margin,
                         int32_t *fallback, double *p, double *qd) {
  int rc = SO_OK;
  int n = cu_q[b + 1] - cu_q[b];
  int K = n - 1;
  if (n < 1 || n > max_q) return SO_ERR_ARG;
  size_t t0 = (size_t)cu_q[b];
  size_t d0 = (size_t)cu_q[b] - (size_t)b;
  for (int j = 0; j < max_q; ++j) out_tok[(size_t)b * max_q + j] = -1;
  double marg = INFINITY;
  int fb = 0;
  int a = K, y = -1;
  if (temperature == 0.0) {
    for (int i = 0; i < K; ++i) {
      int am;
      if ((rc = argmax_row(tgt, dtype, t0 + i, vocab, &am)) != SO_OK) return rc;
      int x = draft_tok[d0 + i];
      if (x != am) {
        a = i;
        y = am;
        break;
      }
    }
    if (a == K && (rc = argmax_row(tgt, dtype, t0 + K, vocab, &y)) != SO_OK) return rc;
  } else {
    for (int i = 0; i < K; ++i) {
      int x = draft_tok[d0 + i];
      if (x < 0 || x >= vocab) return SO_ERR_TOKEN;
      if ((rc = softmax_row(tgt, dtype, t0 + i, vocab, temperature, p)) != SO_OK) return rc;
      if ((rc = softmax_row(drf, dtype, d0 + i, vocab, temperature, qd)) != SO_OK) return rc;
      double ratio = qd[x] > 0.0 ? p[x] / qd[x] : INFINITY;
      double thr = ratio < 1.0 ? ratio : 1.0;
      double u = (double)u_acc[d0 + i];
      double dist = fabs(u - thr);
      if (dist < marg) marg = dist;
      if (!(u < thr)) {
        a = i;
        break;
      }
    }
    double m2 = INFINITY;
    double ur = (double)u_res[b];
    if (a < K) {
      /* p and qd still hold row a */
      double S = 0.0;
      for (int v = 0; v < vocab; ++v) {
        double r = p[v] - qd[v];
        qd[v] = r > 0.0 ? r : 0.0;
        S += qd[v];
      }
      if (S > 0.0) {
        y = inverse_cdf(qd, vocab, ur * S, S, &m2);
      } else {
        fb = 1;
        y = inverse_cdf(p, vocab, ur, 1.0, &m2);
      }
    } else {
      if ((rc = softmax_row(tgt, dtype, t0 + K, vocab, temperature, p)) != SO_OK) return rc;
      y = inverse_cdf(p, vocab, ur, 1.0, &m2);
    }
    if (m2 < marg) marg = m2;
  }
  accept_cnt[b] = a;
  for (int j = 0; j < a; ++j) out_tok[(size_t)b * max_q + j] = draft_tok[d0 + j];
  out_tok[(size_t)b * max_q + a] = y;
  num_out[b] = a + 1;
  if (margin) margin[b] = marg;
  if (fallback) fallback[b] = fb;
  return SO_OK;
}

int so_rejection_sample(int batch, int vocab, const int32_t *cu_q, const void *tgt, const void *drf,
                        int dtype, const int32_t *draft_tok, const float *u_acc, const float *u_res,
                        double temperature, int max_q, int32_t *accept_cnt, int32_t *out_tok,
                        int32_t *num_out, double *margin, int32_t *fallback) {
  if (batch < 0 || vocab <= 0 || max_q <= 0) return SO_ERR_ARG;
  int rc_all = SO_OK;
#pragma omp parallel
  {
    double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
    double *qd = (double *)malloc(sizeof(double) * (size_t)vocab);
#pragma omp for schedule(dynamic, 1)
    for (int b = 0; b < batch; ++b) {
      int rc = (p && qd) ? rejection_one(b, vocab, cu_q, tgt, drf, dtype, draft_tok, u_acc, u_res, temperature,
                                         max_q, accept_cnt, out_tok, num_out, margin, fallback, p, qd)
                         : SO_ERR_NOMEM;
      if (rc != SO_OK) {
#pragma omp critical(so_rc)
        rc_all = rc;
      }
    }
    free(p);
    free(qd);
  }
  return rc_all;
}

/*
 * Greedy verification of a draft tree. Sequence b has n rows: row 0 is the
 * root (last emitted token), rows 1..n-1 are tree nodes with parent row
 * parent[cu_q[b]+j] (-1 for the root) and token node_tok[cu_q[b]-b+j-1].
 * Starting at the root: while some child of the current node carries the
 * argmax token of the current node's target row, move to that child (the
 * lowest such row). y = argmax of the final node's row.
 * Outputs: accept_cnt[b] = path length a; path_nodes[b][0..a-1] = the rows of
 * the accepted nodes (rest -1); out_tok[b][0..a] = their tokens then y;
 * num_out[b] = a + 1.
 */
int so_tree_greedy(int batch, int vocab, const int32_t *cu_q, const void *tgt, int dtype,
                   const int32_t *node_tok, const int32_t *parent, int max_q, int32_t *accept_cnt,
                   int32_t *path_nodes, int32_t *out_tok, int32_t *num_out) {
  if (batch < 0 || vocab <= 0 || max_q <= 0) return SO_ERR_ARG;
  for (int b = 0; b < batch; ++b) {
    int n = cu_q[b + 1] - cu_q[b];
    if (n < 1 || n > max_q) return SO_ERR_ARG;
    size_t t0 = (size_t)cu_q[b];
    size_t d0 = (size_t)cu_q[b] - (size_t)b;
    for (int j = 0; j < max_q; ++j) {
      out_tok[(size_t)b * max_q + j] = -1;
      path_nodes[(size_t)b * max_q + j] = -1;
    }
    int cur = 0, a = 0, am = -1;
    for (;;) {
      int rc = argmax_row(tgt, dtype, t0 + cur, vocab, &am);
      if (rc != SO_OK) return rc;
      int next = -1;
      for (int j = 1; j < n; ++j)
        if (parent[t0 + j] == cur && node_tok[d0 + j - 1] == am) {
          next = j;
          break;
        }
      if (next < 0) break;
      path_nodes[(size_t)b * max_q + a] = next;
      out_tok[(size_t)b * max_q + a] = am;
      ++a;
      cur = next;
    }
    out_tok[(size_t)b * max_q + a] = am;
    accept_cnt[b] = a;
    num_out[b] = a + 1;
  }
  return SO_OK;
}

/*
 * Lossless verification of a draft tree at temperature T > 0.
 *
 * The pages fix only the greedy tree rule; the reading taken: a node's
 * children carry distinct candidate tokens picked without sampling (the top-k
 * of the draft at that node), so each child is a proposal that puts all its
 * mass on its token. The rejection rule with such a proposal accepts x with
 * probability p(x), and on rejection leaves the residual p with x's mass
 * removed, renormalised. Walking from the root: at the current node v (target
 * distribution p_v = softmax(row v / T)), its children are tried in row order;
 * child c with token x is accepted iff u_acc[c] < p'(x), where p' is p_v with
 * the tokens of the siblings rejected before it removed and renormalised (0 if
 * x itself was removed); the first accepted child becomes the current node.
 * When no child is accepted (or v has none), y is drawn by inverse CDF with
 * u_res from p' (p_v without the rejected tokens); if they held all of p_v's
 * mass, from p_v itself (fallback[b] = 1). Each emitted token is distributed
 * as the target's p at its position.
 *
 * Node j >= 1 of sequence b: row cu_q[b]+j, parent row parent[cu_q[b]+j],
 * token node_tok[cu_q[b]-b+j-1], accept uniform u_acc[cu_q[b]-b+j-1].
 * Outputs as so_tree_greedy; margin[b] = the smallest distance between a
 * uniform and the threshold it was compared with (u_acc against p'(x), and the
 * CDF crossing of the draw).
 */
int so_tree_sample(int batch, int vocab, const int32_t *cu_q, const void *tgt, int dtype, const int32_t *node_tok,
                   const int32_t *parent, const float *u_acc, const float *u_res, double temperature, int max_q,
                   int32_t *accept_cnt, int32_t *path_nodes, int32_t *out_tok, int32_t *num_out, double *margin,
                   int32_t *fallback) {
  if (batch < 0 || vocab <= 0 || max_q <= 0 || !(temperature > 0.0)) return SO_ERR_ARG;
  double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
  double *w = (double *)malloc(sizeof(double) * (size_t)vocab);
  if (!p || !w) {
    free(p);
    free(w);
    return SO_ERR_NOMEM;
  }
  int rc = SO_OK;
  for (int b = 0; b < batch && rc == SO_OK; ++b) {
    int n = cu_q[b + 1] - cu_q[b];
    if (n < 1 || n > max_q) {
      rc = SO_ERR_ARG;
      break;
    }
    size_t t0 = (size_t)cu_q[b];
    size_t d0 = (size_t)cu_q[b] - (size_t)b;
    for (int j = 0; j < max_q; ++j) {
      out_tok[(size_t)b * max_q + j] = -1;
      path_nodes[(size_t)b * max_q + j] = -1;
    }
    double marg = INFINITY;
    int cur = 0, a = 0, y = -1, fb = 0;
    for (;;) {
      if ((rc = softmax_row(tgt, dtype, t0 + cur, vocab, temperature, p)) != SO_OK) break;
      for (int v = 0; v < vocab; ++v) w[v] = p[v];  /* p' before normalisation: removed tokens get 0 */
      double removed = 0.0;
      int next = -1;
      for (int j = 1; j < n && next < 0; ++j) {
        if (parent[t0 + j] != cur) continue;
        int x = node_tok[d0 + j - 1];
        if (x < 0 || x >= vocab) {
          rc = SO_ERR_TOKEN;
          break;
        }
        double thr = removed < 1.0 ? w[x] / (1.0 - removed) : 0.0;
        double u = (double)u_acc[d0 + j - 1];
        double dist = fabs(u - thr);
        if (dist < marg) marg = dist;
        if (u < thr) {
          next = j;
        } else {
          removed += w[x];
          w[x] = 0.0;
        }
      }
      if (rc != SO_OK) break;
      if (next < 0) {
        double S = 0.0, m2 = INFINITY;
        for (int v = 0; v < vocab; ++v) S += w[v];
        double ur = (double)u_res[b];
        if (S > 0.0) {
          y = inverse_cdf(w, vocab, ur * S, S, &m2);
        } else {
          fb = 1;
          y = inverse_cdf(p, vocab, ur, 1.0, &m2);
        }
        if (m2 < marg) marg = m2;
        break;
      }
      path_nodes[(size_t)b * max_q + a] = next;
      out_tok[(size_t)b * max_q + a] = node_tok[d0 + next - 1];
      ++a;
      cur = next;
    }
    if (rc != SO_OK) break;
    out_tok[(size_t)b * max_q + a] = y;
    accept_cnt[b] = a;
    num_out[b] = a + 1;
    if (margin) margin[b] = marg;
    if (fallback) fallback[b] = fb;
  }
  free(p);
  free(w);
  return rc;
}
