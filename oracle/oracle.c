/*
 * oracle.c — plain CPU oracle for token-tree verification (TEST INFRASTRUCTURE ONLY).
 *
 * This file is the slow, obviously-correct definition of what the GPU library
 * computes.  Only the test-suite, the smoke check and the benchmark's CPU
 * baseline may load it; the library never links it and shares no code with it.
 * All arithmetic is fp64 on the exact input values (bf16 inputs arrive here as
 * the fp32 numbers they represent exactly).  Loops are written in the order the
 * definitions are stated; OpenMP only spreads independent output units over
 * cores and never changes the order of any sum.
 *
 * Sources (titles and sections of the pages this follows):
 *   [SI]  "SpecInfer: Accelerating Generative Large Language Model Serving with
 *          Tree-based Speculative Inference and Verification", §2 Overview
 *          (tree verification: each token's activations see all its ancestors),
 *          §4 Token Tree Verifier (Tree Attention; Tree-Based Parallel Decoding
 *          with topology-aware causal masking over one shared KV cache; Token
 *          Verification with multi-step speculative sampling), §6 Evaluation
 *          (greedy verification emits exactly the incremental-decoding tokens).
 *   [SSD] "Accelerating LLM Inference with Staged Speculative Decoding", §3
 *          Methods, Implementation (attention split between the KV cache and
 *          the in-batch tree tokens; positions set per tree node).
 *   The multi-step speculative sampling rule itself (accept child x with
 *   probability min(1, P_LLM(x)/P_SSM(x)), else continue from the normalised
 *   residual max(0, P_LLM - P_SSM)) is the statement this library is specified
 *   against; the pages name the method and its guarantee without the formula.
 *
 * Conventions shared with the library (readings of the pages, stated once):
 *   - A request's tree is a parent array in topological order: parent[i] is -1
 *     (a root) or an earlier node (0 <= parent[i] < i).  Anything else is a bad
 *     tree (status 2).  Verification additionally needs exactly one root, node 0.
 *   - Tree node i of request b sits in the KV cache at row prefix_len[b] + i
 *     ([SI] §4: verified and speculated tokens share one cache).
 *   - Query head h reads KV head h / (Hq/Hkv).
 *   - Emitted path: path[0] = 0 (the root, already verified), then accepted
 *     nodes; unused entries are -1.  accept_len = number of accepted non-root
 *     nodes; bonus = the extra token taken at the node where the walk stops.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_TREE 2
#define ORACLE_NONFINITE 6

#define NEAR_TIE_EPS 1e-6

/* ------------------------------------------------------------------------ */
/* Tree structure                                                            */
/* ------------------------------------------------------------------------ */

/* Checks the topological parent-array convention for one request. */
static int tree_is_valid(const int32_t* parent, int32_t n) {
  for (int32_t i = 0; i < n; ++i) {
    if (parent[i] < -1 || parent[i] >= i) return 0;
  }
  return 1;
}

/*
 * Ancestor sets of one request's tree, as a dense n x n 0/1 matrix:
 * anc[i*n + j] = 1 iff node j lies on the root-to-node path of i (i included).
 * depth[i] = number of strict ancestors.  Computed by walking parent links
 * upward from every node ([SI] §2: a node's sequence is its root-to-node path).
 * Returns ORACLE_OK or ORACLE_BAD_TREE.
 */
int oracle_tree_ancestors(const int32_t* parent, int32_t n, uint8_t* anc, int32_t* depth) {
  if (!tree_is_valid(parent, n)) return ORACLE_BAD_TREE;
  memset(anc, 0, (size_t)n * (size_t)n);
  for (int32_t i = 0; i < n; ++i) {
    int32_t d = -1;
    for (int32_t j = i; j != -1; j = parent[j]) {
      anc[(size_t)i * n + j] = 1;
      ++d;
    }
    depth[i] = d;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Tree attention                                                            */
/* ------------------------------------------------------------------------ */

/*
 * Tree attention ([SI] §4 "Tree Attention"; [SSD] §3 Implementation).
 *
 * For request b, node i < n_b, query head h (KV head g = h / (Hq/Hkv)):
 *   key set  J(i) = {0 .. P_b-1}  U  {P_b + a : a on the root-to-i path}
 *   s_j      = scale * sum_d q[i,h,d] * k[b,j,g,d]
 *   out[i,h] = sum_{j in J(i)} exp(s_j - max s) v[b,j,g,:] / sum_{j in J(i)} exp(s_j - max s)
 * i.e. ordinary attention over the token sequence node i stands for.
 *
 * q, out:  [N, Hq, D] row-major (N = node_offsets[B]).
 * k_cache, v_cache: element (b, l, g, d) at b*stride_b + l*stride_l + g*stride_h + d.
 * node_offsets: [B+1]; request b owns rows node_offsets[b] .. node_offsets[b+1]-1.
 * status[b] receives ORACLE_OK, ORACLE_BAD_TREE (outputs of b left zero) or
 * ORACLE_NONFINITE.  Returns the first non-OK status, else ORACLE_OK.
 */
int oracle_tree_attention(const float* q, const float* k_cache, const float* v_cache,
                          int64_t stride_b, int64_t stride_l, int64_t stride_h,
                          const int32_t* prefix_len, const int32_t* node_offsets,
                          const int32_t* parent, int32_t B, int32_t Hq, int32_t Hkv,
                          int32_t D, double scale, double* out, int32_t* status) {
  const int32_t G = Hq / Hkv;
  int rc = ORACLE_OK;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t off = node_offsets[b];
    const int32_t n = node_offsets[b + 1] - off;
    const int32_t P = prefix_len[b];
    const int32_t* par = parent + off;
    status[b] = ORACLE_OK;
    memset(out + (size_t)off * Hq * D, 0, sizeof(double) * (size_t)n * Hq * D);
    if (!tree_is_valid(par, n)) {
      status[b] = ORACLE_BAD_TREE;
      if (rc == ORACLE_OK) rc = ORACLE_BAD_TREE;
      continue;
    }
    int nonfinite = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(| : nonfinite)
    for (int32_t i = 0; i < n; ++i) {
      for (int32_t h = 0; h < Hq; ++h) {
        const int32_t g = h / G;
        /* Key rows of J(i): the prefix, then the root-to-i path in root-first order. */
        int32_t* path_rev = (int32_t*)malloc(sizeof(int32_t) * (size_t)(i + 1));
        int32_t plen = 0;
        for (int32_t a = i; a != -1; a = par[a]) path_rev[plen++] = a;
        const int32_t nkeys = P + plen;
        double* s = (double*)malloc(sizeof(double) * (size_t)nkeys);
        int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)nkeys);
        for (int32_t j = 0; j < P; ++j) row[j] = j;
        for (int32_t t = 0; t < plen; ++t) row[P + t] = (int64_t)P + path_rev[plen - 1 - t];
        free(path_rev);

        const float* qv = q + ((size_t)(off + i) * Hq + h) * D;
        double smax = -INFINITY;
        for (int32_t j = 0; j < nkeys; ++j) {
          const float* kv = k_cache + (int64_t)b * stride_b + row[j] * stride_l + (int64_t)g * stride_h;
          double dot = 0.0;
          for (int32_t d = 0; d < D; ++d) dot += (double)qv[d] * (double)kv[d];
          s[j] = scale * dot;
          if (!isfinite(s[j])) nonfinite = 1;
          if (s[j] > smax) smax = s[j];
        }
        double denom = 0.0;
        for (int32_t j = 0; j < nkeys; ++j) {
          s[j] = exp(s[j] - smax);
          denom += s[j];
        }
        double* o = out + ((size_t)(off + i) * Hq + h) * D;
        for (int32_t j = 0; j < nkeys; ++j) {
          const float* vv = v_cache + (int64_t)b * stride_b + row[j] * stride_l + (int64_t)g * stride_h;
          for (int32_t d = 0; d < D; ++d) o[d] += s[j] * (double)vv[d];
        }
        for (int32_t d = 0; d < D; ++d) {
          o[d] /= denom;
          if (!isfinite(o[d])) nonfinite = 1;
        }
        free(s);
        free(row);
      }
    }
    if (nonfinite) {
      status[b] = ORACLE_NONFINITE;
      if (rc == ORACLE_OK) rc = ORACLE_NONFINITE;
    }
  }
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Verification helpers                                                      */
/* ------------------------------------------------------------------------ */

/* Verification needs exactly one root, node 0. */
static int tree_is_verifiable(const int32_t* parent, int32_t n) {
  if (n < 1 || parent[0] != -1) return 0;
  for (int32_t i = 1; i < n; ++i) {
    if (parent[i] < 0 || parent[i] >= i) return 0;
  }
  return 1;
}

/* 1 iff every entry of the row is finite (the inputs' contract). */
static int row_is_finite(const float* x, int64_t V) {
  for (int64_t t = 0; t < V; ++t) {
    if (!isfinite(x[t])) return 0;
  }
  return 1;
}

/* Index of the first maximum (ties go to the lowest index). */
static int64_t first_argmax(const float* x, int64_t V) {
  int64_t best = 0;
  for (int64_t t = 1; t < V; ++t) {
    if (x[t] > x[best]) best = t;
  }
  return best;
}

static void clear_outputs(int32_t* path, int32_t n, int32_t* accept_len, int32_t* bonus) {
  for (int32_t t = 0; t < n; ++t) path[t] = -1;
  *accept_len = 0;
  *bonus = -1;
}

/* ------------------------------------------------------------------------ */
/* Greedy verification                                                       */
/* ------------------------------------------------------------------------ */

/*
 * Greedy token-tree verification ([SI] §4 Token Tree Verification; §6: the
 * emitted tokens equal incremental decoding's).  logits row u (of the request's
 * rows) is the LLM's next-token score after node u's sequence.
 *   u = 0, path = [0]
 *   repeat: a = argmax logits[u] (lowest index on ties);
 *           c = lowest-index child of u whose token is a; stop if none;
 *           u = c, append c.
 *   bonus = argmax at the stop node.
 * Outputs per request b: path[off_b ..] (local node indices, -1 padded),
 * accept_len[b] = len(path) - 1, bonus[b].  A bad tree gives status 2, path -1,
 * accept_len 0, bonus -1.
 */
int oracle_verify_greedy(const float* logits, int64_t V, const int32_t* tokens,
                         const int32_t* parent, const int32_t* node_offsets, int32_t B,
                         int32_t* path, int32_t* accept_len, int32_t* bonus, int32_t* status) {
  int rc = ORACLE_OK;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t off = node_offsets[b];
    const int32_t n = node_offsets[b + 1] - off;
    const int32_t* par = parent + off;
    const int32_t* tok = tokens + off;
    int32_t* pth = path + off;
    clear_outputs(pth, n, &accept_len[b], &bonus[b]);
    status[b] = ORACLE_OK;
    if (!tree_is_verifiable(par, n)) {
      status[b] = ORACLE_BAD_TREE;
      if (rc == ORACLE_OK) rc = ORACLE_BAD_TREE;
      continue;
    }
    int32_t u = 0, len = 0;
    pth[len++] = 0;
    for (;;) {
      if (!row_is_finite(logits + (size_t)(off + u) * V, V)) {
        status[b] = ORACLE_NONFINITE;
        if (rc == ORACLE_OK) rc = ORACLE_NONFINITE;
      }
      const int64_t a = first_argmax(logits + (size_t)(off + u) * V, V);
      int32_t next = -1;
      for (int32_t c = u + 1; c < n; ++c) {
        if (par[c] == u && tok[c] == a) {
          next = c;
          break;
        }
      }
      if (next < 0) {
        bonus[b] = (int32_t)a;
        break;
      }
      u = next;
      pth[len++] = u;
    }
    accept_len[b] = len - 1;
  }
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Stochastic verification: multi-step speculative sampling                  */
/* ------------------------------------------------------------------------ */

/* p = softmax(x / T) in fp64. */
static void softmax_row(const float* x, int64_t V, double T, double* p) {
  double m = -INFINITY;
  for (int64_t t = 0; t < V; ++t) {
    const double z = (double)x[t] / T;
    if (z > m) m = z;
  }
  double s = 0.0;
  for (int64_t t = 0; t < V; ++t) {
    p[t] = exp((double)x[t] / T - m);
    s += p[t];
  }
  for (int64_t t = 0; t < V; ++t) p[t] /= s;
}

/*
 * Multi-step speculative sampling ([SI] §1 Correctness, §4 Token Verification).
 *   u = 0, path = [0], p = softmax(llm_logits[u] / T)
 *   repeat:
 *     for each child c of u in increasing index, x = token[c], q = ssm_probs[c]:
 *       accept iff u_acc[c] * q[x] < p[x]        (u_acc < min(1, p[x]/q[x]))
 *         -> u = c, append c, p = softmax(llm_logits[c] / T), next round
 *       reject -> r = max(0, p - q); Z = sum r; if Z > 0: p = r / Z
 *     no child accepted -> stop
 *   bonus = smallest x with cumsum(p)[x] > u_smp[u] * sum(p)
 *           (if rounding leaves none, the last x with p[x] > 0).
 * Row c of ssm_probs is the distribution node c's token was drawn from; it is
 * used as given.
 *
 * Diagnostics per request: n_tried[b] = number of children tried; n_near_tie[b]
 * = decisions whose margin is below 1e-6 (|u_acc - p[x]/q[x]| for an accept
 * test, p[x] itself when q[x] = 0, and for the bonus draw the distance of the
 * target to the neighbouring cumulative sums, over sum(p));
 * tie_path_len[b] = len(path) at the first such decision (-1 if none).  Two
 * implementations that round differently may part ways only from that point.
 */
/*
 * Warping of the LLM distribution before verification: top-k, then top-p
 * (nucleus), as samplers apply them (SpecInfer's evaluation samples with
 * top-k; the task asks for top-k/top-p).  Reading: tokens are ranked by their
 * logit, larger first, equal logits by lower token index (p is an increasing
 * function of the logit, so this is the ranking by probability with a fixed
 * tie rule).  top_k > 0 keeps the first top_k tokens of the ranking (all when
 * top_k <= 0 or >= V); 0 < top_p < 1 then keeps the shortest prefix of that
 * ranking whose share of the kept mass reaches top_p.  p is set to zero
 * elsewhere and renormalised.  A top-p cut whose cumulative share is within
 * NEAR_TIE_EPS of top_p is reported through *near_tie.
 */
static const float* g_rank_logits;
static int rank_cmp(const void* a, const void* b) {
  const int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
  const float li = g_rank_logits[i], lj = g_rank_logits[j];
  if (li > lj) return -1;
  if (li < lj) return 1;
  return (i > j) - (i < j);
}

static void warp_row(const float* logits, int64_t V, int32_t top_k, double top_p, double* p,
                     int* near_tie) {
  const int use_k = top_k > 0 && (int64_t)top_k < V;
  const int use_p = top_p < 1.0;
  if (!use_k && !use_p) return;
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)V);
  for (int64_t t = 0; t < V; ++t) order[t] = t;
  g_rank_logits = logits;
  qsort(order, (size_t)V, sizeof(int64_t), rank_cmp);
  const int64_t K = use_k ? (int64_t)top_k : V;
  double mass_k = 0.0;
  for (int64_t j = 0; j < K; ++j) mass_k += p[order[j]];
  int64_t keep = K;
  if (use_p) {
    double cum = 0.0, prev = 0.0;
    for (int64_t j = 0; j < K; ++j) {
      prev = cum;
      cum += p[order[j]];
      if (cum >= top_p * mass_k) {
        keep = j + 1;
        break;
      }
    }
    if (fabs(cum - top_p * mass_k) < NEAR_TIE_EPS * mass_k ||
        fabs(prev - top_p * mass_k) < NEAR_TIE_EPS * mass_k)
      *near_tie = 1;
  }
  double mass = 0.0;
  for (int64_t j = 0; j < keep; ++j) mass += p[order[j]];
  for (int64_t j = keep; j < V; ++j) p[order[j]] = 0.0;
  for (int64_t j = 0; j < keep; ++j) p[order[j]] /= mass;
  free(order);
}

int oracle_verify_stochastic(const float* llm_logits, const float* ssm_probs, int64_t V,
                             const int32_t* tokens, const int32_t* parent,
                             const int32_t* node_offsets, const float* u_acc,
                             const float* u_smp, int32_t B, double temperature, int32_t top_k,
                             double top_p, int32_t* path,
                             int32_t* accept_len, int32_t* bonus, int32_t* n_tried,
                             int32_t* n_near_tie, int32_t* tie_path_len, int32_t* status) {
  int rc = ORACLE_OK;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  for (int32_t b = 0; b < B; ++b) {
    const int32_t off = node_offsets[b];
    const int32_t n = node_offsets[b + 1] - off;
    const int32_t* par = parent + off;
    const int32_t* tok = tokens + off;
    int32_t* pth = path + off;
    clear_outputs(pth, n, &accept_len[b], &bonus[b]);
    n_tried[b] = 0;
    n_near_tie[b] = 0;
    tie_path_len[b] = -1;
    status[b] = ORACLE_OK;
    if (!tree_is_verifiable(par, n)) {
      status[b] = ORACLE_BAD_TREE;
      if (rc == ORACLE_OK) rc = ORACLE_BAD_TREE;
      continue;
    }
    int32_t u = 0, len = 0;
    pth[len++] = 0;
    int warp_tie = 0;
    softmax_row(llm_logits + (size_t)(off + u) * V, V, temperature, p);
    warp_row(llm_logits + (size_t)(off + u) * V, V, top_k, top_p, p, &warp_tie);
    if (warp_tie) {
      if (n_near_tie[b] == 0) tie_path_len[b] = len;
      n_near_tie[b] += 1;
    }
    for (;;) {
      int32_t next = -1;
      for (int32_t c = u + 1; c < n && next < 0; ++c) {
        if (par[c] != u) continue;
        const int64_t x = tok[c];
        const float* q = ssm_probs + (size_t)(off + c) * V;
        if (!row_is_finite(q, V) || !row_is_finite(llm_logits + (size_t)(off + u) * V, V)) {
          status[b] = ORACLE_NONFINITE;
          if (rc == ORACLE_OK) rc = ORACLE_NONFINITE;
        }
        const double qx = (double)q[x];
        const double ua = (double)u_acc[off + c];
        n_tried[b] += 1;
        const double margin = qx > 0.0 ? fabs(ua - p[x] / qx) : p[x];
        if (margin < NEAR_TIE_EPS) {
          if (n_near_tie[b] == 0) tie_path_len[b] = len;
          n_near_tie[b] += 1;
        }
        if (ua * qx < p[x]) {
          next = c;
        } else {
          double Z = 0.0;
          for (int64_t t = 0; t < V; ++t) {
            const double r = p[t] - (double)q[t];
            Z += r > 0.0 ? r : 0.0;
          }
          if (Z > 0.0) {
            for (int64_t t = 0; t < V; ++t) {
              const double r = p[t] - (double)q[t];
              p[t] = (r > 0.0 ? r : 0.0) / Z;
            }
          }
        }
      }
      if (next < 0) break;
      u = next;
      pth[len++] = u;
      softmax_row(llm_logits + (size_t)(off + u) * V, V, temperature, p);
      warp_tie = 0;
      warp_row(llm_logits + (size_t)(off + u) * V, V, top_k, top_p, p, &warp_tie);
      if (warp_tie) {
        if (n_near_tie[b] == 0) tie_path_len[b] = len;
        n_near_tie[b] += 1;
      }
    }
    accept_len[b] = len - 1;

    /* Bonus token: inverse-CDF draw from p with the stop node's uniform. */
    double total = 0.0;
    for (int64_t t = 0; t < V; ++t) total += p[t];
    const double target = (double)u_smp[off + u] * total;
    double cum = 0.0, below = 0.0;
    int64_t pick = -1, last_pos = -1;
    for (int64_t t = 0; t < V; ++t) {
      if (p[t] > 0.0) last_pos = t;
      below = cum;
      cum += p[t];
      if (cum > target) {
        pick = t;
        break;
      }
    }
    if (pick < 0) {
      pick = last_pos;
      below = cum;
    }
    if (target - below < NEAR_TIE_EPS * total || cum - target < NEAR_TIE_EPS * total) {
      if (n_near_tie[b] == 0) tie_path_len[b] = len;
      n_near_tie[b] += 1;
    }
    bonus[b] = (int32_t)pick;
  }
  free(p);
  return rc;
}

/* Threads the OpenMP loops above use (1 when built without OpenMP), and a way
 * to change that for later calls from the calling thread (the benchmark times
 * the oracle on all host cores and on one).  Results do not depend on it: the
 * loops only spread independent output units over threads. */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
void oracle_set_num_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
}
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_num_threads(int n) { (void)n; }
#endif
