/*
 * eagle3_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow CPU implementation of the integer / decision steps of one EAGLE-3
 * draft-and-verify round.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline leg may load this file's library.  It shares no code with the
 * CUDA path under eagle_speculative_decoding_round_gb300/csrc/.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math), so
 * that every fp32 operation below is one correctly rounded IEEE operation and
 * fmaf() is the correctly rounded fused multiply-add of C99.
 *
 * Sources (web pages on EAGLE-3; cited by page title and section):
 *  [EAGLE系列] "EAGLE 系列与 DFlash" (pzsr.cn news 22952):
 *      §二 EAGLE-2 阶段一 (top-K expansion, K=3 -> 3 -> 9 nodes),
 *      §二 阶段二 (flatten to [x_1,x_2,x_3,x_1a,...]; 步骤① positions;
 *      步骤② 0/1 tree mask: x_1a sees x_1 and the root, never x_2),
 *      §二 阶段三 (one target forward; accept the longest coherent prefix;
 *      roll back to the last accepted node), §四 DFlash (accept with
 *      min(1, p_target/p_draft), dice left to right).
 *  [SpecForge] "SpecForge：把 EAGLE3 从训练样本交付到 SGLang":
 *      "先看 checkpoint 最终要参与什么计算" (accept the prefix, correct at the
 *      rejection point; output distribution equals the target's),
 *      "从序列到动态草稿树" (node budget by confidence; ancestor-only attention).
 *  [TB] "Thinking Budget 与 EAGLE-3", "一棵候选树怎样被验证" (positions, mask,
 *      one forward, accept by target probabilities, commit only the path's KV).
 *  [EAGLE-3 deep dive] "论文专题讲解：EAGLE-3", "Draft tree 配置" (10 nodes
 *      per expansion, depth 6, 60 draft tokens for 8B).
 *
 * Readings taken where the pages leave a step open (each also listed in the
 * design notes):
 *  - Draft confidence = cumulative draft log-probability at temperature 1.
 *  - Softmax masses are fixed point: Q_j = floor(2^40 * E(s_j - m)) with E a
 *    written-out fp32 exp (Cody-Waite reduction + degree-7 Taylor polynomial,
 *    Horner with fmaf).  Integer sums make the decisions order independent.
 *  - The tree's children are deterministic top-k proposals, so the page's
 *    min(1, p/q) rule is applied with q the point mass on the proposed token:
 *    accept child c with probability p_res(c), else remove it from the residual
 *    and try the next sibling; with no child accepted, sample the bonus token
 *    from the residual (this is the "correction at the rejection point").
 *  - Greedy (T <= 0): accept the child whose token is the row argmax.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* fp32 decision arithmetic                                                  */
/* ------------------------------------------------------------------------ */

/* Cody & Waite (1980) split of ln 2: the high part has 16 significant bits,
 * so n * LN2_HI is exact for |n| < 2^8. */
static const float OR_LOG2E = 0x1.715476p+0f;  /* log2(e)  */
static const float OR_LN2_HI = 0x1.62e4p-1f;   /* 0.693145751953125 */
static const float OR_LN2_LO = 0x1.7f7d1cp-20f; /* ln2 - LN2_HI */
static const float OR_SQRT2 = 0x1.6a09e6p+0f;

static float or_pow2(int n) { /* exact 2^n for -126 <= n <= 127 */
  uint32_t b = (uint32_t)(n + 127) << 23;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

/* E(x) ~ exp(x) for x <= 0 (x finite).  Returns 0 below -32 (exp(-32) < 2^-46,
 * which maps to Q = 0 anyway). */
float e3o_exp(float x) {
  if (x < -32.0f) return 0.0f;
  float t = x * OR_LOG2E;
  float n = rintf(t); /* round half to even */
  float r = fmaf(-n, OR_LN2_HI, x);
  r = fmaf(-n, OR_LN2_LO, r);
  /* Taylor polynomial of exp(r) to degree 7: coefficients 1/k! rounded to fp32 */
  float p = 0x1.a01a02p-13f;          /* 1/5040 */
  p = fmaf(p, r, 0x1.6c16c2p-10f);    /* 1/720 */
  p = fmaf(p, r, 0x1.111112p-7f);     /* 1/120 */
  p = fmaf(p, r, 0x1.555556p-5f);     /* 1/24 */
  p = fmaf(p, r, 0x1.555556p-3f);     /* 1/6 */
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return p * or_pow2((int)n);
}

/* Fixed-point mass of one logit: floor(2^40 * E(s - m)).  s <= m. */
uint64_t e3o_qmass(float s, float m) {
  float e = e3o_exp(s - m);
  float y = e * 0x1p40f; /* exact power-of-two scaling */
  return (uint64_t)y;    /* truncation toward zero = floor for y >= 0 */
}

/* ell = ln(Q * 2^-40) for Q >= 2^40: exponent extraction plus
 * ln f = 2 atanh((f-1)/(f+1)) summed to t^11. */
float e3o_ell(uint64_t Q) {
  float y = (float)Q; /* round to nearest */
  uint32_t b;
  memcpy(&b, &y, 4);
  int e = (int)(b >> 23) - 127;
  uint32_t mb = (b & 0x7FFFFFu) | 0x3F800000u;
  float f;
  memcpy(&f, &mb, 4);
  if (f > OR_SQRT2) {
    f = f * 0.5f;
    e += 1;
  }
  float t = (f - 1.0f) / (f + 1.0f);
  float t2 = t * t;
  float P = 0x1.745d18p-4f;        /* 1/11 */
  P = fmaf(P, t2, 0x1.c71c72p-4f); /* 1/9 */
  P = fmaf(P, t2, 0x1.24924ap-3f); /* 1/7 */
  P = fmaf(P, t2, 0x1.99999ap-3f); /* 1/5 */
  P = fmaf(P, t2, 0x1.555556p-2f); /* 1/3 */
  P = fmaf(P, t2, 1.0f);
  float lnf = (t * P) * 2.0f;
  float k = (float)(e - 40);
  return fmaf(k, OR_LN2_HI, fmaf(k, OR_LN2_LO, lnf));
}

static float or_inv_temp(float T) { return T > 0.0f ? 1.0f / T : 1.0f; }

/* Softmax statistics of one logit row z[V] at temperature T:
 *   s_j = z_j * (1/T) (s_j = z_j when T <= 0), m = max s, argmax (lowest id on
 *   ties), Q = sum_j floor(2^40 E(s_j - m)).  Returns 1 if a logit is not finite. */
int e3o_row_stats(const float* z, int V, float T, float* m_out, uint64_t* Q_out,
                  int* argmax_out) {
  float it = or_inv_temp(T);
  float m = -INFINITY;
  int am = 0;
  for (int j = 0; j < V; ++j) {
    if (!isfinite(z[j])) return 1;
    float s = z[j] * it;
    if (s > m) {
      m = s;
      am = j;
    }
  }
  uint64_t Q = 0;
  for (int j = 0; j < V; ++j) Q += e3o_qmass(z[j] * it, m);
  *m_out = m;
  *Q_out = Q;
  *argmax_out = am;
  return 0;
}

void e3o_row_stats_batch(const float* z, int M, int V, const float* T, float* m_out,
                         uint64_t* Q_out, int* argmax_out, int* nonfinite) {
  for (int i = 0; i < M; ++i)
    nonfinite[i] = e3o_row_stats(z + (size_t)i * V, V, T[i], m_out + i, Q_out + i,
                                 argmax_out + i);
}

/* ------------------------------------------------------------------------ */
/* a2: one depth of dynamic-tree expansion, one request                      */
/* ------------------------------------------------------------------------ */

/* Candidate key order used everywhere: score descending, then candidate index
 * ascending.  Returns 1 if a comes before b. */
static int or_key_before(float sa, int ia, float sb, int ib) {
  if (sa != sb) return sa > sb;
  return ia < ib;
}

/* Top-k of one row by s (descending), ties to the lower token id: k passes of a
 * plain arg-max over the tokens not yet taken. */
static void or_topk_row(const float* z, int V, float it, int k, int* out_tok) {
  for (int r = 0; r < k; ++r) {
    int best = -1;
    float bs = 0.0f;
    for (int j = 0; j < V; ++j) {
      int taken = 0;
      for (int q = 0; q < r; ++q)
        if (out_tok[q] == j) taken = 1;
      if (taken) continue;
      float s = z[j] * it;
      if (best < 0 || s > bs) {
        best = j;
        bs = s;
      }
    }
    out_tok[r] = best;
  }
}

/* Expand F frontier rows (logits[F][V]).  Row f's r-th child is written at
 * candidate index cand_offset + f*k + r with
 *   score = (S_parent + (s_c - m)) - ell,   ell = ln(Q * 2^-40).
 * Then the next frontier = the first min(W, F*k) of these F*k children in key
 * order.  Returns the next frontier size, or -1 if a logit is not finite. */
int e3o_expand(const float* logits, int F, int V, int k, int W, float inv_T,
               const float* parent_score, const int* parent_id, int depth,
               int cand_offset, int* c_tok, int* c_parent, float* c_score,
               int* c_depth, int* next_id, float* next_score) {
  int* top = (int*)malloc(sizeof(int) * (size_t)k);
  for (int f = 0; f < F; ++f) {
    const float* z = logits + (size_t)f * V;
    float m = -INFINITY;
    for (int j = 0; j < V; ++j) {
      if (!isfinite(z[j])) {
        free(top);
        return -1;
      }
      float s = z[j] * inv_T;
      if (s > m) m = s;
    }
    uint64_t Q = 0;
    for (int j = 0; j < V; ++j) Q += e3o_qmass(z[j] * inv_T, m);
    float ell = e3o_ell(Q);
    or_topk_row(z, V, inv_T, k, top);
    for (int r = 0; r < k; ++r) {
      int ci = cand_offset + f * k + r;
      float sc = z[top[r]] * inv_T;
      c_tok[ci] = top[r];
      c_parent[ci] = parent_id[f];
      c_score[ci] = (parent_score[f] + (sc - m)) - ell;
      c_depth[ci] = depth;
    }
  }
  free(top);
  /* selection of the next frontier: repeated pick of the best remaining child */
  int n = F * k;
  int nf = W < n ? W : n;
  char* used = (char*)calloc((size_t)n, 1);
  for (int q = 0; q < nf; ++q) {
    int best = -1;
    for (int i = 0; i < n; ++i) {
      if (used[i]) continue;
      int ci = cand_offset + i;
      if (best < 0 || or_key_before(c_score[ci], ci, c_score[cand_offset + best],
                                    cand_offset + best))
        best = i;
    }
    used[best] = 1;
    next_id[q] = cand_offset + best;
    next_score[q] = c_score[cand_offset + best];
  }
  free(used);
  return nf;
}

/* ------------------------------------------------------------------------ */
/* a3: rerank, flatten, positions, ancestor mask -- one request               */
/* ------------------------------------------------------------------------ */

/* Keep the N best of C candidates (key order), flatten breadth first with the
 * root as node 0: depth by depth, ordered by (parent's flat index, candidate
 * index).  pos = kv_len + depth.  mask row i (mask_words uint64 words) has bit j
 * set iff node j is node i or one of its ancestors.  Returns 0, or 1 if the kept
 * set is not closed under parents (cannot happen for scores from e3o_expand). */
int e3o_build_tree_cand(int C, const int* c_tok, const int* c_parent, const float* c_score,
                        const int* c_depth, int N, int root_tok, int kv_len, int* tok,
                        int* parent, int* depth, int* pos, uint64_t* mask, int mask_words,
                        int* node_cand);

int e3o_build_tree(int C, const int* c_tok, const int* c_parent, const float* c_score,
                   const int* c_depth, int N, int root_tok, int kv_len, int* tok,
                   int* parent, int* depth, int* pos, uint64_t* mask, int mask_words) {
  return e3o_build_tree_cand(C, c_tok, c_parent, c_score, c_depth, N, root_tok, kv_len, tok,
                             parent, depth, pos, mask, mask_words, NULL);
}

/* As e3o_build_tree; node_cand (nullable, [N+1]) receives the candidate index
 * of each flattened node (-1 for the root). */
int e3o_build_tree_cand(int C, const int* c_tok, const int* c_parent, const float* c_score,
                        const int* c_depth, int N, int root_tok, int kv_len, int* tok,
                        int* parent, int* depth, int* pos, uint64_t* mask, int mask_words,
                        int* node_cand) {
  int R = N + 1;
  char* kept = (char*)calloc((size_t)C, 1);
  for (int q = 0; q < N; ++q) { /* N picks of the best remaining candidate */
    int best = -1;
    for (int i = 0; i < C; ++i) {
      if (kept[i]) continue;
      if (best < 0 || or_key_before(c_score[i], i, c_score[best], best)) best = i;
    }
    kept[best] = 1;
  }
  int* flat = (int*)malloc(sizeof(int) * (size_t)C); /* candidate -> flat index */
  for (int i = 0; i < C; ++i) flat[i] = -1;
  tok[0] = root_tok;
  parent[0] = -1;
  depth[0] = 0;
  pos[0] = kv_len;
  if (node_cand) node_cand[0] = -1;
  int next = 1, rc = 0;
  int maxd = 0;
  for (int i = 0; i < C; ++i)
    if (kept[i] && c_depth[i] > maxd) maxd = c_depth[i];
  for (int d = 1; d <= maxd; ++d) {
    for (;;) { /* repeatedly take the smallest (parent flat, cand idx) at depth d */
      int best = -1, bpf = 0;
      for (int i = 0; i < C; ++i) {
        if (!kept[i] || c_depth[i] != d || flat[i] >= 0) continue;
        int pf;
        if (c_parent[i] < 0)
          pf = 0;
        else
          pf = flat[c_parent[i]];
        if (pf < 0) { /* parent not kept */
          rc = 1;
          pf = 1 << 30;
        }
        if (best < 0 || pf < bpf || (pf == bpf && i < best)) {
          best = i;
          bpf = pf;
        }
      }
      if (best < 0) break;
      flat[best] = next;
      if (node_cand) node_cand[next] = best;
      tok[next] = c_tok[best];
      parent[next] = bpf < (1 << 30) ? bpf : -2;
      depth[next] = d;
      pos[next] = kv_len + d;
      ++next;
    }
  }
  for (int i = 0; i < R; ++i) {
    uint64_t* row = mask + (size_t)i * mask_words;
    for (int w = 0; w < mask_words; ++w) row[w] = 0;
    /* walk to the root through parent[] */
    int j = i;
    while (j >= 0) {
      row[j >> 6] |= (uint64_t)1 << (j & 63);
      j = parent[j] >= 0 ? parent[j] : -1;
    }
  }
  free(kept);
  free(flat);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* a6: speculative-sampling accept / reject on the flattened tree            */
/* ------------------------------------------------------------------------ */

static uint64_t or_mulhi32(uint32_t u, uint64_t R) { /* (u * R) >> 32, exact */
  unsigned __int128 p = (unsigned __int128)u * (unsigned __int128)R;
  return (uint64_t)(p >> 32);
}

/* One request.  logits: [R][V] fp32 target logits of the flattened nodes.
 * u_acc[c]: uniform for testing child c; u_bonus[u]: uniform for the bonus
 * draw at node u.  Writes acc_len, path[D+1] (flat ids, root first, -1 pad),
 * out_tok[D+1] (accepted tokens then the bonus token, -1 pad).
 * Returns 0, or 1 if a visited row has a non-finite logit. */
int e3o_accept(const int* tok, const int* parent, int R, int D, const float* logits,
               int V, float T, const uint32_t* u_acc, const uint32_t* u_bonus,
               int* acc_len, int* path, int* out_tok) {
  for (int j = 0; j <= D; ++j) path[j] = out_tok[j] = -1;
  char* removed = (char*)calloc((size_t)V, 1);
  int u = 0, a = 0, rc = 0;
  path[0] = 0;
  float it = or_inv_temp(T);
  for (;;) {
    const float* z = logits + (size_t)u * V;
    float m;
    uint64_t Rmass;
    int am;
    if (e3o_row_stats(z, V, T, &m, &Rmass, &am)) {
      rc = 1;
      break;
    }
    int accepted = -1;
    memset(removed, 0, (size_t)V);
    for (int c = u + 1; c < R; ++c) { /* children of u in flattened order */
      if (parent[c] != u) continue;
      int t = tok[c];
      if (T <= 0.0f) {
        if (t == am) {
          accepted = c;
          break;
        }
        continue;
      }
      uint64_t q = e3o_qmass(z[t] * it, m);
      if (or_mulhi32(u_acc[c], Rmass) < q) {
        accepted = c;
        break;
      }
      Rmass -= q; /* residual: remove the rejected proposal's mass */
      removed[t] = 1;
    }
    if (accepted >= 0 && a < D) {
      ++a;
      path[a] = accepted;
      out_tok[a - 1] = tok[accepted];
      u = accepted;
      continue;
    }
    /* bonus / correction token from row u */
    int bonus = -1;
    if (T <= 0.0f) {
      bonus = am;
    } else {
      uint64_t x = or_mulhi32(u_bonus[u], Rmass);
      uint64_t cum = 0;
      for (int j = 0; j < V; ++j) {
        if (removed[j]) continue;
        cum += e3o_qmass(z[j] * it, m);
        if (cum > x) {
          bonus = j;
          break;
        }
      }
    }
    out_tok[a] = bonus;
    break;
  }
  *acc_len = a;
  free(removed);
  return rc;
}

/* Many independent requests that share one tree (tok/parent) and one logits
 * block, each with its own uniforms: used by the losslessness test. */
void e3o_accept_many(int n, const int* tok, const int* parent, int R, int D,
                     const float* logits, int V, float T, const uint32_t* u_acc,
                     const uint32_t* u_bonus, int* acc_len, int* path, int* out_tok) {
  for (int i = 0; i < n; ++i)
    e3o_accept(tok, parent, R, D, logits, V, T, u_acc + (size_t)i * R,
               u_bonus + (size_t)i * R, acc_len + i, path + (size_t)i * (D + 1),
               out_tok + (size_t)i * (D + 1));
}

/* ------------------------------------------------------------------------ */
/* Sampled drafts: children drawn from the draft distribution q, accepted     */
/* with min(1, p_res / q_res) ("EAGLE 系列与 DFlash", §四 DFlash)               */
/* ------------------------------------------------------------------------ */

/* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): the stream started at `seed` has the i-th output
 * (i >= 1) mix(seed + i * 0x9E3779B97F4A7C15). */
uint64_t e3o_splitmix64_at(uint64_t seed, uint64_t i) {
  uint64_t z = seed + i * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Exponential variate of the draw for token j of frontier row f at `depth` of
 * request b: output number n + 1 of the stream at `seed`, with the counter
 * n = b 2^44 + depth 2^36 + f 2^24 + j; U = (top 24 bits + 1) 2^-24 in (0, 1]
 * and E = 0 - ln U, with ln by the same recipe as ell (U = Q' 2^-40 for the
 * integer Q' = (top 24 bits + 1) 2^16). */
float e3o_exp_variate(uint64_t seed, int b, int depth, int f, int j) {
  uint64_t n = ((uint64_t)b << 44) | ((uint64_t)depth << 36) | ((uint64_t)f << 24) | (uint64_t)j;
  uint64_t u24 = e3o_splitmix64_at(seed, n + 1) >> 40;
  return 0.0f - e3o_ell((u24 + 1) << 16);
}

/* The k children of one row drawn without replacement with probabilities
 * proportional to the recipe's e_j = E(s_j - m): each token's arrival time is
 * E_j / e_j (an exponential clock of rate e_j); children are the k earliest
 * arrivals, earliest first, equal times to the lower token id.  A token whose
 * fixed-point mass floor(2^40 e_j) is 0 never arrives (time +inf). */
static void or_sample_row(const float* z, int V, float it, float m, int k, uint64_t seed, int b,
                          int depth, int f, int* out_tok, float* t_buf) {
  for (int j = 0; j < V; ++j) {
    float s = z[j] * it;
    float e = e3o_exp(s - m);
    if ((uint64_t)(e * 0x1p40f) == 0) {
      t_buf[j] = INFINITY;
      continue;
    }
    t_buf[j] = e3o_exp_variate(seed, b, depth, f, j) / e;
  }
  for (int r = 0; r < k; ++r) { /* k passes of a plain arg-min over the tokens not taken */
    int best = -1;
    for (int j = 0; j < V; ++j) {
      int taken = 0;
      for (int q = 0; q < r; ++q)
        if (out_tok[q] == j) taken = 1;
      if (taken) continue;
      if (best < 0 || t_buf[j] < t_buf[best]) best = j;
    }
    out_tok[r] = best;
  }
}

/* As e3o_expand, but row f's children are its k sampled tokens in arrival
 * order (request b, draws keyed by `seed`); scores, candidate layout and the
 * next frontier (by score) are as in e3o_expand.  row_m[f] / row_Q[f] receive
 * the row's maximum and fixed-point total mass (the draft statistics that the
 * sampled accept uses).  Returns the next frontier size, or -1 on a non-finite
 * logit. */
int e3o_expand_sampled(const float* logits, int F, int V, int k, int W, float inv_T,
                       const float* parent_score, const int* parent_id, int depth,
                       int cand_offset, uint64_t seed, int b, int* c_tok, int* c_parent,
                       float* c_score, int* c_depth, int* next_id, float* next_score,
                       float* row_m, uint64_t* row_Q) {
  int* top = (int*)malloc(sizeof(int) * (size_t)k);
  float* t_buf = (float*)malloc(sizeof(float) * (size_t)V);
  for (int f = 0; f < F; ++f) {
    const float* z = logits + (size_t)f * V;
    float m = -INFINITY;
    for (int j = 0; j < V; ++j) {
      if (!isfinite(z[j])) {
        free(top);
        free(t_buf);
        return -1;
      }
      float s = z[j] * inv_T;
      if (s > m) m = s;
    }
    uint64_t Q = 0;
    for (int j = 0; j < V; ++j) Q += e3o_qmass(z[j] * inv_T, m);
    float ell = e3o_ell(Q);
    row_m[f] = m;
    row_Q[f] = Q;
    or_sample_row(z, V, inv_T, m, k, seed, b, depth, f, top, t_buf);
    for (int r = 0; r < k; ++r) {
      int ci = cand_offset + f * k + r;
      float sc = z[top[r]] * inv_T;
      c_tok[ci] = top[r];
      c_parent[ci] = parent_id[f];
      c_score[ci] = (parent_score[f] + (sc - m)) - ell;
      c_depth[ci] = depth;
    }
  }
  free(top);
  free(t_buf);
  int n = F * k;
  int nf = W < n ? W : n;
  char* used = (char*)calloc((size_t)n, 1);
  for (int q = 0; q < nf; ++q) {
    int best = -1;
    for (int i = 0; i < n; ++i) {
      if (used[i]) continue;
      int ci = cand_offset + i;
      if (best < 0 || or_key_before(c_score[ci], ci, c_score[cand_offset + best],
                                    cand_offset + best))
        best = i;
    }
    used[best] = 1;
    next_id[q] = cand_offset + best;
    next_score[q] = c_score[cand_offset + best];
  }
  free(used);
  return nf;
}

static uint64_t or_muldiv(uint64_t a, uint64_t b, uint64_t c) { /* floor(a b / c), c > 0 */
  unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
  return (uint64_t)(p / c);
}

/* One request whose children were drawn from the draft distribution.
 * qlogits: [R][V] fp32; row u holds the draft logits from which node u's
 * children were drawn (rows of nodes without children are not read), at inverse
 * temperature inv_Tq.  At node u the target residual is kept as integer masses
 * Rm[j] (initially floor(2^40 E(z_j/T - m)), total SR) and the draft residual
 * as Dm[j] (initially floor(2^40 E(zq_j inv_Tq - m_q)), total SD).  Children in
 * flattened order (= draw order):
 *   a child whose token has Dm[t] = 0 was not drawn (the row had fewer than k
 *   tokens of positive mass) and is skipped;
 *   Qs = floor(Dm[t] SR / SD) is the draft mass of t in the target's units;
 *   accept iff u_acc[c] Qs < Rm[t] 2^32: probability min(1, p_res(t) / q_res(t));
 *   on reject every Rm[j] -= min(Rm[j], floor(Dm[j] SR / SD)) (the residual
 *   max(0, p_res - q_res) up to normalisation) and Dm[t] = 0 (t leaves q_res).
 * With no child accepted (or at a leaf) the bonus token is the smallest j whose
 * cumulative Rm exceeds (u_bonus[u] SR) >> 32.  T <= 0: greedy, as e3o_accept.
 * Returns 0, or 1 on a non-finite logit in a visited row. */
int e3o_accept_sampled(const int* tok, const int* parent, int R, int D, const float* logits,
                       int V, float T, const float* qlogits, float inv_Tq,
                       const uint32_t* u_acc, const uint32_t* u_bonus, int* acc_len,
                       int* path, int* out_tok) {
  if (T <= 0.0f)
    return e3o_accept(tok, parent, R, D, logits, V, T, u_acc, u_bonus, acc_len, path, out_tok);
  for (int j = 0; j <= D; ++j) path[j] = out_tok[j] = -1;
  uint64_t* Rm = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
  uint64_t* Dm = (uint64_t*)calloc((size_t)V, sizeof(uint64_t));
  float it = or_inv_temp(T);
  int u = 0, a = 0, rc = 0;
  path[0] = 0;
  for (;;) {
    const float* z = logits + (size_t)u * V;
    float m;
    uint64_t SR;
    int am;
    if (e3o_row_stats(z, V, T, &m, &SR, &am)) {
      rc = 1;
      break;
    }
    for (int j = 0; j < V; ++j) Rm[j] = e3o_qmass(z[j] * it, m);
    int has_child = 0;
    for (int c = u + 1; c < R; ++c)
      if (parent[c] == u) has_child = 1;
    uint64_t SD = 0;
    if (has_child) {
      const float* zq = qlogits + (size_t)u * V;
      float mq = -INFINITY;
      for (int j = 0; j < V; ++j) {
        if (!isfinite(zq[j])) rc = 1;
        float s = zq[j] * inv_Tq;
        if (s > mq) mq = s;
      }
      if (rc) break;
      for (int j = 0; j < V; ++j) {
        Dm[j] = e3o_qmass(zq[j] * inv_Tq, mq);
        SD += Dm[j];
      }
    }
    int accepted = -1;
    for (int c = u + 1; c < R && has_child; ++c) {
      if (parent[c] != u) continue;
      int t = tok[c];
      if (t < 0 || t >= V || Dm[t] == 0) continue;
      uint64_t qs = or_muldiv(Dm[t], SR, SD);
      if ((unsigned __int128)u_acc[c] * qs < ((unsigned __int128)Rm[t] << 32)) {
        accepted = c;
        break;
      }
      uint64_t nSR = 0;
      for (int j = 0; j < V; ++j) {
        uint64_t qj = or_muldiv(Dm[j], SR, SD);
        Rm[j] = Rm[j] > qj ? Rm[j] - qj : 0;
        nSR += Rm[j];
      }
      SR = nSR;
      SD -= Dm[t];
      Dm[t] = 0;
    }
    if (accepted >= 0 && a < D) {
      ++a;
      path[a] = accepted;
      out_tok[a - 1] = tok[accepted];
      u = accepted;
      continue;
    }
    uint64_t x = or_mulhi32(u_bonus[u], SR);
    uint64_t cum = 0;
    int bonus = -1;
    for (int j = 0; j < V; ++j) {
      cum += Rm[j];
      if (cum > x) {
        bonus = j;
        break;
      }
    }
    out_tok[a] = bonus;
    break;
  }
  *acc_len = a;
  free(Rm);
  free(Dm);
  return rc;
}

/* n independent rounds of a small synthetic model with sampled drafts (the
 * losslessness test): trial i draws its tree with seed0 + i -- depth d's
 * frontier row f has draft logits qtab[d-1][f] ([D][Fmax][V]), k children per
 * row, the next frontier the W best by score, every candidate kept -- and the
 * target logits of a node depend on its token only (ptab[0] for the root,
 * ptab[1 + tok] otherwise; [V+1][V]).  Uniforms: u_acc / u_bonus [n][Rcap].
 * Outputs acc_len[n] and out_tok[n][D+1].  Returns the trees' node count R, or
 * -1 if they do not fit Rcap. */
int e3o_sampled_trials(int n, int V, int k, int W, int D, const float* qtab, int Fmax,
                       float inv_Tq, const float* ptab, float T, uint64_t seed0,
                       const uint32_t* u_acc, const uint32_t* u_bonus, int Rcap,
                       int* acc_len, int* out_tok) {
  int C = 0, F = 1;
  for (int d = 0; d < D; ++d) {
    C += F * k;
    F = W < F * k ? W : F * k;
  }
  int R = C + 1;
  if (R > Rcap) return -1;
  int *c_tok = malloc(sizeof(int) * C), *c_par = malloc(sizeof(int) * C);
  int* c_dep = malloc(sizeof(int) * C);
  float* c_sc = malloc(sizeof(float) * C);
  int *fid = malloc(sizeof(int) * (C + 1)), *nid = malloc(sizeof(int) * (C + 1));
  float *fsc = malloc(sizeof(float) * (C + 1)), *nsc = malloc(sizeof(float) * (C + 1));
  float* rm = malloc(sizeof(float) * (C + 1));
  uint64_t* rq = malloc(sizeof(uint64_t) * (C + 1));
  int* qrow_of_cand = malloc(sizeof(int) * (C + 1)); /* cand -> index into qtab rows, -1 */
  int *tok = malloc(sizeof(int) * R), *par = malloc(sizeof(int) * R);
  int *dep = malloc(sizeof(int) * R), *pos = malloc(sizeof(int) * R);
  int* ncand = malloc(sizeof(int) * R);
  int words = (R + 63) / 64;
  uint64_t* mask = malloc(sizeof(uint64_t) * (size_t)R * words);
  float* zt = malloc(sizeof(float) * (size_t)R * V);
  float* zq = calloc((size_t)R * V, sizeof(float));
  int path[64];
  for (int i = 0; i < n; ++i) {
    uint64_t seed = seed0 + (uint64_t)i;
    int Fd = 1, off = 0, root_row = 0;
    fid[0] = -1;
    fsc[0] = 0.0f;
    for (int c = 0; c < C; ++c) qrow_of_cand[c] = -1;
    for (int d = 1; d <= D; ++d) {
      const float* rows = qtab + (size_t)(d - 1) * Fmax * V;
      for (int f = 0; f < Fd; ++f) {
        int row = (d - 1) * Fmax + f;
        if (fid[f] < 0)
          root_row = row;
        else
          qrow_of_cand[fid[f]] = row;
      }
      int nf = e3o_expand_sampled(rows, Fd, V, k, W, inv_Tq, fsc, fid, d, off, seed, 0, c_tok,
                                  c_par, c_sc, c_dep, nid, nsc, rm, rq);
      off += Fd * k;
      for (int f = 0; f < nf; ++f) {
        fid[f] = nid[f];
        fsc[f] = nsc[f];
      }
      Fd = nf;
    }
    e3o_build_tree_cand(C, c_tok, c_par, c_sc, c_dep, C, 0, 0, tok, par, dep, pos, mask, words,
                        ncand);
    for (int u = 0; u < R; ++u) {
      const float* src = ptab + (size_t)(u == 0 ? 0 : 1 + tok[u]) * V;
      memcpy(zt + (size_t)u * V, src, sizeof(float) * V);
      int qr = u == 0 ? root_row : qrow_of_cand[ncand[u]];
      if (qr >= 0) memcpy(zq + (size_t)u * V, qtab + (size_t)qr * V, sizeof(float) * V);
    }
    tok[0] = 0;
    e3o_accept_sampled(tok, par, R, D, zt, V, T, zq, inv_Tq, u_acc + (size_t)i * Rcap,
                       u_bonus + (size_t)i * Rcap, acc_len + i, path, out_tok + (size_t)i * (D + 1));
  }
  free(c_tok); free(c_par); free(c_dep); free(c_sc); free(fid); free(nid); free(fsc); free(nsc);
  free(rm); free(rq); free(qrow_of_cand); free(tok); free(par); free(dep); free(pos); free(ncand);
  free(mask); free(zt); free(zq);
  return R;
}
