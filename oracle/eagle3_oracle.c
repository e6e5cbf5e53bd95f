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
int e3o_build_tree(int C, const int* c_tok, const int* c_parent, const float* c_score,
                   const int* c_depth, int N, int root_tok, int kv_len, int* tok,
                   int* parent, int* depth, int* pos, uint64_t* mask, int mask_words) {
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
