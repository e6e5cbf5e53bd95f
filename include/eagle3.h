/*
 * eagle3.h -- C ABI of libeagle3, one EAGLE-3 draft-and-verify round on one GPU.
 *
 * The round (sources are web pages on EAGLE-3, cited by title and section):
 *   eagle3_fuse      g = W_f [h_low; h_mid; h_high]
 *                    ("论文专题讲解：EAGLE-3", 推理流程：多层特征融合 + 单层 draft decoder;
 *                     "SpecForge：把 EAGLE3 从训练样本交付到 SGLang", 多层特征融合到底融合了什么)
 *   eagle3_expand    one depth of the EAGLE-2 dynamic draft tree: top-k children
 *                    per frontier node, cumulative confidence, next frontier
 *                    ("EAGLE 系列与 DFlash", §二 EAGLE-2 阶段一; "论文专题讲解：EAGLE-3",
 *                     Draft tree 配置)
 *   tree_build_mask  keep the N most confident nodes, flatten breadth first,
 *                    positions and the ancestor-only 0/1 mask
 *                    ("EAGLE 系列与 DFlash", §二 阶段二, 关键新增步骤① and ②)
 *   tree_verify_attn one tree-masked attention layer of the single verify pass
 *                    ("EAGLE 系列与 DFlash", §二 阶段三; "Thinking Budget 与 EAGLE-3",
 *                     一棵候选树怎样被验证; prefix and tree segments merged by
 *                     log-sum-exp as in "EAGLE-3 投机解码与 USP 长序列训练优化",
 *                     USP 核心设计：三步走)
 *   lmhead_logits    per-node target logits and softmax statistics
 *                    ("SpecForge…", 先看 checkpoint 最终要参与什么计算: the target
 *                     computes the true probabilities of the tree)
 *   spec_accept      speculative-sampling accept/reject along the tree, residual
 *                    correction at the rejection point, longest accepted path
 *                    ("EAGLE 系列与 DFlash", §四 DFlash worked example and §二 阶段三;
 *                     "SpecForge…", 接受连续前缀，拒绝处进行校正)
 *   kv_compact       commit only the accepted path's KV
 *                    ("Thinking Budget 与 EAGLE-3", 一棵候选树怎样被验证, step 5)
 *
 * Conventions (every call):
 *  - All data pointers are DEVICE pointers owned by the caller, unless a
 *    parameter says "host".  The library keeps no allocation across calls.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and return after enqueue.
 *  - Shape and argument errors are detected on the host before any launch and
 *    return a non-OK status without touching device memory;
 *    eagle3_last_error() then gives a message (thread local).
 *  - Data-dependent errors found on the device (non-finite logits, a page
 *    table too short for kv_len + R, a wait that ran out) are OR-ed into the
 *    caller's `dev_err` word (int32, device, nullable) with the E3_DEV_ERR_*
 *    bits; kernels never trap.
 *  - Row-major layouts, innermost dimension last.  bf16 is IEEE bfloat16.
 *  - Calls may come from several host threads at once: the library's one-time
 *    setup (kernel attributes, cluster sizes) is thread safe and the error
 *    message is per thread.  Calls share no device state, except the fixed
 *    scratch of eagle3_fuse_noalloc (see there).
 *  - One device per process: that one-time setup (shared-memory and cluster
 *    attributes of the kernels, occupancy queries) is done once per process, on
 *    the device current at the first call.  Use one process per GPU.
 */
#ifndef EAGLE3_H
#define EAGLE3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define E3_API __attribute__((visibility("default")))
#else
#define E3_API
#endif

typedef struct CUstream_st* e3_stream_t; /* same type as cudaStream_t */

typedef enum {
  E3_OK = 0,
  E3_ERR_INVALID_ARG = 1, /* null pointer, bad enum, misaligned pointer */
  E3_ERR_SHAPE = 2,       /* sizes out of the supported range or inconsistent */
  E3_ERR_UNSUPPORTED = 3, /* valid request this build does not implement */
  E3_ERR_CAPACITY = 4,    /* a buffer or workspace is too small */
  E3_ERR_NONFINITE = 5,   /* reserved for synchronous callers; see E3_DEV_ERR_NONFINITE */
  E3_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed */
  E3_ERR_TIMEOUT = 7      /* reserved for synchronous callers; see E3_DEV_ERR_TIMEOUT */
} e3_status;

typedef enum { E3_F32 = 0, E3_BF16 = 1 } e3_dtype;

/* bits of the device error word */
#define E3_DEV_ERR_NONFINITE 1 /* a logit was NaN or +-Inf */
#define E3_DEV_ERR_CAPACITY 2  /* kv_len + R exceeds the request's pages (verify,
                                  compaction); an internal candidate list of
                                  eagle3_expand overflowed (not expected) */
#define E3_DEV_ERR_TIMEOUT 4   /* a bounded on-device wait ran out; outputs invalid */

/* Limits of this build. */
#define E3_MAX_TOPK 32     /* k of eagle3_expand */
#define E3_MAX_FRONTIER 64 /* W of eagle3_expand */
#define E3_MAX_NODES 255   /* N of tree_build_mask; R = N + 1 <= 256 */
#define E3_MAX_DEPTH 16    /* D */
#define E3_MAX_CAND 4096   /* candidates per request */
#define E3_MAX_LAYERS 128  /* L of kv_compact */

/* Candidate list of the dynamic tree, structure of arrays, [B][cap] each
 * (device).  Candidate c of request b lives at index b*cap + c. */
typedef struct {
  int32_t* tok;    /* token id */
  int32_t* parent; /* candidate index of the parent within the request; -1 = root */
  float* score;    /* cumulative draft log-probability (confidence) */
  int32_t* depth;  /* 1 for the root's children */
  int cap;         /* candidates per request */
} e3_cand;

/* Draft statistics of one frontier row, written by eagle3_expand_sampled for
 * the node the row expanded and read by spec_accept_sampled (device array
 * [B][1 + cands->cap]: slot 0 = the root, slot 1 + c = candidate c). */
typedef struct {
  const float* row; /* the row's draft logits [V] fp32 (device) */
  uint64_t Q;       /* sum_j floor(2^40 E(z_j * inv_temp - m)) */
  float m;          /* max_j z_j * inv_temp */
  float inv_temp;   /* the draft inverse temperature of the expansion */
} e3_qstat;

/* One layer's paged KV cache.  k and v: [n_pages][n_kv_heads][page_size][head_dim]
 * of dtype dt (device).  Logical token t of request b is slot t % page_size of
 * page page_table[b*max_pages + t / page_size].
 * flags: 0, or E3_KV_PREFIX_STABLE -- a promise about ordering that lets
 * tree_verify_attn start earlier: the prefix K/V (slots below kv_len[b]),
 * kv_len and the page table are NOT written by the kernel enqueued immediately
 * before the tree_verify_attn call on its stream (in a decoder the preceding
 * kernel is the previous layer's attention or this layer's QKV projection,
 * which write neither; kv_compact and page allocation happen earlier).  The
 * kernel then reads the lengths and page table and starts loading prefix K/V
 * while that preceding kernel is still finishing; Q, the mask and the tree
 * slots are read only after it has completed.  Breaking the promise can make
 * the call read stale prefix data.  Other calls ignore the flag. */
#define E3_KV_PREFIX_STABLE 1
/* E3_KV_SELFTEST_STALL: failure-detection self-test, never for production (no
 * counterpart in the pages).  In tree_verify_attn's tensor-core kernel the MMA
 * thread waits on a barrier that nothing arrives on: the bounded wait runs out
 * after about a second, the kernel sets E3_DEV_ERR_TIMEOUT in dev_err, waits for
 * its own copies in flight, frees its tensor memory and returns; O and lse are not
 * valid.  Other paths and calls ignore the bit. */
#define E3_KV_SELFTEST_STALL 0x40000000
typedef struct {
  void* k;
  void* v;
  const int32_t* page_table; /* [B][max_pages], device */
  int n_pages;
  int page_size;
  int max_pages;
  int n_kv_heads;
  int head_dim;
  e3_dtype dt;
  int flags;                 /* 0, E3_KV_PREFIX_STABLE, E3_KV_SELFTEST_STALL */
} e3_kv_layer;

/* ---------------------------------------------------------------------------
 * eagle3_fuse: g[m, o] = sum_j W_f[o, j] x[m, j] (+ bias[o]),
 *   x[m] = [h_low[m]; h_mid[m]; h_high[m]] (3*d values), fp32 accumulation.
 * h_low/h_mid/h_high: [M][d] dtype dt; W_f: [d_out][3*d] dtype dt;
 * bias: [d_out] fp32 or NULL; g: [M][d_out] dtype dt.
 * Limits: 1 <= M <= 65536; d % 64 == 0 and d_out % 128 == 0 for bf16
 * (any positive d, d_out for fp32).  Pointers 16-byte aligned.
 * ws: scratch of eagle3_fuse_workspace_bytes() bytes (device), or NULL if that is 0
 * (bf16 with d % 64 == 0 runs split-K on the tensor cores and needs it).
 * dev_err: E3_DEV_ERR_TIMEOUT if a bounded on-device wait ran out.
 * ------------------------------------------------------------------------- */
E3_API e3_status eagle3_fuse(const void* h_low, const void* h_mid, const void* h_high,
                      const void* W_f, const float* bias, void* g, int M, int d,
                      int d_out, e3_dtype dt, void* ws, size_t ws_bytes,
                      int32_t* dev_err, e3_stream_t stream);
E3_API size_t eagle3_fuse_workspace_bytes(int M, int d, int d_out, e3_dtype dt);

/* ---------------------------------------------------------------------------
 * eagle3_fuse_noalloc: eagle3_fuse for callers that cannot allocate device
 * memory (no cudaMalloc or allocating library call may happen where they run the
 * fusion: allocator-free serving loops, embedders without a device allocator).
 * The pages have no counterpart: this is a library-level convenience.
 * Same inputs, output and numerics as eagle3_fuse, but the split-K scratch is a
 * fixed array inside the library (eagle3_fuse_noalloc_max_scratch_bytes(), 4 MiB;
 * held on every GPU that loads the library until exit).  Shapes whose scratch
 * (eagle3_fuse_workspace_bytes) exceeds it return E3_ERR_CAPACITY before any
 * launch.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress), so make it before any stream capture.  All calls share
 * the array: calls that overlap on the GPU race and must be ordered by the caller.
 * ------------------------------------------------------------------------- */
E3_API e3_status eagle3_fuse_noalloc(const void* h_low, const void* h_mid, const void* h_high,
                                     const void* W_f, const float* bias, void* g, int M, int d,
                                     int d_out, e3_dtype dt, int32_t* dev_err, e3_stream_t stream);
E3_API size_t eagle3_fuse_noalloc_max_scratch_bytes(void);

/* ---------------------------------------------------------------------------
 * eagle3_expand: one depth of the dynamic draft tree, B requests at once.
 * draft_logits: [B][F][V] fp32, row f = frontier node f of the request.
 * parent_score: [B][F] fp32 (the root has 0); parent_id: [B][F] int32
 *   (candidate index of the frontier node, -1 = root).
 * For each row: s_j = z_j * inv_temp (fp32), m = max s,
 *   Q = sum_j floor(2^40 E(s_j - m)), ell = ln(Q 2^-40) (fixed-point recipe),
 *   the k largest s (ties -> lower token id) become children r = 0..k-1 at
 *   candidate index cand_offset + f*k + r with
 *   score = (parent_score + (s_c - m)) - ell and depth = `depth`.
 * Next frontier: the first Wn = min(W, F*k) of these children in the order
 *   (score descending, candidate index ascending) -> next_id [B][Wn] (candidate
 *   index) and next_score [B][Wn].
 * Non-finite logits set E3_DEV_ERR_NONFINITE; E3_DEV_ERR_CAPACITY marks a row
 * whose children may be wrong (an internal list overflowed; its size bound makes
 * this unreachable).
 * Limits: 1 <= k <= E3_MAX_TOPK, k <= V, 1 <= W <= E3_MAX_FRONTIER or W >= F*k,
 *   F*k <= 2048, cand_offset + F*k <= cands->cap <= E3_MAX_CAND.
 * ------------------------------------------------------------------------- */
E3_API e3_status eagle3_expand(const float* draft_logits, int B, int F, int V, int k, int W,
                        float inv_temp, const float* parent_score,
                        const int32_t* parent_id, int depth, int cand_offset,
                        const e3_cand* cands /* host struct, device arrays */,
                        int32_t* next_id, float* next_score, int32_t* dev_err,
                        e3_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle3_expand_sampled: as eagle3_expand, but the k children of a row are
 * DRAWN from the draft distribution q_j = Q_j / Q (Q_j = floor(2^40 E(s_j - m)))
 * without replacement, in draw order ("EAGLE 系列与 DFlash", §四 DFlash: drafts
 * proposed by the drafter and checked with min(1, p_target / p_draft)):
 *   token j of row f (request b) gets the arrival time E_j / e_j, e_j = E(s_j - m),
 *   E_j = 0 - ell(((x >> 40) + 1) << 16) = -ln U_j, x = output number n + 1 of
 *   the SplitMix64 stream started at `seed`, n = b 2^44 + depth 2^36 + f 2^24 + j;
 *   tokens with Q_j = 0 never arrive; the children are the k earliest arrivals
 *   (equal times: lower token id first), child r the r-th.
 * Child scores, candidate layout and the next frontier are exactly those of
 * eagle3_expand.  q_stats [B][1 + cands->cap] (device): the entry of the node
 * each row expanded (slot 1 + parent_id, or 0 for the root) receives the row's
 * address, Q, m and inv_temp, for spec_accept_sampled.
 * Limits: those of eagle3_expand; V < 2^24, F < 4096, depth < 256, B < 2^20.
 * ------------------------------------------------------------------------- */
E3_API e3_status eagle3_expand_sampled(const float* draft_logits, int B, int F, int V, int k,
                                       int W, float inv_temp, const float* parent_score,
                                       const int32_t* parent_id, int depth, int cand_offset,
                                       const e3_cand* cands /* host struct, device arrays */,
                                       int32_t* next_id, float* next_score, uint64_t seed,
                                       e3_qstat* q_stats, int32_t* dev_err, e3_stream_t stream);

/* ---------------------------------------------------------------------------
 * tree_build_mask: per request, keep the N best of the first n_cand candidates
 * in the order (score descending, candidate index ascending) -- closed under
 * parents because a child's score never exceeds its parent's -- and flatten
 * with the root as node 0, then depth by depth ordered by (parent's flat
 * index, candidate index).  R = N + 1.
 * Outputs ([B][R] int32 each): tok (root = root_tok[b]), parent (root -1),
 * depth (root 0), pos = kv_len[b] + depth; mask [B][R][W64] uint64 with
 * W64 = ceil(R/64): bit j of row i set iff node j is node i or an ancestor.
 * node_cand [B][R] int32 (nullable): candidate index of each node (root -1).
 * Limits: 1 <= N <= min(n_cand, E3_MAX_NODES), n_cand <= cands->cap.
 * With sampled children (eagle3_expand_sampled) pass N = n_cand: dropping a
 * drawn child by its own score would bias the accepted tokens.
 * ------------------------------------------------------------------------- */
E3_API e3_status tree_build_mask(const e3_cand* cands, int B, int n_cand, int N,
                          const int32_t* root_tok, const int32_t* kv_len, int32_t* tok,
                          int32_t* parent, int32_t* depth, int32_t* pos, uint64_t* mask,
                          int32_t* node_cand, e3_stream_t stream);

/* ---------------------------------------------------------------------------
 * tree_verify_attn: one attention layer of the verify pass.
 * For request b (P = kv_len[b]), node i < R, query head h < n_q_heads:
 *   keys = prefix [0, P) and tree slots {P + j : bit j of mask[b][i]},
 *   o = softmax(sm_scale * q . k) v,  lse = ln(sum exp(sm_scale * q . k)).
 * The caller has written the tree nodes' K/V at logical slots P .. P+R-1.
 * Query head h reads KV head h / (n_q_heads / n_kv_heads).
 * Q: [B][R][n_q_heads][head_dim] dtype kv->dt; O: same shape and dtype;
 * lse: [B][R][n_q_heads] fp32.  Pages must cover P + R tokens, else
 * E3_DEV_ERR_CAPACITY and the request's outputs are left unwritten.
 * Limits: head_dim 64 or 128 (fp32: any multiple of 32 up to 256); R <= 256;
 *   n_q_heads % n_kv_heads == 0; page_size % 16 == 0.
 * ws: eagle3_verify_workspace_bytes(B, R, n_q_heads, n_kv_heads, head_dim,
 *   max_kv_len, dt) bytes (device scratch), where max_kv_len bounds every kv_len[b].
 * ------------------------------------------------------------------------- */
E3_API e3_status tree_verify_attn(const void* Q, const e3_kv_layer* kv /* host struct */,
                           const int32_t* kv_len, const uint64_t* mask, int B, int R,
                           int n_q_heads, int max_kv_len, float sm_scale, void* O,
                           float* lse, int32_t* dev_err, void* ws, size_t ws_bytes,
                           e3_stream_t stream);
E3_API size_t eagle3_verify_workspace_bytes(int B, int R, int n_q_heads, int n_kv_heads,
                                     int head_dim, int max_kv_len, e3_dtype dt);

/* ---------------------------------------------------------------------------
 * lmhead_logits: logits[m][v] = sum_j h[m][j] W_lm[v][j] (fp32 accumulation),
 * then the softmax statistics of each row at temperature T = temp_per_row[m]:
 *   s_v = z_v * (1/T) (s_v = z_v when T <= 0), row_max[m] = max s,
 *   row_argmax[m] = argmax s (lowest id on ties),
 *   row_Q[m] = sum_v floor(2^40 E(s_v - row_max)) (fixed-point recipe).
 * h: [M][d] dtype dt; W_lm: [V][d] dtype dt; temp_per_row: [M] fp32;
 * logits: [M][V] fp32; row_max [M] fp32; row_Q [M] uint64; row_argmax [M] int32.
 * Non-finite logits set E3_DEV_ERR_NONFINITE.
 * Limits: 1 <= M <= 4000000; bf16: d % 64 == 0, V % 4 == 0.
 * ------------------------------------------------------------------------- */
E3_API e3_status lmhead_logits(const void* h, const void* W_lm, int M, int d, int V,
                        const float* temp_per_row, float* logits, float* row_max,
                        uint64_t* row_Q, int32_t* row_argmax, int32_t* dev_err,
                        e3_dtype dt, e3_stream_t stream);

/* ---------------------------------------------------------------------------
 * spec_accept: accept/reject along each request's flattened tree.
 * Rows of logits/row_* are b*R + i.  temp: [B]; row statistics must have been
 * computed with temp[b] for the rows of request b.  u_acc, u_bonus: [B][R]
 * uint32 uniforms (u_acc[c] tests child c; u_bonus[u] draws the bonus at u).
 * mode E3_ACCEPT_TREE_DET (deterministic top-k children): starting at the root
 * u, for each child c of u in flattened order with token t:
 *   T > 0:  accept iff (u_acc[c] * Rmass) >> 32 < q_t,  q_t = floor(2^40 E(s_t - m_u));
 *           on reject Rmass -= q_t and t leaves the residual (Rmass starts at
 *           row_Q[u] at every node);
 *   T <= 0: accept iff t == row_argmax[u].
 * An accepted child becomes u.  When no child of u is accepted (or u is a
 * leaf), the bonus token is drawn at u: greedy -> row_argmax[u]; sampled ->
 * the smallest token id whose cumulative residual mass exceeds
 * (u_bonus[u] * Rmass) >> 32 (ascending token ids).
 * Outputs: acc_len [B]; path [B][D+1] (flat node ids, root first, -1 padded);
 * out_tok [B][D+1] (accepted tokens then the bonus token, -1 padded);
 * status [B] (0, or E3_DEV_ERR_* bits for that request).
 * Limits: R <= 256, D <= E3_MAX_DEPTH, depth of every node <= D.
 * ------------------------------------------------------------------------- */
#define E3_ACCEPT_TREE_DET 0
#define E3_ACCEPT_SAMPLED 1 /* children drawn from q: spec_accept_sampled (it needs q) */
E3_API e3_status spec_accept(const int32_t* tok, const int32_t* parent, int B, int R, int D,
                      const float* logits, const float* row_max, const uint64_t* row_Q,
                      const int32_t* row_argmax, int V, const float* temp,
                      const uint32_t* u_acc, const uint32_t* u_bonus, int mode,
                      int32_t* acc_len, int32_t* path, int32_t* out_tok, int32_t* status,
                      e3_stream_t stream);

/* ---------------------------------------------------------------------------
 * spec_accept_sampled: accept/reject for trees whose children were drawn from
 * the draft distribution (eagle3_expand_sampled; every candidate kept):
 * "EAGLE 系列与 DFlash", §四 DFlash, acceptance min(1, p_target / p_draft), the
 * dice rolled in order; "SpecForge…", 接受连续前缀，拒绝处进行校正.
 * At node u (T = temp[b] > 0) the target residual is held as integer masses
 * R_j = floor(2^40 E(s_j - m_u)) (total SR = row_Q[u]) and the draft residual
 * as D_j = floor(2^40 E(zq_j inv_temp - m_q)) (total SD = Q) from the q_stats
 * entry of u (slot 1 + node_cand[u]; root slot 0).  Children in flattened
 * (= draw) order, token t:
 *   D_t = 0: not a draw (the row had fewer than k tokens of positive mass), skipped;
 *   accept iff u_acc[c] * floor(D_t SR / SD) < R_t 2^32
 *     (probability min(1, p_res(t) / q_res(t)));
 *   on reject, for every j: R_j -= min(R_j, floor(D_j SR / SD)) (the residual
 *     max(0, p_res - q_res)), SR = sum R_j; then SD -= D_t, D_t = 0.
 * An accepted child becomes u (the residuals restart from its rows).  With no
 * child accepted, or at a leaf, the bonus token is the smallest token id whose
 * cumulative R exceeds (u_bonus[u] * SR) >> 32.  T <= 0: exactly spec_accept's
 * greedy rule.  Other arguments and outputs as spec_accept; node_cand from
 * tree_build_mask; q_cap = 1 + cands->cap (entries per request of q_stats).
 * Non-finite target or draft statistics set E3_DEV_ERR_NONFINITE in status[b].
 * Lifetime: q_stats entries point INTO the draft logit buffers given to
 * eagle3_expand_sampled; those rows must stay allocated and unchanged until this
 * call has run, and the entries of every node with children must come from the
 * expansions that produced this tree (a NULL row is reported, a stale one is not
 * detectable).
 * ------------------------------------------------------------------------- */
E3_API e3_status spec_accept_sampled(const int32_t* tok, const int32_t* parent,
                                     const int32_t* node_cand, int B, int R, int D,
                                     const float* logits, const float* row_max,
                                     const uint64_t* row_Q, const int32_t* row_argmax, int V,
                                     const float* temp, const e3_qstat* q_stats, int q_cap,
                                     const uint32_t* u_acc, const uint32_t* u_bonus,
                                     int32_t* acc_len, int32_t* path, int32_t* out_tok,
                                     int32_t* status, e3_stream_t stream);

/* ---------------------------------------------------------------------------
 * kv_compact: for every layer l < L, request b (P = kv_len[b]) and accepted
 * node j = 1..acc_len[b], K and V of logical slot P + path[b][j] move to slot
 * P + j (all KV heads).  Every source is read before any destination is
 * written, so a slot that is both (path [0,3,4,5]) is handled.  Afterwards
 * kv_len[b] += 1 + acc_len[b] (root + accepted tokens; the bonus token becomes
 * the next root and has no KV yet).
 * layers: host array of L descriptors (same page_table/page_size/heads/dtype in
 * all layers).  path: [B][D+1].
 * Limits: 1 <= L <= E3_MAX_LAYERS, D <= E3_MAX_DEPTH.
 * ------------------------------------------------------------------------- */
E3_API e3_status kv_compact(const e3_kv_layer* layers, int L, int B, const int32_t* path,
                     const int32_t* acc_len, int D, int32_t* kv_len, int32_t* dev_err,
                     e3_stream_t stream);

/* ---------------------------------------------------------------------------
 * eagle3_draft_step: one step of the drafter -- a single decoder layer -- for
 * the frontier rows of one depth of the draft tree, B requests at once.
 * "论文专题讲解：EAGLE-3", 推理流程：多层特征融合 + 单层 draft decoder (one decoder
 * layer; the first step reads the fused feature g and the token's embedding,
 * later steps the drafter's own previous output a) and 方法主线：为什么叫
 * Training-time Test; "SpecForge…", 第二步为什么没有"正确隐藏状态"可用 and 从序列
 * 到动态草稿树 (a node attends to its ancestors only).
 * Row f of request b at depth t (1-based), node u = frontier[b][f] (a candidate
 * index of cands; -1 = the root, the only row at t = 1):
 *   tok = root_tok[b] (t = 1) or cands->tok[b][u];
 *   h   = g[b] (t = 1) or a of u's parent (a_slots[b][parent's slot]);
 *   x = W_in [e(tok); h];  y = RMSNorm(x) norm1;  [q; k; v] = W_qkv y, rotary
 *   position pos = kv_len[b] + t - 1 applied to q and k (dimension i paired with
 *   i + hd/2, angle pos * rope_base^(-2i/hd));  o = attention of q over the
 *   drafter's cache: prefix [0, kv_len[b]) and the tree slots of u's ancestors
 *   and u (scale 1/sqrt(hd));  x += W_o o;  y = RMSNorm(x) norm2;
 *   a = x + W_down (silu(W_gate y) * W_up y);
 *   logits = W_lm (RMSNorm(a) norm_f) with lmhead_logits' row statistics at T = 1.
 *   RMSNorm(x) = x / sqrt(mean(x^2) + eps).
 * Slots: u gets tree slot s = slot_base + f: its k and v go to logical position
 *   kv_len[b] + s of the drafter's cache, its a (fp32) to a_slots[b][s], its mask
 *   row to mask[b][s] = mask[b][parent's slot] | bit s.  The parent's slot is
 *   slot_base_prev + f' where frontier_prev[b][f'] = cands->parent[b][u].  At t = 1
 *   every mask row is reset to its own bit.
 * Layouts (device; bf16 weights row-major, K innermost):
 *   drafter (host struct) as e3_drafter; drafter_kv: the drafter's paged cache
 *   (bf16, head_dim hd, n_kv_heads KVH; pages for kv_len[b] + R_slots tokens);
 *   frontier [B][F], frontier_prev [B][F_prev] int32; root_tok [B]; g [B][d] bf16;
 *   a_slots [B][R_slots][d] fp32 and mask [B][R_slots][ceil(R_slots/64)] uint64
 *   (kept by the caller across the depths of one tree); logits [B][F][V] fp32
 *   (the rows eagle3_expand reads), row_max/row_Q/row_argmax [B*F].
 * ws: eagle3_draft_workspace_bytes(drafter, B, F_max, R_slots, max_kv_len) bytes.
 * Limits: bf16; d, H*hd, ffn multiples of 128; hd even; R_slots <= 256;
 *   1 <= t <= E3_MAX_DEPTH; slot_base + F <= R_slots; B*F <= 1024.
 * dev_err: E3_DEV_ERR_CAPACITY (pages, a parent not in the previous frontier),
 *   E3_DEV_ERR_TIMEOUT.
 * ------------------------------------------------------------------------- */
typedef struct {
  const void* emb;      /* [V][d]: token embedding */
  const void* W_in;     /* [d][2d]: input projection of [e(tok); h] */
  const float* norm1;   /* [d] */
  const void* W_qkv;    /* [(H + 2 KVH) hd][d]: rows of W_q, then W_k, then W_v */
  const void* W_o;      /* [d][H hd] */
  const float* norm2;   /* [d] */
  const void* W_gu;     /* [2 ffn][d]: rows of W_gate, then W_up */
  const void* W_down;   /* [d][ffn] */
  const float* norm_f;  /* [d] */
  const void* W_lm;     /* [V][d] */
  int d, n_heads, n_kv_heads, head_dim, ffn, V;
  float rope_base, eps;
} e3_drafter;
E3_API e3_status eagle3_draft_step(const e3_drafter* drafter, const e3_kv_layer* drafter_kv,
                                   const int32_t* kv_len, int max_kv_len, int B, int depth, int F,
                                   const int32_t* frontier, int slot_base, int F_prev,
                                   const int32_t* frontier_prev, int slot_base_prev, int R_slots,
                                   const e3_cand* cands, const int32_t* root_tok, const void* g,
                                   float* a_slots, uint64_t* mask, float* logits, float* row_max,
                                   uint64_t* row_Q, int32_t* row_argmax, void* ws, size_t ws_bytes,
                                   int32_t* dev_err, e3_stream_t stream);
E3_API size_t eagle3_draft_workspace_bytes(const e3_drafter* drafter, int B, int F_max, int R_slots,
                                           int max_kv_len);

/* ---------------------------------------------------------------------------
 * Adaptive draft-tree budget for a serving loop (host code only: no device
 * memory, no stream, no kernel).
 * "Thinking Budget 与 EAGLE-3", 服务端应怎样联合控制 (the execution controller):
 * the speculative budget -- never the target's decoding -- is lowered when the
 * recent accepted length is low or drafting is costly, raised cautiously when
 * acceptance is stable and verification has spare capacity, always within
 * bounds, behind a cool-down window and with a fallback baseline.  The budget is
 * a ladder of tree shapes, cheapest first ("论文专题讲解：EAGLE-3", Draft tree 配置:
 * a node budget and a depth).
 *
 * Per request (state entry b, all host memory, owned by the caller):
 *   mean <- mean + alpha (a - mean),  dev <- dev + alpha (|a - mean_old| - dev)
 * with a = acc_len[b] (drafted tokens accepted in the round just run at the
 * request's level).  While hold > 0 it counts down and the level stays.  Else,
 * after `warmup` rounds at the level, with D = depth[level]:
 *   lower one level (not below min_level) if mean < low D or draft_cost > max_draft_cost;
 *   raise one level (not above max_level) if mean >= high D, dev <= spread D,
 *     spare >= min_spare and draft_cost <= max_draft_cost;
 * a change sets hold = cooldown and restarts the round count.  An observation
 * outside [0, depth[level]] (a finished or failed request) or a state outside the
 * bounds resets the entry to the baseline (base_level, mean midway between the
 * thresholds).  spare: the verify step's free capacity as a fraction in [0, 1]
 * (the caller's measure, e.g. 1 - verify share of the step budget); draft_cost:
 * the drafting share of the round time.  level[b] receives the new level.
 * Errors: E3_ERR_INVALID_ARG / E3_ERR_SHAPE for bad policies or pointers.
 * ------------------------------------------------------------------------- */
#define E3_MAX_BUDGET_LEVELS 16
typedef struct {
  int n_levels;                        /* ladder length, 1 .. E3_MAX_BUDGET_LEVELS */
  int nodes[E3_MAX_BUDGET_LEVELS];     /* node budget N of each level (non-decreasing) */
  int depth[E3_MAX_BUDGET_LEVELS];     /* tree depth D of each level (non-decreasing, <= N) */
  int min_level, max_level;            /* bounds */
  int base_level;                      /* fallback baseline, within the bounds */
  float alpha;                         /* weight of the newest round, (0, 1] */
  float low, high;                     /* 0 <= low <= high <= 1, fractions of the depth */
  float spread;                        /* stability bound on dev, fraction of the depth */
  float min_spare;                     /* spare verify capacity needed to raise */
  float max_draft_cost;                /* drafting share above which the budget falls */
  int cooldown;                        /* rounds a new level is held (>= 0) */
  int warmup;                          /* rounds at a level before it may change (>= 1) */
} e3_budget_policy;
typedef struct {
  int32_t level, hold, rounds;
  float mean, dev;
} e3_budget_state;
E3_API e3_status eagle3_budget_init(const e3_budget_policy* pol, e3_budget_state* st, int B);
E3_API e3_status eagle3_budget_update(const e3_budget_policy* pol, e3_budget_state* st, int B,
                                      const int32_t* acc_len, float spare, float draft_cost,
                                      int32_t* level);

/* Last error message of the calling thread ("" if none). */
E3_API const char* eagle3_last_error(void);

/* ABI version: 3 (2 had no e3_kv_layer.flags and no budget controller; 1 had no
 * sampled-draft calls and no node_cand output). */
E3_API int eagle3_abi_version(void);

/* Diagnostic with no counterpart in the method: the number of kernels this
 * library has launched in the calling process since it was loaded (summed over
 * threads; a launch counts once its launch call has succeeded, whether or not
 * the kernel has run yet).  Read it before and after a sequence of calls to
 * learn how many kernels the sequence enqueued.  Never fails. */
E3_API uint64_t eagle3_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE3_H */
