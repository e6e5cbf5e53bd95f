// capi.cu -- the extern "C" entry points of libeagle3 (declared in include/eagle3.h).
// Host-side validation happens here, before any launch; kernels live in k_*.cu.
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

static thread_local char g_err[512] = {0};

// Kernels this library has launched in this process (every launch site calls
// note_launch() once the launch call has succeeded).
static std::atomic<unsigned long long> g_launches{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

void clear_error() { g_err[0] = 0; }

e3_status cuda_status(cudaError_t e, const char* what) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  return E3_ERR_CUDA;
}

static bool valid_dtype(e3_dtype dt) { return dt == E3_F32 || dt == E3_BF16; }

static e3_status check_kv_layer(const e3_kv_layer* kv, const char* fn) {
  E3_REQUIRE(kv != nullptr, E3_ERR_INVALID_ARG, "%s: null kv descriptor", fn);
  E3_REQUIRE(kv->k && kv->v && kv->page_table, E3_ERR_INVALID_ARG, "%s: null k/v/page_table", fn);
  E3_REQUIRE(valid_dtype(kv->dt), E3_ERR_INVALID_ARG, "%s: bad dtype %d", fn, static_cast<int>(kv->dt));
  E3_REQUIRE(kv->n_pages > 0 && kv->max_pages > 0 && kv->n_kv_heads > 0, E3_ERR_SHAPE,
             "%s: n_pages, max_pages, n_kv_heads must be positive", fn);
  E3_REQUIRE(kv->page_size > 0 && kv->page_size % 16 == 0, E3_ERR_SHAPE, "%s: page_size %d not a multiple of 16",
             fn, kv->page_size);
  E3_REQUIRE(kv->head_dim >= 32 && kv->head_dim <= 256 && kv->head_dim % 32 == 0, E3_ERR_SHAPE,
             "%s: head_dim %d must be a multiple of 32 in [32, 256]", fn, kv->head_dim);
  E3_REQUIRE(aligned16(kv->k) && aligned16(kv->v), E3_ERR_INVALID_ARG, "%s: k/v not 16-byte aligned", fn);
  E3_REQUIRE((kv->flags & ~(E3_KV_PREFIX_STABLE | E3_KV_SELFTEST_STALL)) == 0, E3_ERR_INVALID_ARG,
             "%s: unknown kv flags %#x", fn, kv->flags);
  return E3_OK;
}

}  // namespace e3

using namespace e3;

extern "C" {

E3_API const char* eagle3_last_error(void) { return g_err; }

E3_API int eagle3_abi_version(void) { return 3; }

E3_API uint64_t eagle3_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

static bool fuse_uses_tc(int d, int d_out, e3_dtype dt) { return dt == E3_BF16 && d % 64 == 0 && d_out >= 1; }

E3_API size_t eagle3_fuse_workspace_bytes(int M, int d, int d_out, e3_dtype dt) {
  if (M < 1 || d < 1 || d_out < 1) return 0;
  return fuse_uses_tc(d, d_out, dt) ? tc_fuse_workspace_bytes(M, d, d_out) : 0;
}

E3_API e3_status eagle3_fuse(const void* h_low, const void* h_mid, const void* h_high, const void* W_f,
                             const float* bias, void* g, int M, int d, int d_out, e3_dtype dt, void* ws,
                             size_t ws_bytes, int32_t* dev_err, e3_stream_t stream) {
  g_err[0] = 0;
  E3_REQUIRE(h_low && h_mid && h_high && W_f && g, E3_ERR_INVALID_ARG, "eagle3_fuse: null pointer");
  E3_REQUIRE(valid_dtype(dt), E3_ERR_INVALID_ARG, "eagle3_fuse: bad dtype");
  E3_REQUIRE(M >= 1 && M <= 65536 && d >= 1 && d_out >= 1, E3_ERR_SHAPE, "eagle3_fuse: bad sizes M=%d d=%d d_out=%d",
             M, d, d_out);
  E3_REQUIRE(static_cast<long>(d) * 3 < (1L << 30), E3_ERR_SHAPE, "eagle3_fuse: d too large");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fuse_uses_tc(d, d_out, dt)) {
    E3_REQUIRE(aligned16(h_low) && aligned16(h_mid) && aligned16(h_high) && aligned16(W_f), E3_ERR_INVALID_ARG,
               "eagle3_fuse: bf16 operands must be 16-byte aligned");
    return launch_fuse_tc(h_low, h_mid, h_high, W_f, bias, g, M, d, d_out, ws, ws_bytes, dev_err, s);
  }
  return launch_gemm_simt(h_low, h_mid, h_high, d, W_f, bias, g, dt == E3_F32, M, d_out, 3 * d, dt, s);
}

static e3_status check_expand(const char* fn, const float* draft_logits, int B, int F, int V, int k, int W,
                              float inv_temp, const float* parent_score, const int32_t* parent_id, int depth,
                              int cand_offset, const e3_cand* cands, int32_t* next_id, float* next_score) {
  E3_REQUIRE(draft_logits && parent_score && parent_id && cands && next_id && next_score, E3_ERR_INVALID_ARG,
             "%s: null pointer", fn);
  E3_REQUIRE(cands->tok && cands->parent && cands->score && cands->depth, E3_ERR_INVALID_ARG,
             "%s: null candidate array", fn);
  E3_REQUIRE(B >= 1 && F >= 1 && V >= 1, E3_ERR_SHAPE, "%s: B, F, V must be positive", fn);
  E3_REQUIRE(k >= 1 && k <= E3_MAX_TOPK && k <= V, E3_ERR_SHAPE, "%s: k=%d out of [1, min(%d, V)]", fn, k,
             E3_MAX_TOPK);
  E3_REQUIRE(F * k <= 2048, E3_ERR_SHAPE, "%s: F*k=%d > 2048", fn, F * k);
  E3_REQUIRE(W >= 1 && (W <= E3_MAX_FRONTIER || W >= F * k), E3_ERR_SHAPE, "%s: W=%d", fn, W);
  E3_REQUIRE(depth >= 1 && depth <= E3_MAX_DEPTH, E3_ERR_SHAPE, "%s: depth=%d", fn, depth);
  E3_REQUIRE(cands->cap >= 1 && cands->cap <= E3_MAX_CAND, E3_ERR_SHAPE, "%s: cap=%d", fn, cands->cap);
  E3_REQUIRE(cand_offset >= 0 && cand_offset + F * k <= cands->cap, E3_ERR_CAPACITY,
             "%s: cand_offset %d + F*k %d exceeds cap %d", fn, cand_offset, F * k, cands->cap);
  E3_REQUIRE(static_cast<long>(B) * F <= 2147483647L / 1, E3_ERR_SHAPE, "%s: too many rows", fn);
  E3_REQUIRE(inv_temp > 0.0f && inv_temp < 1e30f, E3_ERR_INVALID_ARG, "%s: inv_temp must be > 0", fn);
  return E3_OK;
}

E3_API e3_status eagle3_expand(const float* draft_logits, int B, int F, int V, int k, int W, float inv_temp,
                        const float* parent_score, const int32_t* parent_id, int depth, int cand_offset,
                        const e3_cand* cands, int32_t* next_id, float* next_score, int32_t* dev_err,
                        e3_stream_t stream) {
  g_err[0] = 0;
  const e3_status st = check_expand("eagle3_expand", draft_logits, B, F, V, k, W, inv_temp, parent_score, parent_id,
                                    depth, cand_offset, cands, next_id, next_score);
  if (st != E3_OK) return st;
  return launch_expand(draft_logits, B, F, V, k, W, inv_temp, parent_score, parent_id, depth, cand_offset,
                       *cands, next_id, next_score, false, 0ull, nullptr, dev_err,
                       reinterpret_cast<cudaStream_t>(stream));
}

E3_API e3_status eagle3_expand_sampled(const float* draft_logits, int B, int F, int V, int k, int W, float inv_temp,
                                       const float* parent_score, const int32_t* parent_id, int depth,
                                       int cand_offset, const e3_cand* cands, int32_t* next_id, float* next_score,
                                       uint64_t seed, e3_qstat* q_stats, int32_t* dev_err, e3_stream_t stream) {
  g_err[0] = 0;
  const e3_status st = check_expand("eagle3_expand_sampled", draft_logits, B, F, V, k, W, inv_temp, parent_score,
                                    parent_id, depth, cand_offset, cands, next_id, next_score);
  if (st != E3_OK) return st;
  E3_REQUIRE(q_stats, E3_ERR_INVALID_ARG, "eagle3_expand_sampled: null q_stats");
  E3_REQUIRE(V < (1 << 24) && F < 4096 && B < (1 << 20), E3_ERR_SHAPE,
             "eagle3_expand_sampled: V=%d F=%d B=%d beyond the draw counter's fields", V, F, B);
  return launch_expand(draft_logits, B, F, V, k, W, inv_temp, parent_score, parent_id, depth, cand_offset,
                       *cands, next_id, next_score, true, seed, q_stats, dev_err,
                       reinterpret_cast<cudaStream_t>(stream));
}

E3_API e3_status tree_build_mask(const e3_cand* cands, int B, int n_cand, int N, const int32_t* root_tok,
                          const int32_t* kv_len, int32_t* tok, int32_t* parent, int32_t* depth, int32_t* pos,
                          uint64_t* mask, int32_t* node_cand, e3_stream_t stream) {
  g_err[0] = 0;
  E3_REQUIRE(cands && root_tok && kv_len && tok && parent && depth && pos && mask, E3_ERR_INVALID_ARG,
             "tree_build_mask: null pointer");
  E3_REQUIRE(cands->tok && cands->parent && cands->score && cands->depth, E3_ERR_INVALID_ARG,
             "tree_build_mask: null candidate array");
  E3_REQUIRE(B >= 1, E3_ERR_SHAPE, "tree_build_mask: B=%d", B);
  E3_REQUIRE(n_cand >= 1 && n_cand <= cands->cap && cands->cap <= E3_MAX_CAND, E3_ERR_SHAPE,
             "tree_build_mask: n_cand=%d cap=%d", n_cand, cands->cap);
  E3_REQUIRE(N >= 1 && N <= n_cand && N <= E3_MAX_NODES, E3_ERR_SHAPE, "tree_build_mask: N=%d (n_cand=%d, max %d)",
             N, n_cand, E3_MAX_NODES);
  return launch_tree_build(*cands, B, n_cand, N, root_tok, kv_len, tok, parent, depth, pos, mask, node_cand,
                           reinterpret_cast<cudaStream_t>(stream));
}

E3_API size_t eagle3_verify_workspace_bytes(int B, int R, int n_q_heads, int n_kv_heads, int head_dim, int max_kv_len,
                                     e3_dtype dt) {
  if (B < 1 || R < 1 || n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1 || max_kv_len < 0) return 0;
  return verify_workspace_bytes(B, R, n_q_heads, n_kv_heads, head_dim, max_kv_len,
                                verify_uses_mma(dt, head_dim));
}

E3_API e3_status tree_verify_attn(const void* Q, const e3_kv_layer* kv, const int32_t* kv_len, const uint64_t* mask, int B,
                           int R, int n_q_heads, int max_kv_len, float sm_scale, void* O, float* lse,
                           int32_t* dev_err, void* ws, size_t ws_bytes, e3_stream_t stream) {
  g_err[0] = 0;
  e3_status st = check_kv_layer(kv, "tree_verify_attn");
  if (st != E3_OK) return st;
  E3_REQUIRE(Q && kv_len && mask && O && lse, E3_ERR_INVALID_ARG, "tree_verify_attn: null pointer");
  E3_REQUIRE(B >= 1 && R >= 1 && R <= E3_MAX_NODES + 1, E3_ERR_SHAPE, "tree_verify_attn: B=%d R=%d", B, R);
  E3_REQUIRE(n_q_heads >= 1 && n_q_heads % kv->n_kv_heads == 0, E3_ERR_SHAPE,
             "tree_verify_attn: n_q_heads %d not a multiple of n_kv_heads %d", n_q_heads, kv->n_kv_heads);
  E3_REQUIRE(max_kv_len >= 0, E3_ERR_SHAPE, "tree_verify_attn: max_kv_len=%d", max_kv_len);
  E3_REQUIRE(static_cast<long>(max_kv_len) + R <= static_cast<long>(kv->max_pages) * kv->page_size,
             E3_ERR_CAPACITY, "tree_verify_attn: max_kv_len + R = %d exceeds max_pages*page_size = %d",
             max_kv_len + R, kv->max_pages * kv->page_size);
  E3_REQUIRE(sm_scale > 0.0f && sm_scale < 1e30f, E3_ERR_INVALID_ARG, "tree_verify_attn: sm_scale must be > 0");
  if (kv->dt == E3_BF16) {
    E3_REQUIRE(aligned16(Q), E3_ERR_INVALID_ARG, "tree_verify_attn: Q not 16-byte aligned");
  }
  return launch_verify(Q, *kv, kv_len, mask, B, R, n_q_heads, max_kv_len, sm_scale, O, lse, dev_err, ws, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

E3_API e3_status lmhead_logits(const void* h, const void* W_lm, int M, int d, int V, const float* temp_per_row,
                        float* logits, float* row_max, uint64_t* row_Q, int32_t* row_argmax, int32_t* dev_err,
                        e3_dtype dt, e3_stream_t stream) {
  g_err[0] = 0;
  E3_REQUIRE(h && W_lm && temp_per_row && logits && row_max && row_Q && row_argmax, E3_ERR_INVALID_ARG,
             "lmhead_logits: null pointer");
  E3_REQUIRE(valid_dtype(dt), E3_ERR_INVALID_ARG, "lmhead_logits: bad dtype");
  E3_REQUIRE(M >= 1 && M <= 4000000 && d >= 1 && V >= 1, E3_ERR_SHAPE, "lmhead_logits: M=%d d=%d V=%d", M, d, V);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == E3_BF16 && d % 64 == 0 && V % 4 == 0 && aligned16(logits)) {
    E3_REQUIRE(aligned16(h) && aligned16(W_lm), E3_ERR_INVALID_ARG, "lmhead_logits: bf16 operands must be 16-byte aligned");
    return launch_lmhead_tc(h, W_lm, M, d, V, temp_per_row, logits, row_max, row_Q, row_argmax, dev_err, s);
  }
  e3_status st = launch_gemm_simt(h, h, h, d, W_lm, nullptr, logits, true, M, V, d, dt, s);
  if (st != E3_OK) return st;
  return launch_row_stats(logits, M, V, temp_per_row, row_max, row_Q, row_argmax, dev_err, s);
}

E3_API e3_status spec_accept(const int32_t* tok, const int32_t* parent, int B, int R, int D, const float* logits,
                      const float* row_max, const uint64_t* row_Q, const int32_t* row_argmax, int V,
                      const float* temp, const uint32_t* u_acc, const uint32_t* u_bonus, int mode,
                      int32_t* acc_len, int32_t* path, int32_t* out_tok, int32_t* status, e3_stream_t stream) {
  g_err[0] = 0;
  E3_REQUIRE(tok && parent && logits && row_max && row_Q && row_argmax && temp && u_acc && u_bonus && acc_len &&
                 path && out_tok && status,
             E3_ERR_INVALID_ARG, "spec_accept: null pointer");
  E3_REQUIRE(mode != E3_ACCEPT_SAMPLED, E3_ERR_UNSUPPORTED,
             "spec_accept: E3_ACCEPT_SAMPLED needs the draft statistics: call spec_accept_sampled");
  E3_REQUIRE(mode == E3_ACCEPT_TREE_DET, E3_ERR_UNSUPPORTED, "spec_accept: mode %d not supported", mode);
  E3_REQUIRE(B >= 1 && R >= 1 && R <= E3_MAX_NODES + 1, E3_ERR_SHAPE, "spec_accept: B=%d R=%d", B, R);
  E3_REQUIRE(D >= 0 && D <= E3_MAX_DEPTH, E3_ERR_SHAPE, "spec_accept: D=%d", D);
  E3_REQUIRE(V >= 1, E3_ERR_SHAPE, "spec_accept: V=%d", V);
  return launch_accept(tok, parent, B, R, D, logits, row_max, row_Q, row_argmax, V, temp, u_acc, u_bonus, acc_len,
                       path, out_tok, status, reinterpret_cast<cudaStream_t>(stream));
}

E3_API e3_status spec_accept_sampled(const int32_t* tok, const int32_t* parent, const int32_t* node_cand, int B, int R,
                                     int D, const float* logits, const float* row_max, const uint64_t* row_Q,
                                     const int32_t* row_argmax, int V, const float* temp, const e3_qstat* q_stats,
                                     int q_cap, const uint32_t* u_acc, const uint32_t* u_bonus, int32_t* acc_len,
                                     int32_t* path, int32_t* out_tok, int32_t* status, e3_stream_t stream) {
  g_err[0] = 0;
  E3_REQUIRE(tok && parent && node_cand && logits && row_max && row_Q && row_argmax && temp && q_stats && u_acc &&
                 u_bonus && acc_len && path && out_tok && status,
             E3_ERR_INVALID_ARG, "spec_accept_sampled: null pointer");
  E3_REQUIRE(B >= 1 && R >= 1 && R <= E3_MAX_NODES + 1, E3_ERR_SHAPE, "spec_accept_sampled: B=%d R=%d", B, R);
  E3_REQUIRE(D >= 0 && D <= E3_MAX_DEPTH, E3_ERR_SHAPE, "spec_accept_sampled: D=%d", D);
  E3_REQUIRE(V >= 1 && V < (1 << 24), E3_ERR_SHAPE, "spec_accept_sampled: V=%d", V);
  E3_REQUIRE(q_cap >= 1 && q_cap <= E3_MAX_CAND + 1, E3_ERR_SHAPE, "spec_accept_sampled: q_cap=%d", q_cap);
  return launch_accept_sampled(tok, parent, node_cand, B, R, D, logits, row_max, row_Q, row_argmax, V, temp, q_stats,
                               q_cap, u_acc, u_bonus, acc_len, path, out_tok, status,
                               reinterpret_cast<cudaStream_t>(stream));
}

E3_API e3_status kv_compact(const e3_kv_layer* layers, int L, int B, const int32_t* path, const int32_t* acc_len, int D,
                     int32_t* kv_len, int32_t* dev_err, e3_stream_t stream) {
  g_err[0] = 0;
  E3_REQUIRE(layers && path && acc_len && kv_len, E3_ERR_INVALID_ARG, "kv_compact: null pointer");
  E3_REQUIRE(L >= 1 && L <= E3_MAX_LAYERS, E3_ERR_SHAPE, "kv_compact: L=%d", L);
  E3_REQUIRE(B >= 1 && D >= 0 && D <= E3_MAX_DEPTH, E3_ERR_SHAPE, "kv_compact: B=%d D=%d", B, D);
  CompactLayers cl;
  memset(&cl, 0, sizeof(cl));
  for (int l = 0; l < L; ++l) {
    e3_status st = check_kv_layer(&layers[l], "kv_compact");
    if (st != E3_OK) return st;
    E3_REQUIRE(layers[l].page_table == layers[0].page_table && layers[l].page_size == layers[0].page_size &&
                   layers[l].max_pages == layers[0].max_pages && layers[l].n_kv_heads == layers[0].n_kv_heads &&
                   layers[l].head_dim == layers[0].head_dim && layers[l].dt == layers[0].dt &&
                   layers[l].n_pages == layers[0].n_pages,
               E3_ERR_SHAPE, "kv_compact: layer %d geometry differs from layer 0", l);
    cl.k[l] = layers[l].k;
    cl.v[l] = layers[l].v;
  }
  const int esz = layers[0].dt == E3_F32 ? 4 : 2;
  E3_REQUIRE((layers[0].head_dim * esz) % 16 == 0 && layers[0].head_dim * esz <= 1024, E3_ERR_SHAPE,
             "kv_compact: row of %d bytes", layers[0].head_dim * esz);
  return launch_compact(cl, layers[0], L, B, path, acc_len, D, kv_len, dev_err,
                        reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
