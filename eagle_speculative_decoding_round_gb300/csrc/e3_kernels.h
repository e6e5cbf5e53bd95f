// e3_kernels.h -- internal launchers of libeagle3 (not part of the C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/eagle3.h"

namespace e3 {

struct CompactLayers {
  void* k[E3_MAX_LAYERS];
  void* v[E3_MAX_LAYERS];
};

e3_status launch_expand(const float* logits, int B, int F, int V, int k, int W, float inv_temp,
                        const float* parent_score, const int32_t* parent_id, int depth, int cand_offset,
                        const e3_cand& c, int32_t* next_id, float* next_score, bool sampled, uint64_t seed,
                        e3_qstat* q_stats, int32_t* dev_err, cudaStream_t s);

e3_status launch_tree_build(const e3_cand& c, int B, int n_cand, int N, const int32_t* root_tok,
                            const int32_t* kv_len, int32_t* tok, int32_t* parent, int32_t* depth, int32_t* pos,
                            uint64_t* mask, int32_t* node_cand, cudaStream_t s);

size_t verify_workspace_bytes(int B, int R, int H, int KVH, int hd, int max_kv_len, bool mma);
bool verify_uses_mma(e3_dtype dt, int hd);
e3_status launch_verify(const void* Q, const e3_kv_layer& kv, const int32_t* kv_len, const uint64_t* mask,
                        int B, int R, int H, int max_kv_len, float sm_scale, void* O, float* lse,
                        int32_t* dev_err, void* ws, size_t ws_bytes, cudaStream_t s);

// How the keys of one (request, KV head) are split across CTAs: n_pre prefix
// segments of `chunk` keys, S partial records per row; fold = 1 when the tree
// slots are processed by the last prefix segment (no separate tree segment).
struct VerifySplit {
  int n_pre, S, chunk, fold;
};
bool verify_tc_supported(const e3_kv_layer& kv, int H);
// On entry *split is the workspace's split (at most split->S records per row);
// on return, the split the partial records were written with (when not merged).
e3_status launch_verify_tc(const void* Q, const e3_kv_layer& kv, const int32_t* kv_len, const uint64_t* mask, int B,
                           int R, int H, int max_kv_len, float sm_scale, VerifySplit* split, float* ws_o,
                           float2* ws_ml, void* O, float* lse, bool* merged, int32_t* dev_err, cudaStream_t s);

e3_status launch_gemm_simt(const void* a0, const void* a1, const void* a2, int dseg, const void* W,
                           const float* bias, void* out, bool out_f32, int M, int N, int K, e3_dtype dt,
                           cudaStream_t s);
e3_status launch_row_stats(const float* logits, int M, int V, const float* temp, float* row_max,
                           uint64_t* row_Q, int32_t* row_argmax, int32_t* dev_err, cudaStream_t s);

bool tc_gemm_supported(int d_k, int n_rows);
// Split-K partial sums part[z][m][n] (fp32, z < *splits) of out[m][n] = W[n] . [src_0[m]; ..;
// src_{n_src-1}[m]] with W [N][n_src*K] and src_i [M][K] bf16 (K % 64 == 0), on the tensor cores.
int linear_splits(int M, int K_total, int N);
size_t linear_partial_bytes(int M, int K_total, int N);
e3_status launch_linear_tc(const void* W, const void* const* src, int n_src, int K, int M, int N, float* part,
                           int* splits, int32_t* dev_err, cudaStream_t s);
size_t tc_fuse_workspace_bytes(int M, int d, int d_out);
e3_status launch_fuse_tc(const void* h_low, const void* h_mid, const void* h_high, const void* W_f, const float* bias,
                         void* g, int M, int d, int d_out, void* ws, size_t ws_bytes, int32_t* dev_err,
                         cudaStream_t s);
e3_status launch_lmhead_tc(const void* h, const void* W_lm, int M, int d, int V, const float* temp, float* logits,
                           float* row_max, uint64_t* row_Q, int32_t* row_argmax, int32_t* dev_err, cudaStream_t s);

e3_status launch_accept(const int32_t* tok, const int32_t* parent, int B, int R, int D, const float* logits,
                        const float* row_max, const uint64_t* row_Q, const int32_t* row_argmax, int V,
                        const float* temp, const uint32_t* u_acc, const uint32_t* u_bonus, int32_t* acc_len,
                        int32_t* path, int32_t* out_tok, int32_t* status, cudaStream_t s);

e3_status launch_accept_sampled(const int32_t* tok, const int32_t* parent, const int32_t* node_cand, int B, int R,
                                int D, const float* logits, const float* row_max, const uint64_t* row_Q,
                                const int32_t* row_argmax, int V, const float* temp, const e3_qstat* q_stats,
                                int q_cap, const uint32_t* u_acc, const uint32_t* u_bonus, int32_t* acc_len,
                                int32_t* path, int32_t* out_tok, int32_t* status, cudaStream_t s);

e3_status launch_compact(const CompactLayers& layers, const e3_kv_layer& geo, int L, int B, const int32_t* path,
                         const int32_t* acc_len, int D, int32_t* kv_len, int32_t* dev_err, cudaStream_t s);

}  // namespace e3
