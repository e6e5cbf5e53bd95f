// k_tree.cu -- tree_build_mask: rerank, flatten, positions, ancestor bit mask.
//
// "EAGLE 系列与 DFlash", §二 EAGLE-2 阶段二: the tree is flattened to one
// sequence [x_1, x_2, x_3, x_1a, x_1b, x_1c, x_2a, ...]; 关键新增步骤① gives every
// node a position from its depth; 关键新增步骤② builds the 0/1 tree mask in which
// x_1a sees only x_1 and the root, never its cousin x_2.
// "SpecForge…", 从序列到动态草稿树: the node budget goes to the most confident
// candidates.
//
// One CTA per request: bitonic sort of the candidate keys (score desc, index
// asc) in shared memory; the first N are kept.  Flat indices are assigned
// depth by depth with a parallel rank count on (parent's flat index, candidate
// index); each mask row is the OR of the bits on its ancestor walk.
#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kTreeThreads = 256;

__global__ void __launch_bounds__(kTreeThreads)
tree_build_kernel(e3_cand c, int n_cand, int N, const int32_t* __restrict__ root_tok,
                  const int32_t* __restrict__ kv_len, int32_t* tok, int32_t* parent, int32_t* depth,
                  int32_t* pos, uint64_t* mask) {
  extern __shared__ uint64_t sh[];
  uint64_t* keys = sh;                                       // [np]
  const int b = blockIdx.x;
  int np = 1;
  while (np < n_cand) np <<= 1;
  int16_t* flat_of = reinterpret_cast<int16_t*>(keys + np);  // [n_cand]
  __shared__ int kc[E3_MAX_NODES], kd[E3_MAX_NODES], pfl[E3_MAX_NODES];
  __shared__ int pflat[E3_MAX_NODES + 1];
  __shared__ int cnt[E3_MAX_DEPTH + 2], base[E3_MAX_DEPTH + 2];

  const size_t cb = static_cast<size_t>(b) * c.cap;
  for (int i = threadIdx.x; i < np; i += blockDim.x)
    keys[i] = i < n_cand ? pack_best(c.score[cb + i], static_cast<uint32_t>(i)) : 0ull;
  for (int i = threadIdx.x; i < n_cand; i += blockDim.x) flat_of[i] = -1;
  if (threadIdx.x < E3_MAX_DEPTH + 2) cnt[threadIdx.x] = 0;
  __syncthreads();
  block_bitonic_desc(keys, np);

  const int R = N + 1;
  const int P = kv_len[b];
  const int i = threadIdx.x;
  int my_c = -1, my_d = 0, my_p = -1;
  if (i < N) {
    my_c = static_cast<int>(packed_id(keys[i]));
    my_d = c.depth[cb + my_c];
    my_p = c.parent[cb + my_c];
    if (my_p >= n_cand) my_p = -1;  // malformed parent: hang the node off the root
    if (my_d < 1) my_d = 1;
    if (my_d > E3_MAX_DEPTH) my_d = E3_MAX_DEPTH;
    kc[i] = my_c;
    kd[i] = my_d;
    atomicAdd(&cnt[my_d], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 1;
    for (int d = 1; d <= E3_MAX_DEPTH; ++d) {
      base[d] = acc;
      acc += cnt[d];
    }
    pflat[0] = -1;
  }
  __syncthreads();
  for (int d = 1; d <= E3_MAX_DEPTH; ++d) {
    if (cnt[d] == 0) continue;  // uniform across the block
    if (i < N && my_d == d) {
      int pf = my_p < 0 ? 0 : flat_of[my_p];
      if (pf < 0) pf = 0;  // parent not kept: cannot happen for expansion scores
      pfl[i] = pf;
    }
    __syncthreads();
    if (i < N && my_d == d) {
      const int pf = pfl[i];
      int rank = 0;
      for (int j = 0; j < N; ++j) {
        if (kd[j] != d) continue;
        const int pj = pfl[j];
        rank += (pj < pf) || (pj == pf && kc[j] < my_c);
      }
      const int fl = base[d] + rank;
      flat_of[my_c] = static_cast<int16_t>(fl);
      pflat[fl] = pf;
      const size_t o = static_cast<size_t>(b) * R + fl;
      tok[o] = c.tok[cb + my_c];
      parent[o] = pf;
      depth[o] = d;
      pos[o] = P + d;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const size_t o = static_cast<size_t>(b) * R;
    tok[o] = root_tok[b];
    parent[o] = -1;
    depth[o] = 0;
    pos[o] = P;
  }
  // ancestor-or-self bit rows
  const int words = (R + 63) >> 6;
  if (i < R) {
    uint64_t w[4] = {0ull, 0ull, 0ull, 0ull};
    int j = i;
    for (int step = 0; step <= E3_MAX_DEPTH && j >= 0; ++step) {
      w[j >> 6] |= 1ull << (j & 63);
      j = pflat[j];
    }
    uint64_t* row = mask + (static_cast<size_t>(b) * R + i) * words;
    for (int q = 0; q < words; ++q) row[q] = w[q];
  }
}

}  // namespace

e3_status launch_tree_build(const e3_cand& c, int B, int n_cand, int N, const int32_t* root_tok,
                            const int32_t* kv_len, int32_t* tok, int32_t* parent, int32_t* depth,
                            int32_t* pos, uint64_t* mask, cudaStream_t s) {
  int np = 1;
  while (np < n_cand) np <<= 1;
  const size_t smem = static_cast<size_t>(np) * 8 + static_cast<size_t>(n_cand) * 2 + 16;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e, "tree_build_kernel smem attribute");
  }
  tree_build_kernel<<<B, kTreeThreads, smem, s>>>(c, n_cand, N, root_tok, kv_len, tok, parent, depth,
                                                  pos, mask);
  E3_LAUNCH_CHECK("tree_build_kernel");
  return E3_OK;
}

}  // namespace e3
