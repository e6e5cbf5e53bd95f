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
// asc), one key per thread in registers (shuffles within a warp, shared memory
// across warps); the first N are kept.  Flat indices are assigned depth by
// depth with a parallel rank count on (parent's flat index, candidate index);
// each mask row is the OR of the bits on its ancestor walk.  Optionally the
// candidate index of every flat node is written (node_cand), which is how the
// sampled accept finds the draft row a node's children were drawn from.
#include <algorithm>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kTreeThreads = 256;  // at least E3_MAX_NODES + 1 (one thread per flat row)

// Descending bitonic sort of n = blockDim.x keys (a power of two, <= 1024), one
// key per thread: partners within a warp exchange through shuffles, the others
// through two alternating shared-memory buffers (one barrier per such step).
__device__ __forceinline__ uint64_t bitonic_desc_thread(uint64_t v, uint64_t* buf /* [2][n] */) {
  const int n = blockDim.x, tid = threadIdx.x;
  int flip = 0;
  for (int kk = 2; kk <= n; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      uint64_t o;
      if (j >= 32) {
        uint64_t* b = buf + flip * n;
        b[tid] = v;
        __syncthreads();
        o = b[tid ^ j];
        flip ^= 1;
      } else {
        o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
      }
      const bool lower = (tid & j) == 0;  // the lower index of the pair keeps the larger key...
      const bool desc = (tid & kk) == 0;  // ...in the descending halves of the merge
      v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

__global__ void __launch_bounds__(1024)
tree_build_kernel(e3_cand c, int n_cand, int N, const int32_t* __restrict__ root_tok,
                  const int32_t* __restrict__ kv_len, int32_t* tok, int32_t* parent, int32_t* depth,
                  int32_t* pos, uint64_t* mask, int32_t* node_cand) {
  extern __shared__ uint64_t sh[];
  uint64_t* keys = sh;  // [2 * max(np, blockDim.x)]: the two exchange buffers, or the in-place sort
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  int np = 1;
  while (np < n_cand) np <<= 1;
  const bool per_thread = np <= static_cast<int>(blockDim.x);  // then blockDim.x == np
  int16_t* flat_of = reinterpret_cast<int16_t*>(keys + 2 * max(np, static_cast<int>(blockDim.x)));  // [n_cand]
  __shared__ int kkey[E3_MAX_NODES];  // per level: (parent flat index, candidate index) of its nodes
  __shared__ int pflat[E3_MAX_NODES + 1];
  __shared__ int cnt[E3_MAX_DEPTH + 2], base[E3_MAX_DEPTH + 2];

  const size_t cb = static_cast<size_t>(b) * c.cap;
  const int i = threadIdx.x;
  for (int q = i; q < n_cand; q += blockDim.x) flat_of[q] = -1;
  if (i < E3_MAX_DEPTH + 2) cnt[i] = 0;
  const int P = kv_len[b];
  uint64_t top;  // (thread i < N) the i-th best candidate key
  // (one key per thread) this thread's candidate's depth, parent and token, requested
  // with its score and kept in registers through the sort; after it, the kept nodes
  // read them from shared memory instead of global memory
  int pre_d = 0, pre_p = -1, pre_t = 0;
  if (per_thread) {
    uint64_t v = 0ull;
    if (i < n_cand) {
      v = pack_best(c.score[cb + i], static_cast<uint32_t>(i));
      pre_d = c.depth[cb + i];
      pre_p = c.parent[cb + i];
      pre_t = c.tok[cb + i];
    }
    top = bitonic_desc_thread(v, keys);
  } else {
    for (int q = i; q < np; q += blockDim.x)
      keys[q] = q < n_cand ? pack_best(c.score[cb + q], static_cast<uint32_t>(q)) : 0ull;
    __syncthreads();
    block_bitonic_desc(keys, np);
    top = i < np ? keys[i] : 0ull;
  }
  // the kept nodes' candidate data: staged in shared memory by the candidates' own
  // threads (per-thread sort: the exchange buffers are free again), else from global
  int* cdat = reinterpret_cast<int*>(keys);  // [3][n_cand] (needs 12 n_cand <= 16 max(np, blockDim) bytes)
  if (per_thread) {
    __syncthreads();  // every thread is done with the sort's exchange buffers
    if (i < n_cand) {
      cdat[i] = pre_d;
      cdat[n_cand + i] = pre_p;
      cdat[2 * n_cand + i] = pre_t;
    }
    __syncthreads();
  }
  int my_c = -1, my_d = 0, my_p = -1, my_tok = 0;
  if (i < N) {
    my_c = static_cast<int>(packed_id(top));
    if (per_thread) {
      my_d = cdat[my_c];
      my_p = cdat[n_cand + my_c];
      my_tok = cdat[2 * n_cand + my_c];
    } else {
      my_d = c.depth[cb + my_c];
      my_p = c.parent[cb + my_c];
      my_tok = c.tok[cb + my_c];
    }
    if (my_p >= n_cand) my_p = -1;  // malformed parent: hang the node off the root
    if (my_d < 1) my_d = 1;
    if (my_d > E3_MAX_DEPTH) my_d = E3_MAX_DEPTH;
    atomicAdd(&cnt[my_d], 1);
  }
  __syncthreads();
  if (i == 0) {
    int acc = 1;
    for (int d = 1; d <= E3_MAX_DEPTH; ++d) {
      base[d] = acc;
      acc += cnt[d];
    }
    pflat[0] = -1;
  }
  __syncthreads();
  // flat indices depth by depth: rank among the level's nodes by (parent's flat
  // index, candidate index), packed into one integer key (both below 2^12)
  int my_fl = 0, my_pf = 0;
  for (int d = 1; d <= E3_MAX_DEPTH; ++d) {
    if (cnt[d] == 0) continue;  // uniform across the block
    if (i < N) {
      int key = 0x7FFFFFFF;
      if (my_d == d) {
        int pf = my_p < 0 ? 0 : flat_of[my_p];
        if (pf < 0) pf = 0;  // parent not kept: cannot happen for expansion scores
        my_pf = pf;
        key = (pf << 12) | my_c;
      }
      kkey[i] = key;
    }
    __syncthreads();
    if (i < N && my_d == d) {
      const int mine = (my_pf << 12) | my_c;
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < N; ++j) rank += kkey[j] < mine;
      my_fl = base[d] + rank;
      flat_of[my_c] = static_cast<int16_t>(my_fl);
      pflat[my_fl] = my_pf;
    }
    __syncthreads();
  }
  const int R = N + 1;
  if (i < N) {
    const size_t o = static_cast<size_t>(b) * R + my_fl;
    tok[o] = my_tok;
    parent[o] = my_pf;
    depth[o] = my_d;
    pos[o] = P + my_d;
    if (node_cand) node_cand[o] = my_c;
  }
  if (i == 0) {
    const size_t o = static_cast<size_t>(b) * R;
    tok[o] = root_tok[b];
    parent[o] = -1;
    depth[o] = 0;
    pos[o] = P;
    if (node_cand) node_cand[o] = -1;
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
                            int32_t* pos, uint64_t* mask, int32_t* node_cand, cudaStream_t s) {
  int np = 1;
  while (np < n_cand) np <<= 1;
  // one thread per sort key up to 1024 keys (sorted in registers and shuffles),
  // else 1024 threads over a shared-memory sort
  const int threads = std::max(kTreeThreads, std::min(np, 1024));
  const size_t smem = static_cast<size_t>(std::max(np, threads)) * 16 + static_cast<size_t>(n_cand) * 2 + 16;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e, "tree_build_kernel smem attribute");
  }
  const cudaError_t e = launch_pdl(tree_build_kernel, dim3(B), dim3(threads), smem, s, 1, c, n_cand, N, root_tok, kv_len,
                                   tok, parent, depth, pos, mask, node_cand);
  if (e != cudaSuccess) return cuda_status(e, "tree_build_kernel");
  return E3_OK;
}

}  // namespace e3
