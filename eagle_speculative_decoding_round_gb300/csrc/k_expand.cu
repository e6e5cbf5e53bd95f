// k_expand.cu -- eagle3_expand: one depth of the EAGLE-2 dynamic draft tree.
//
// "EAGLE 系列与 DFlash", §二 EAGLE-2 阶段一: every frontier node keeps its top-K
// tokens as children; "论文专题讲解：EAGLE-3", Draft tree 配置: 10 nodes are
// chosen per expansion, by draft confidence.
//
// Kernel 1 (one CTA per frontier row): stream the row once for the maximum, a
// per-thread top-KMAX list (packed (value, id) keys, so ties go to the lower
// token id) and the non-finite check; merge the lists warp by warp; stream the
// row again (L2-resident) for the fixed-point mass Q; write the k children.
// Kernel 2 (one CTA per request): sort the F*k children by (score desc,
// candidate index asc) in shared memory and emit the next frontier.
#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kExpandThreads = 512;

template <int KMAX>
__device__ __forceinline__ void topk_insert(uint64_t (&keys)[KMAX], uint64_t key) {
  if (key <= keys[KMAX - 1]) return;
#pragma unroll
  for (int i = KMAX - 1; i > 0; --i) {
    if (key > keys[i - 1])
      keys[i] = keys[i - 1];
    else if (key > keys[i])
      keys[i] = key;
  }
  if (key > keys[0]) keys[0] = key;
}

// Merge the 32 sorted lists of a warp; lane 0 returns the best k in out[0..k).
template <int KMAX>
__device__ void warp_merge_topk(uint64_t (&keys)[KMAX], int k, uint64_t* out) {
  for (int r = 0; r < k; ++r) {
    uint64_t head = keys[0];
    uint64_t best = warp_reduce(head, MaxU64());
    if (head == best && best != 0ull) {
#pragma unroll
      for (int i = 0; i < KMAX - 1; ++i) keys[i] = keys[i + 1];
      keys[KMAX - 1] = 0ull;
    }
    if ((threadIdx.x & 31) == 0) out[r] = best;
  }
}

template <int KMAX>
__global__ void __launch_bounds__(kExpandThreads)
expand_rows_kernel(const float* __restrict__ logits, int F, int V, int k, float it,
                   const float* __restrict__ parent_score, const int32_t* __restrict__ parent_id,
                   int depth, int cand_offset, e3_cand c, int32_t* dev_err) {
  const int row = blockIdx.x;  // b * F + f
  const int b = row / F, f = row % F;
  const float* z = logits + static_cast<size_t>(row) * V;
  __shared__ uint64_t warp_lists[kExpandThreads / 32][E3_MAX_TOPK];
  __shared__ uint64_t red64[32];
  __shared__ int redi[32];

  uint64_t keys[KMAX];
#pragma unroll
  for (int i = 0; i < KMAX; ++i) keys[i] = 0ull;
  int bad = 0;
  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    for (int q = threadIdx.x; q < (V >> 2); q += blockDim.x) {
      float4 v = __ldg(z4 + q);
      float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        bad |= !isfinite(e[u]);
        topk_insert(keys, pack_best(__fmul_rn(e[u], it), static_cast<uint32_t>(4 * q + u)));
      }
    }
  } else {
    for (int j = threadIdx.x; j < V; j += blockDim.x) {
      float v = __ldg(z + j);
      bad |= !isfinite(v);
      topk_insert(keys, pack_best(__fmul_rn(v, it), static_cast<uint32_t>(j)));
    }
  }
  bad = block_reduce(bad, OrI(), redi);
  if (bad) {
    if (threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_NONFINITE);
    return;
  }
  const int warp = threadIdx.x >> 5;
  warp_merge_topk(keys, k, warp_lists[warp]);
  __syncthreads();
  __shared__ uint64_t top[E3_MAX_TOPK];
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    uint64_t lk[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
      lk[i] = (static_cast<int>(threadIdx.x) < nw && i < k) ? warp_lists[threadIdx.x][i] : 0ull;
    warp_merge_topk(lk, k, top);
  }
  __syncthreads();
  const float m = unord_f32(static_cast<uint32_t>(top[0] >> 32));
  // second pass: fixed-point mass of the row
  uint64_t Q = 0;
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    for (int q = threadIdx.x; q < (V >> 2); q += blockDim.x) {
      float4 v = __ldg(z4 + q);
      Q += fx_mass(__fmul_rn(v.x, it), m) + fx_mass(__fmul_rn(v.y, it), m) +
           fx_mass(__fmul_rn(v.z, it), m) + fx_mass(__fmul_rn(v.w, it), m);
    }
  } else {
    for (int j = threadIdx.x; j < V; j += blockDim.x) Q += fx_mass(__fmul_rn(__ldg(z + j), it), m);
  }
  Q = block_reduce(Q, SumU64(), red64);
  if (threadIdx.x < k) {
    const int r = threadIdx.x;
    const float ell = fx_ell(Q);
    const uint32_t t = packed_id(top[r]);
    const float sc = unord_f32(static_cast<uint32_t>(top[r] >> 32));
    const float ps = parent_score[row];
    const size_t ci = static_cast<size_t>(b) * c.cap + cand_offset + f * k + r;
    c.tok[ci] = static_cast<int32_t>(t);
    c.parent[ci] = parent_id[row];
    c.score[ci] = __fsub_rn(__fadd_rn(ps, __fsub_rn(sc, m)), ell);
    c.depth[ci] = depth;
  }
}

}  // namespace

namespace {

__global__ void __launch_bounds__(256)
expand_frontier_kernel(int n, int Wn, int cand_offset, e3_cand c, int32_t* next_id,
                       float* next_score, const int32_t* dev_err) {
  __shared__ uint64_t keys[2048];
  const int b = blockIdx.x;
  int np = 1;
  while (np < n) np <<= 1;
  for (int i = threadIdx.x; i < np; i += blockDim.x) {
    uint64_t key = 0ull;
    if (i < n) {
      const int ci = cand_offset + i;
      key = pack_best(c.score[static_cast<size_t>(b) * c.cap + ci], static_cast<uint32_t>(ci));
    }
    keys[i] = key;
  }
  __syncthreads();
  block_bitonic_desc(keys, np);
  for (int q = threadIdx.x; q < Wn; q += blockDim.x) {
    const uint32_t ci = packed_id(keys[q]);
    next_id[static_cast<size_t>(b) * Wn + q] = static_cast<int32_t>(ci);
    next_score[static_cast<size_t>(b) * Wn + q] = c.score[static_cast<size_t>(b) * c.cap + ci];
  }
}

}  // namespace

e3_status launch_expand(const float* logits, int B, int F, int V, int k, int W, float inv_temp,
                        const float* parent_score, const int32_t* parent_id, int depth,
                        int cand_offset, const e3_cand& c, int32_t* next_id, float* next_score,
                        int32_t* dev_err, cudaStream_t s) {
  const int rows = B * F;
  dim3 grid(rows), block(kExpandThreads);
#define E3_EXPAND_CASE(KM)                                                                   \
  expand_rows_kernel<KM><<<grid, block, 0, s>>>(logits, F, V, k, inv_temp, parent_score,     \
                                                parent_id, depth, cand_offset, c, dev_err)
  if (k <= 2)
    E3_EXPAND_CASE(2);
  else if (k <= 4)
    E3_EXPAND_CASE(4);
  else if (k <= 8)
    E3_EXPAND_CASE(8);
  else if (k <= 16)
    E3_EXPAND_CASE(16);
  else
    E3_EXPAND_CASE(32);
#undef E3_EXPAND_CASE
  E3_LAUNCH_CHECK("expand_rows_kernel");
  const int n = F * k;
  const int Wn = W < n ? W : n;
  expand_frontier_kernel<<<B, 256, 0, s>>>(n, Wn, cand_offset, c, next_id, next_score, dev_err);
  E3_LAUNCH_CHECK("expand_frontier_kernel");
  return E3_OK;
}

}  // namespace e3
