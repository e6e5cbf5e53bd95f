// k_expand.cu -- eagle3_expand: one depth of the EAGLE-2 dynamic draft tree.
//
// "EAGLE 系列与 DFlash", §二 EAGLE-2 阶段一: every frontier node keeps its top-K
// tokens as children; "论文专题讲解：EAGLE-3", Draft tree 配置: 10 nodes are
// chosen per expansion, by draft confidence.
//
// Kernel 1 (one 16- or 8-CTA cluster per frontier row): each CTA reads its part
// of the row once into shared memory, then builds a per-thread top-KMAX list
// (packed (value, id) keys, so ties go to the lower token id); the row maximum,
// the fixed-point mass Q and the top-k lists are combined through distributed
// shared memory; CTA 0 writes the k children.
// Kernel 2 (one CTA per request): sort the F*k children by (score desc,
// candidate index asc) in shared memory and emit the next frontier.
#include <cooperative_groups.h>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kExpandThreads = 512;
constexpr int kMaxCluster = 16;  // CTAs per frontier row (at most)
constexpr int kPreferCluster = 8;  // eight-CTA clusters keep every row of a depth in one wave

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

// One cluster of CL CTAs per frontier row (CL = 16 where the device allows
// clusters of that size, else 8).  CTA r stages chunk r of the row in shared
// memory; the row maximum, the non-finite flag, the fixed-point mass and the
// per-CTA top-k lists are exchanged through distributed shared memory.
template <int KMAX>
__global__ void __launch_bounds__(kExpandThreads)
expand_rows_kernel(const float* __restrict__ logits, int F, int V, int k, float it,
                   const float* __restrict__ parent_score, const int32_t* __restrict__ parent_id,
                   int depth, int cand_offset, e3_cand c, int32_t* dev_err, int cand_cap) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.x / CL;  // b * F + f
  const int b = row / F, f = row % F;
  const float* z = logits + static_cast<size_t>(row) * V;
  extern __shared__ float4 chunk4[];
  __shared__ uint64_t warp_lists[kExpandThreads / 32][E3_MAX_TOPK];
  __shared__ uint64_t ltop[E3_MAX_TOPK];   // this CTA's best k keys
  __shared__ uint64_t lbest;               // this CTA's best key
  __shared__ uint64_t lQ;                  // this CTA's mass
  __shared__ int lbad;
  __shared__ uint64_t red64[32];
  __shared__ int redi[32];
  __shared__ uint64_t all_top[kMaxCluster * E3_MAX_TOPK];
  __shared__ uint64_t top[E3_MAX_TOPK];
  __shared__ int s_cnt;

  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
  const int nvec = vec ? (V >> 2) : V;
  const int per = (nvec + CL - 1) / CL;
  const int v0 = min(nvec, rank * per), v1 = min(nvec, v0 + per);
  float* chunk = reinterpret_cast<float*>(chunk4);

  // stage the chunk (scaled by 1/T) in shared memory with independent, unrolled loads
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
#pragma unroll 4
    for (int q = v0 + threadIdx.x; q < v1; q += blockDim.x) {
      float4 v = __ldg(z4 + q);
      v.x = __fmul_rn(v.x, it);
      v.y = __fmul_rn(v.y, it);
      v.z = __fmul_rn(v.z, it);
      v.w = __fmul_rn(v.w, it);
      chunk4[q - v0] = v;
    }
  } else {
#pragma unroll 4
    for (int j = v0 + threadIdx.x; j < v1; j += blockDim.x) chunk[j - v0] = __fmul_rn(__ldg(z + j), it);
  }
  __syncthreads();
  const int e0 = vec ? 4 * v0 : v0;  // token id of chunk[0]
  const int n_local = vec ? 4 * (v1 - v0) : (v1 - v0);
  // (1) per-thread maximum key (value desc, token id asc) and the non-finite flag
  uint64_t tmax = 0ull;
  int bad = 0;
  for (int j = threadIdx.x; j < n_local; j += blockDim.x) {
    const float sj = chunk[j];
    bad |= !isfinite(sj);
    const uint64_t key = pack_best(sj, static_cast<uint32_t>(e0 + j));
    tmax = key > tmax ? key : tmax;
  }
  bad = block_reduce(bad, OrI(), redi);
  // (2) thr = k-th largest per-thread maximum: every element of this CTA's top k
  // is >= thr, and only threads whose maximum is >= thr can hold one
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    uint64_t v = tmax;
    for (int r = 0; r < k; ++r) {
      const uint64_t best = warp_reduce(v, MaxU64());
      if (v == best) v = 0ull;  // keys are distinct: exactly one lane (or all-zero lanes)
      if (lane == 0) warp_lists[warp][r] = best;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    uint64_t lk[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
      lk[i] = (lane < nw && i < k) ? warp_lists[lane][i] : 0ull;
    warp_merge_topk(lk, k, top);
  }
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const uint64_t thr = top[k - 1];
  // (3) candidates >= thr, then their exact ranks
  uint64_t* cand = reinterpret_cast<uint64_t*>(chunk4 + (per + 1));
  for (int j = threadIdx.x; j < n_local; j += blockDim.x) {
    const uint64_t key = pack_best(chunk[j], static_cast<uint32_t>(e0 + j));
    if (key >= thr && key != 0ull) {
      const int at = atomicAdd(&s_cnt, 1);
      if (at < cand_cap) cand[at] = key;
    }
  }
  __syncthreads();
  const int ncand = min(s_cnt, cand_cap);
  if (threadIdx.x < E3_MAX_TOPK) ltop[threadIdx.x] = 0ull;
  __syncthreads();
  for (int i = threadIdx.x; i < ncand; i += blockDim.x) {
    const uint64_t key = cand[i];
    int rank = 0;
    for (int j = 0; j < ncand; ++j) rank += cand[j] > key;
    if (rank < k) ltop[rank] = key;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    lbest = ltop[0];
    lbad = bad;
  }
  cluster.sync();  // every CTA's maximum and flag are visible
  __shared__ uint64_t s_gbest;
  __shared__ int s_gbad;
  if (warp == 0) {  // lane r gathers rank r, then a warp reduction
    uint64_t v = 0ull;
    int bd = 0;
    if (lane < CL) {
      v = *cluster.map_shared_rank(&lbest, lane);
      bd = *cluster.map_shared_rank(&lbad, lane);
    }
    v = warp_reduce(v, MaxU64());
    bd = warp_reduce(bd, OrI());
    if (lane == 0) {
      s_gbest = v;
      s_gbad = bd;
    }
  }
  __syncthreads();
  const uint64_t gbest = s_gbest;
  const int gbad = s_gbad;
  if (gbad) {
    if (rank == 0 && threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_NONFINITE);
    cluster.sync();  // nobody leaves while a peer may still read its shared memory
    return;
  }
  const float m = unord_f32(static_cast<uint32_t>(gbest >> 32));
  uint64_t Q = 0;
  for (int j = threadIdx.x; j < n_local; j += blockDim.x) Q += fx_mass(chunk[j], m);
  Q = block_reduce(Q, SumU64(), red64);
  if (threadIdx.x == 0) lQ = Q;
  cluster.sync();  // masses and top-k lists are visible
  if (rank == 0) {
    for (int i = threadIdx.x; i < CL * k; i += blockDim.x)
      all_top[i] = *cluster.map_shared_rank(&ltop[i % k], i / k);
    __shared__ uint64_t s_Qt;
    if (warp == 0) {
      uint64_t v = lane < CL ? static_cast<uint64_t>(*cluster.map_shared_rank(&lQ, lane)) : 0ull;
      v = warp_reduce(v, SumU64());
      if (lane == 0) s_Qt = v;
    }
    __syncthreads();
    const uint64_t Qt = s_Qt;
    if (warp == 0) {
      uint64_t lk[KMAX];
#pragma unroll
      for (int i = 0; i < KMAX; ++i)
        lk[i] = (static_cast<int>(threadIdx.x) < CL && i < k) ? all_top[threadIdx.x * k + i] : 0ull;
      warp_merge_topk(lk, k, top);  // top[] is free again: thr was consumed above
    }
    __syncthreads();
    if (threadIdx.x < k) {
      const int r = threadIdx.x;
      const float ell = fx_ell(Qt);
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
  cluster.sync();  // rank 0 is done reading the peers' shared memory
}

template <int KMAX>
int cluster_size_for() {
  static int cl = 0;
  if (cl == 0) {
    cl = 8;
    if (kPreferCluster == 8) return cl;
    if (cudaFuncSetAttribute(expand_rows_kernel<KMAX>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(kExpandThreads);
      cfg.dynamicSmemBytes = 64 * 1024;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 16;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, expand_rows_kernel<KMAX>, &cfg) == cudaSuccess && n > 0) cl = 16;
    }
    cudaGetLastError();
  }
  return cl;
}

template <int KMAX>
e3_status launch_rows(const float* logits, int rows, int F, int V, int k, float inv_temp, const float* parent_score,
                      const int32_t* parent_id, int depth, int cand_offset, const e3_cand& c, int32_t* dev_err,
                      cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(expand_rows_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_done = true;
  }
  const int CL = cluster_size_for<KMAX>();
  const bool vec = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  const int nvec = vec ? V / 4 : V;
  const int per = (nvec + CL - 1) / CL;
  const int per_thread = ((vec ? per * 4 : per) + kExpandThreads - 1) / kExpandThreads;
  const int cand_cap = k * per_thread + 32;
  const size_t smem = static_cast<size_t>(per + 1) * 16 + static_cast<size_t>(cand_cap) * 8 + 16;
  E3_REQUIRE(smem <= 200 * 1024, E3_ERR_SHAPE, "eagle3_expand: V=%d too large", V);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows * CL);
  cfg.blockDim = dim3(kExpandThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = CL;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, expand_rows_kernel<KMAX>, logits, F, V, k, inv_temp, parent_score,
                                     parent_id, depth, cand_offset, c, dev_err, cand_cap);
  if (e != cudaSuccess) return cuda_status(e, "expand_rows_kernel");
  return E3_OK;
}

}  // namespace

namespace {

__global__ void __launch_bounds__(256)
expand_frontier_kernel(int n, int Wn, int cand_offset, e3_cand c, int32_t* next_id, float* next_score,
                       const int32_t* dev_err) {
  __shared__ uint64_t keys[2048];
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int ci = cand_offset + i;
    keys[i] = pack_best(c.score[static_cast<size_t>(b) * c.cap + ci], static_cast<uint32_t>(ci));
  }
  __syncthreads();
  if (n <= 1024) {
    // exact rank of each child among the n (distinct keys): the first Wn ranks win
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t key = keys[i];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += keys[j] > key;
      if (rank < Wn) {
        const uint32_t ci = packed_id(key);
        next_id[static_cast<size_t>(b) * Wn + rank] = static_cast<int32_t>(ci);
        next_score[static_cast<size_t>(b) * Wn + rank] = c.score[static_cast<size_t>(b) * c.cap + ci];
      }
    }
    return;
  }
  int np = 1;
  while (np < n) np <<= 1;
  for (int i = n + threadIdx.x; i < np; i += blockDim.x) keys[i] = 0ull;
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
  e3_status st;
  if (k <= 2)
    st = launch_rows<2>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c, dev_err, s);
  else if (k <= 4)
    st = launch_rows<4>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c, dev_err, s);
  else if (k <= 8)
    st = launch_rows<8>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c, dev_err, s);
  else if (k <= 16)
    st = launch_rows<16>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c, dev_err, s);
  else
    st = launch_rows<32>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c, dev_err, s);
  if (st != E3_OK) return st;
  E3_LAUNCH_CHECK("expand_rows_kernel");
  const int n = F * k;
  const int Wn = W < n ? W : n;
  expand_frontier_kernel<<<B, 256, 0, s>>>(n, Wn, cand_offset, c, next_id, next_score, dev_err);
  E3_LAUNCH_CHECK("expand_frontier_kernel");
  return E3_OK;
}

}  // namespace e3
