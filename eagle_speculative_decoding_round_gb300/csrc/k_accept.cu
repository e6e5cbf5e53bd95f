// k_accept.cu -- spec_accept: speculative-sampling accept/reject on the tree.
//
// "EAGLE 系列与 DFlash", §四 DFlash: the target scores each draft, the
// acceptance probability is min(1, p_target / p_draft) and the dice are rolled
// left to right; §二 阶段三: the longest coherent accepted prefix is kept and
// decoding rolls back to the last accepted node.  "SpecForge…", 先看 checkpoint
// 最终要参与什么计算: correct at the rejection point so that the output follows
// the target distribution exactly.
//
// The tree's children are deterministic top-k proposals (the draft put all of
// its proposal mass on the proposed token), so min(1, p/q) becomes "accept
// child c with probability p_res(c)"; a rejected child leaves the residual
// distribution, and the next sibling is tested against what remains.  With no
// child accepted, the bonus (correction) token is drawn from the residual.
//
// One cluster of CL CTAs per request (16 where allowed, else 8).  Every CTA
// builds the children lists and each child's fixed-point mass in parallel and
// then walks the tree (integer work only).  For the bonus draw, CTA r owns a
// contiguous chunk of the vocabulary: it computes the residual masses of its
// chunk into shared memory; the chunk sums are exchanged through distributed
// shared memory; the CTA whose chunk holds the target finds the token (warp
// sums, then a warp scan of one 32-token group) and writes the request's
// outputs.
#include <cooperative_groups.h>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kAcceptThreads = 512;
constexpr int kMaxR = E3_MAX_NODES + 1;

__global__ void __launch_bounds__(kAcceptThreads)
accept_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ parent, int R, int D,
              const float* __restrict__ logits, const float* __restrict__ row_max,
              const uint64_t* __restrict__ row_Q, const int32_t* __restrict__ row_argmax, int V,
              const float* __restrict__ temp, const uint32_t* __restrict__ u_acc,
              const uint32_t* __restrict__ u_bonus, int32_t* acc_len, int32_t* path, int32_t* out_tok,
              int32_t* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / CL;
  extern __shared__ unsigned long long qbuf[];  // residual masses of this CTA's chunk
  __shared__ int s_tok[kMaxR], s_par[kMaxR], s_nch[kMaxR], s_first[kMaxR + 1], s_child[kMaxR];
  __shared__ unsigned long long s_qc[kMaxR];  // mass of child c under its parent's row
  __shared__ int s_removed[kMaxR];
  __shared__ int s_path[E3_MAX_DEPTH + 1];
  __shared__ int s_nrem, s_u, s_acc, s_err, s_bonus;
  __shared__ unsigned long long s_x, s_sum;
  __shared__ unsigned long long s_wsum[kAcceptThreads / 32];

  pdl_wait();
  pdl_trigger();
  const size_t rb = static_cast<size_t>(b) * R;
  const float T = temp[b];
  const float it = inv_temp(T);
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    s_tok[i] = tok[rb + i];
    s_par[i] = parent[rb + i];
  }
  __syncthreads();
  // children lists in CSR form (children in ascending flat order) and child masses
  for (int u = threadIdx.x; u < R; u += blockDim.x) {
    int n = 0;
    for (int c = u + 1; c < R; ++c) n += (s_par[c] == u);
    s_nch[u] = n;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int u = 0; u < R; ++u) {
      s_first[u] = acc;
      acc += s_nch[u];
    }
    s_first[R] = acc;
    s_err = 0;
    s_bonus = -1;
    s_path[0] = 0;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < R; c += blockDim.x) {
    const int p = s_par[c];
    s_qc[c] = 0ull;
    if (c == 0 || p < 0 || p >= c) continue;  // root, or not a forward edge
    int rk = 0;
    for (int c2 = p + 1; c2 < c; ++c2) rk += (s_par[c2] == p);
    s_child[s_first[p] + rk] = c;
    const int t = s_tok[c];
    if (T > 0.0f && t >= 0 && t < V) {
      const size_t prow = rb + p;
      s_qc[c] = fx_mass(__fmul_rn(logits[prow * V + t], it), row_max[prow]);
    }
  }
  __syncthreads();
  // the walk (every CTA of the cluster does it; integer work only)
  if (threadIdx.x == 0) {
    int u = 0, a = 0, nrem = 0;
    uint64_t Rm = 0;
    for (;;) {
      const size_t row = rb + u;
      const float m = row_max[row];
      const int am = row_argmax[row];
      if (am < 0 || !isfinite(m)) {
        s_err = E3_DEV_ERR_NONFINITE;
        break;
      }
      Rm = row_Q[row];
      nrem = 0;
      int accepted = -1;
      for (int e = s_first[u]; e < s_first[u] + s_nch[u]; ++e) {
        const int c = s_child[e];
        const int t = s_tok[c];
        if (T <= 0.0f) {
          if (t == am) {
            accepted = c;
            break;
          }
          continue;
        }
        if (t < 0 || t >= V) continue;
        const uint64_t q = s_qc[c];
        if (mulhi32(u_acc[rb + c], Rm) < q) {
          accepted = c;
          break;
        }
        Rm -= q;
        s_removed[nrem++] = t;
      }
      if (accepted >= 0 && a < D) {
        ++a;
        s_path[a] = accepted;
        u = accepted;
        continue;
      }
      if (T <= 0.0f) s_bonus = am;
      break;
    }
    s_u = u;
    s_acc = a;
    s_nrem = nrem;
    s_x = (T > 0.0f) ? mulhi32(u_bonus[rb + u], Rm) : 0ull;
  }
  __syncthreads();
  const int err = s_err;
  int writer = 0;  // the CTA that writes this request's outputs
  const bool sampled = !err && T > 0.0f;  // uniform across the cluster
  if (sampled) {
    const int u = s_u;
    const uint64_t x = s_x;
    const size_t row = rb + u;
    const float m = row_max[row];
    const float* z = logits + row * V;
    const int per = (V + CL - 1) / CL;
    const int j0 = min(V, rank * per), j1 = min(V, j0 + per);
    const int n = j1 - j0;
    // residual masses of the chunk (removed tokens zeroed) and the chunk sum
#pragma unroll 4
    for (int j = threadIdx.x; j < n; j += blockDim.x) qbuf[j] = fx_mass(__fmul_rn(z[j0 + j], it), m);
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 0; i < s_nrem; ++i) {
        const int t = s_removed[i];
        if (t >= j0 && t < j1) qbuf[t - j0] = 0ull;
      }
    }
    __syncthreads();
    // per-warp sums of contiguous sub-segments
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int wseg = (n + nw - 1) / nw;
    const int a0 = min(n, w * wseg), a1 = min(n, a0 + wseg);
    uint64_t local = 0;
    for (int j = a0 + lane; j < a1; j += 32) local += qbuf[j];
    local = warp_reduce(local, SumU64());
    if (lane == 0) s_wsum[w] = local;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t tot = 0;
      for (int i = 0; i < nw; ++i) tot += s_wsum[i];
      s_sum = tot;
    }
    cluster.sync();  // chunk sums visible
    uint64_t excl = 0;
    int found = -1;
    for (int r = 0; r < CL; ++r) {  // the chunk sums partition [0, Rmass)
      const uint64_t sr = *cluster.map_shared_rank(&s_sum, r);
      if (found < 0 && x >= excl && x < excl + sr) found = r;
      excl += sr;
    }
    writer = found < 0 ? 0 : found;
    if (found == rank) {
      uint64_t wex = 0;
      for (int r = 0; r < rank; ++r) wex += *cluster.map_shared_rank(&s_sum, r);
      for (int i = 0; i < w; ++i) wex += s_wsum[i];
      if (x >= wex && x < wex + s_wsum[w]) {  // uniform within the warp
        uint64_t base = wex;
        for (int c0 = a0; c0 < a1; c0 += 32) {
          const int j = c0 + lane;
          const uint64_t q = j < a1 ? qbuf[j] : 0ull;
          uint64_t incl = q;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
          }
          const unsigned hit = __ballot_sync(0xFFFFFFFFu, base + incl > x);
          if (hit) {
            if (lane == __ffs(hit) - 1) s_bonus = j0 + j;
            break;
          }
          base += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
      }
    }
    __syncthreads();
  }
  if (rank == writer && threadIdx.x == 0) {
    const int a = err ? 0 : s_acc;
    const size_t o = static_cast<size_t>(b) * (D + 1);
    for (int j = 0; j <= D; ++j) {
      path[o + j] = (!err && j <= a) ? s_path[j] : -1;
      out_tok[o + j] = -1;
    }
    if (err) {
      path[o] = 0;
    } else {
      for (int j = 1; j <= a; ++j) out_tok[o + j - 1] = s_tok[s_path[j]];
      out_tok[o + a] = s_bonus;
    }
    acc_len[b] = a;
    status[b] = err;
  }
  cluster.sync();  // peers may still read this CTA's chunk sum
}

int accept_cluster_size() {
  static int cl = 0;
  if (cl == 0) {
    cl = 8;
    if (cudaFuncSetAttribute(accept_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(kAcceptThreads);
      cfg.dynamicSmemBytes = 72 * 1024;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 16;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, accept_kernel, &cfg) == cudaSuccess && n > 0) cl = 16;
    }
    cudaGetLastError();
  }
  return cl;
}

}  // namespace

e3_status launch_accept(const int32_t* tok, const int32_t* parent, int B, int R, int D, const float* logits,
                        const float* row_max, const uint64_t* row_Q, const int32_t* row_argmax, int V,
                        const float* temp, const uint32_t* u_acc, const uint32_t* u_bonus, int32_t* acc_len,
                        int32_t* path, int32_t* out_tok, int32_t* status, cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaFuncSetAttribute(accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_done = true;
  }
  const int CL = accept_cluster_size();
  const size_t smem = static_cast<size_t>((V + CL - 1) / CL) * sizeof(unsigned long long) + 16;
  E3_REQUIRE(smem <= 200 * 1024, E3_ERR_SHAPE, "spec_accept: V=%d too large", V);
  E3_REQUIRE(static_cast<long>(B) * CL < (1L << 31), E3_ERR_SHAPE, "spec_accept: B=%d too large", B);
  cudaError_t e = launch_pdl(accept_kernel, dim3(B * CL), dim3(kAcceptThreads), smem, s, static_cast<unsigned>(CL), tok,
                             parent, R, D, logits, row_max, row_Q, row_argmax, V, temp, u_acc, u_bonus, acc_len, path,
                             out_tok, status);
  if (e != cudaSuccess) return cuda_status(e, "accept_kernel");
  return E3_OK;
}

}  // namespace e3
