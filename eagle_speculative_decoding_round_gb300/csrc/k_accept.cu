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
// chunk into shared memory; every CTA pushes its chunk sum into all CTAs'
// shared memory; the CTA whose chunk holds the target finds the token (warp
// sums, then one warp scan over per-lane pieces) and writes the request's
// outputs.
//
// accept_sampled_kernel (spec_accept_sampled) serves children that were drawn
// from the draft distribution: the acceptance probability is the page's
// min(1, p_res / q_res) and a rejection replaces the residual by
// max(0, p_res - q_res), computed over the whole vocabulary in integer masses
// (see the kernel's own comment).
#include <cooperative_groups.h>

#include <mutex>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kAcceptThreads = 512;
constexpr int kMaxR = E3_MAX_NODES + 1;

namespace cg = cooperative_groups;

constexpr int kMaxCluster = 16;

// Inverse-CDF draw over residual masses spread across the cluster: CTA r holds
// the masses of tokens [j0_r, j0_r + n_r) in qbuf[0, n_r) (chunks in rank order).
// Finds the smallest token whose cumulative mass exceeds x: every CTA pushes its
// chunk sum into s_sums[rank] of every CTA (remote stores, no round trips), so
// that after one cluster barrier each CTA reads all sums locally; the CTA whose
// chunk holds x locates the warp, and that warp scans 32 tokens at a time.  Sets
// *s_bonus in that CTA (untouched if the total is <= x) and returns its rank (0
// if none).  Every thread of every CTA calls it; qbuf is complete and visible on
// entry; s_sums ([kMaxCluster], the same variable in every CTA) is not in use.
__device__ int cluster_inverse_cdf(cg::cluster_group& cluster, const unsigned long long* qbuf, int n, int j0,
                                   uint64_t x, unsigned long long* s_wsum, unsigned long long* s_sums,
                                   int* s_bonus) {
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // per-warp sums of contiguous sub-segments
  const int wseg = (n + nw - 1) / nw;
  const int a0 = min(n, w * wseg), a1 = min(n, a0 + wseg);
  uint64_t local = 0;
  for (int j = a0 + lane; j < a1; j += 32) local += qbuf[j];
  local = warp_reduce(local, SumU64());
  if (lane == 0) s_wsum[w] = local;
  __syncthreads();
  if (w == 0) {
    uint64_t tot = 0;
    for (int i = 0; i < nw; ++i) tot += s_wsum[i];
    if (lane < CL) *cluster.map_shared_rank(&s_sums[rank], lane) = tot;
  }
  cluster.sync();  // every CTA holds every chunk sum
  uint64_t excl = 0;
  int found = -1;
  for (int r = 0; r < CL; ++r) {  // the chunk sums partition [0, total)
    const uint64_t sr = s_sums[r];
    if (found < 0 && x >= excl && x < excl + sr) found = r;
    excl += sr;
  }
  if (found == rank) {
    uint64_t wex = 0;
    for (int r = 0; r < rank; ++r) wex += s_sums[r];
    for (int i = 0; i < w; ++i) wex += s_wsum[i];
    if (x >= wex && x < wex + s_wsum[w]) {  // uniform within the warp
      // each lane sums a contiguous piece of the warp's segment; one warp scan
      // finds the lane whose piece holds x, and that lane walks its piece
      const int sub = (a1 - a0 + 31) >> 5;
      const int b0 = min(a1, a0 + lane * sub), b1 = min(a1, b0 + sub);
      uint64_t part = 0;
      for (int j = b0; j < b1; ++j) part += qbuf[j];
      uint64_t incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, wex + incl > x);
      if (hit && lane == __ffs(hit) - 1) {
        uint64_t cum = wex + incl - part;
        for (int j = b0; j < b1; ++j) {
          cum += qbuf[j];
          if (cum > x) {
            *s_bonus = j0 + j;
            break;
          }
        }
      }
    }
  }
  __syncthreads();
  return found < 0 ? 0 : found;
}

__global__ void __launch_bounds__(kAcceptThreads)
accept_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ parent, int R, int D,
              const float* __restrict__ logits, const float* __restrict__ row_max,
              const uint64_t* __restrict__ row_Q, const int32_t* __restrict__ row_argmax, int V,
              const float* __restrict__ temp, const uint32_t* __restrict__ u_acc,
              const uint32_t* __restrict__ u_bonus, int32_t* acc_len, int32_t* path, int32_t* out_tok,
              int32_t* status) {
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
  __shared__ unsigned long long s_x, s_sums[kMaxCluster];
  __shared__ unsigned long long s_wsum[kAcceptThreads / 32];
  __shared__ float s_nmax[kMaxR];  // every node's row statistics, loaded in parallel
  __shared__ int s_nam[kMaxR];
  __shared__ unsigned long long s_nQ[kMaxR];
  __shared__ uint32_t s_ua[kMaxR];  // every child's acceptance uniform (the walk is serial)

  pdl_wait();
  pdl_trigger();
  const size_t rb = static_cast<size_t>(b) * R;
  const float T = temp[b];
  const float it = inv_temp(T);
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    s_tok[i] = tok[rb + i];
    s_par[i] = parent[rb + i];
    s_nmax[i] = row_max[rb + i];
    s_nam[i] = row_argmax[rb + i];
    s_nQ[i] = row_Q[rb + i];
    s_ua[i] = u_acc[rb + i];
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
      s_qc[c] = fx_mass(__fmul_rn(logits[prow * V + t], it), s_nmax[p]);
    }
  }
  __syncthreads();
  // the walk (every CTA of the cluster does it; integer work only)
  if (threadIdx.x == 0) {
    int u = 0, a = 0, nrem = 0;
    uint64_t Rm = 0;
    for (;;) {
      const float m = s_nmax[u];
      const int am = s_nam[u];
      if (am < 0 || !isfinite(m)) {
        s_err = E3_DEV_ERR_NONFINITE;
        break;
      }
      Rm = s_nQ[u];
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
        if (mulhi32(s_ua[c], Rm) < q) {
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
    const float m = s_nmax[u];
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
    writer = cluster_inverse_cdf(cluster, qbuf, n, j0, x, s_wsum, s_sums, &s_bonus);
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

// Children drawn from the draft distribution q (eagle3_expand_sampled): accept
// with min(1, p_res / q_res), residual max(0, p_res - q_res) on each rejection.
// One cluster of CL CTAs per request walks the tree in lockstep: every CTA's
// thread 0 takes the same decisions from the same integers.  CTA r keeps the
// target residual masses R_j of its vocabulary chunk in qbuf once a rejection
// at the current node has made them differ from the row's plain masses
// (`fresh` until then), and a bit per token of the chunk for the draft tokens
// already rejected at this node.  A rejection costs one pass over the chunk
// (new R_j and their sum) and two cluster barriers; an acceptance test reads
// R_t from the owning CTA's shared memory.
__global__ void __launch_bounds__(kAcceptThreads)
accept_sampled_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ parent,
                      const int32_t* __restrict__ node_cand, int R, int D, const float* __restrict__ logits,
                      const float* __restrict__ row_max, const uint64_t* __restrict__ row_Q,
                      const int32_t* __restrict__ row_argmax, int V, const float* __restrict__ temp,
                      const e3_qstat* __restrict__ qs, int q_cap, const uint32_t* __restrict__ u_acc,
                      const uint32_t* __restrict__ u_bonus, int32_t* acc_len, int32_t* path, int32_t* out_tok,
                      int32_t* status) {
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / CL;
  const int per = (V + CL - 1) / CL;
  const int j0 = min(V, rank * per), j1 = min(V, j0 + per);
  const int n = j1 - j0;
  const int nwords = (per + 31) >> 5;
  extern __shared__ unsigned long long qbuf[];                     // [per] R_j of this CTA's tokens
  uint32_t* rbits = reinterpret_cast<uint32_t*>(qbuf + per);      // [nwords] rejected draft tokens
  __shared__ int s_tok[kMaxR], s_par[kMaxR], s_nch[kMaxR], s_first[kMaxR + 1], s_child[kMaxR];
  __shared__ int s_removed[kMaxR];
  __shared__ int s_path[E3_MAX_DEPTH + 1];
  __shared__ int s_nrem, s_u, s_a, s_err, s_bonus, s_fresh, s_dec, s_t, s_am;
  __shared__ unsigned long long s_SR, s_SD, s_Dt, s_parts[kMaxCluster], s_sums[kMaxCluster];
  __shared__ unsigned long long s_wsum[kAcceptThreads / 32];
  __shared__ uint64_t s_red[32];
  __shared__ float s_mp, s_mq, s_itq;
  __shared__ const float* s_zq;
  __shared__ FracMul s_fm;  // floor(D SR / SD) for the current residual totals
  __shared__ uint32_t s_uacc[kMaxR];
  // per node: target statistics and the draft statistics of its children's row;
  // per child: its token's draft and target masses under its parent's rows
  __shared__ float s_nmax[kMaxR], s_nqm[kMaxR], s_nqit[kMaxR];
  __shared__ int s_nam[kMaxR];
  __shared__ unsigned long long s_nQ[kMaxR], s_nqQ[kMaxR], s_Dc[kMaxR], s_Rc[kMaxR];
  __shared__ const float* s_nqrow[kMaxR];

  pdl_wait();
  pdl_trigger();
  const size_t rb = static_cast<size_t>(b) * R;
  const float T = temp[b];
  const float it = inv_temp(T);
  // the tree, and every node's statistics, loaded in parallel (the walk then reads
  // shared memory only); a node's draft entry is read whether or not it has
  // children, and used only if it has
  for (int u = threadIdx.x; u < R; u += blockDim.x) {
    const size_t row = rb + u;
    s_tok[u] = tok[row];
    s_par[u] = parent[row];
    s_uacc[u] = u_acc[row];
    s_nmax[u] = row_max[row];
    s_nam[u] = row_argmax[row];
    s_nQ[u] = row_Q[row];
    s_nqrow[u] = nullptr;
    s_nqQ[u] = 0ull;
    s_nqm[u] = 0.0f;
    s_nqit[u] = 0.0f;
    const int nc = node_cand[row];
    if (T > 0.0f && nc >= -1 && nc + 1 < q_cap) {
      const e3_qstat q = qs[static_cast<size_t>(b) * q_cap + (nc + 1)];
      s_nqrow[u] = q.row;
      s_nqQ[u] = q.Q;
      s_nqm[u] = q.m;
      s_nqit[u] = q.inv_temp;
    }
  }
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) rbits[w] = 0u;
  __syncthreads();
  // children lists in CSR form, children in ascending flat order (= draw order)
  for (int u = threadIdx.x; u < R; u += blockDim.x) {
    int cnt = 0;
    for (int c = u + 1; c < R; ++c) cnt += (s_par[c] == u);
    s_nch[u] = cnt;
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
    s_u = 0;
    s_a = 0;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < R; c += blockDim.x) {
    const int p = s_par[c];
    if (c == 0 || p < 0 || p >= c) continue;
    int rk = 0;
    for (int c2 = p + 1; c2 < c; ++c2) rk += (s_par[c2] == p);
    s_child[s_first[p] + rk] = c;
  }
  for (int c = threadIdx.x; c < R; c += blockDim.x) {
    s_Dc[c] = 0ull;
    s_Rc[c] = 0ull;
    const int p = s_par[c];
    const int t = s_tok[c];
    if (T <= 0.0f || c == 0 || p < 0 || p >= c || t < 0 || t >= V) continue;
    const float* zq = s_nqrow[p];
    if (zq != nullptr && isfinite(s_nqm[p]) && isfinite(s_nmax[p])) {
      s_Dc[c] = fx_mass(__fmul_rn(zq[t], s_nqit[p]), s_nqm[p]);
      s_Rc[c] = fx_mass(__fmul_rn(logits[(rb + p) * V + t], it), s_nmax[p]);
    }
  }
  __syncthreads();

  for (;;) {  // one iteration per visited node, uniform across the cluster
    if (threadIdx.x == 0) {
      const int u = s_u;
      s_mp = s_nmax[u];
      s_am = s_nam[u];
      s_SR = s_nQ[u];
      s_fresh = 1;
      s_nrem = 0;
      s_SD = 0ull;
      s_zq = nullptr;
      if (s_am < 0 || !isfinite(s_mp)) s_err = E3_DEV_ERR_NONFINITE;
      if (!s_err && T > 0.0f && s_nch[u] > 0) {
        if (s_nqrow[u] == nullptr || !isfinite(s_nqm[u]) || s_nqQ[u] == 0ull) {
          s_err = E3_DEV_ERR_NONFINITE;
        } else {
          s_zq = s_nqrow[u];
          s_SD = s_nqQ[u];
          s_mq = s_nqm[u];
          s_itq = s_nqit[u];
          s_fm = frac_mul_prep(s_SR, s_SD);
        }
      }
    }
    __syncthreads();
    if (s_err) break;
    const int u = s_u;
    const size_t row = rb + u;
    const float* z = logits + row * V;
    int accepted = -1;
    for (int e = s_first[u]; e < s_first[u] + s_nch[u]; ++e) {
      const int c = s_child[e];
      if (threadIdx.x == 0) {
        const int t = s_tok[c];
        int dec = 2;  // 0 reject, 1 accept, 2 skip (not a draw)
        if (T <= 0.0f) {
          dec = (t == s_am) ? 1 : 2;
        } else if (t >= 0 && t < V) {
          bool rem = false;
          for (int i = 0; i < s_nrem; ++i) rem |= (s_removed[i] == t);
          const uint64_t Dt = rem ? 0ull : s_Dc[c];
          if (Dt != 0ull) {
            uint64_t Rt;
            if (s_fresh) {
              Rt = s_Rc[c];
            } else {
              const int owner = t / per;
              Rt = cluster.map_shared_rank(qbuf, owner)[t - owner * per];
            }
            // accept iff u * qt < Rt 2^32, compared as (high, low) words
            const uint64_t qt = frac_mul(s_fm, Dt);
            const uint64_t u = s_uacc[c];
            const uint64_t l_hi = __umul64hi(u, qt), l_lo = u * qt;
            const uint64_t r_hi = Rt >> 32, r_lo = Rt << 32;
            dec = (l_hi < r_hi || (l_hi == r_hi && l_lo < r_lo)) ? 1 : 0;
            s_Dt = Dt;
            s_t = t;
          }
        }
        s_dec = dec;
      }
      __syncthreads();
      const int dec = s_dec;
      __syncthreads();  // everyone has read s_dec before thread 0 may write it again
      if (dec == 1) {
        accepted = c;
        break;
      }
      if (dec == 2) continue;
      // rejection: the residual pass over this CTA's tokens
      cluster.sync();  // no CTA still reads a peer's qbuf for the decision above
      const bool fresh = s_fresh != 0;
      const float mq = s_mq, itq = s_itq, mp = s_mp;
      const float* zq = s_zq;
      const FracMul fm = s_fm;  // floor(D_j SR / SD) for every j
      uint64_t local = 0;
      constexpr int kBatch = 8;  // tokens per thread in flight: their loads are issued together
      for (int j = threadIdx.x; j < n; j += kBatch * blockDim.x) {
        float qv[kBatch], zv[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int jj = j + i * blockDim.x;
          qv[i] = jj < n ? zq[j0 + jj] : 0.0f;
          zv[i] = (fresh && jj < n) ? z[j0 + jj] : 0.0f;
        }
        // the recipe's exponentials two lanes at a time: (draft, target) of one
        // token while the target masses are the row's own, else the drafts of two
        float ed[kBatch], er[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; i += 2) {
          const float d0 = __fsub_rn(__fmul_rn(qv[i], itq), mq), d1 = __fsub_rn(__fmul_rn(qv[i + 1], itq), mq);
          if (fresh) {
            const float2 a = fx_exp_x2(make_float2(d0, __fsub_rn(__fmul_rn(zv[i], it), mp)));
            const float2 c = fx_exp_x2(make_float2(d1, __fsub_rn(__fmul_rn(zv[i + 1], it), mp)));
            ed[i] = a.x, er[i] = a.y, ed[i + 1] = c.x, er[i + 1] = c.y;
          } else {
            const float2 a = fx_exp_x2(make_float2(d0, d1));
            ed[i] = a.x, ed[i + 1] = a.y, er[i] = er[i + 1] = 0.0f;
          }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int jj = j + i * blockDim.x;
          if (jj < n) {
            const bool rem = (rbits[jj >> 5] >> (jj & 31)) & 1u;
            const uint64_t Dj = rem ? 0ull : fx_scale40_floor(ed[i]);
            uint64_t Rj = fresh ? fx_scale40_floor(er[i]) : qbuf[jj];
            const uint64_t qj = Dj ? frac_mul(fm, Dj) : 0ull;
            Rj = Rj > qj ? Rj - qj : 0ull;
            qbuf[jj] = Rj;
            local += Rj;
          }
        }
      }
      local = block_reduce(local, SumU64(), s_red);
      if (threadIdx.x < CL) *cluster.map_shared_rank(&s_parts[rank], threadIdx.x) = local;  // to every CTA
      if (threadIdx.x == 0) {
        const int t = s_t;
        if (t >= j0 && t < j1) rbits[(t - j0) >> 5] |= 1u << ((t - j0) & 31);
      }
      cluster.sync();  // partial sums and residuals visible
      if (threadIdx.x == 0) {
        uint64_t tot = 0;
        for (int r = 0; r < CL; ++r) tot += s_parts[r];
        s_SR = tot;
        s_SD -= s_Dt;
        s_removed[s_nrem++] = s_t;
        s_fresh = 0;
        if (s_SD != 0ull) s_fm = frac_mul_prep(s_SR, s_SD);
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      if (accepted >= 0 && s_a < D) {
        s_a += 1;
        s_path[s_a] = accepted;
        s_u = accepted;
        s_dec = 3;
      } else {
        s_dec = 4;
      }
    }
    __syncthreads();
    const bool stop = s_dec == 4;
    for (int w = threadIdx.x; w < nwords; w += blockDim.x) rbits[w] = 0u;  // the next node starts afresh
    __syncthreads();
    if (stop) break;
  }

  const int err = s_err;
  int writer = 0;
  if (!err && T > 0.0f) {
    const int u = s_u;
    const uint64_t x = mulhi32(u_bonus[rb + u], s_SR);
    const float* z = logits + (rb + u) * V;
    const float mp = s_mp;
    const bool fresh = s_fresh != 0;
    cluster.sync();  // no CTA still reads a peer's qbuf
    if (fresh) {
#pragma unroll 4
      for (int j = threadIdx.x; j < n; j += blockDim.x) qbuf[j] = fx_mass(__fmul_rn(z[j0 + j], it), mp);
    }
    __syncthreads();
    writer = cluster_inverse_cdf(cluster, qbuf, n, j0, x, s_wsum, s_sums, &s_bonus);
  } else if (!err && threadIdx.x == 0) {
    s_bonus = s_am;
  }
  if (rank == writer && threadIdx.x == 0) {
    const int a = err ? 0 : s_a;
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
  cluster.sync();  // peers may still read this CTA's shared memory
}

int accept_cluster_size() {
  static const int cl_once = [] {  // computed once, thread-safely
    int cl = 8;
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
    return cl;
  }();
  return cl_once;
}

// 16-CTA clusters of accept_sampled_kernel where the GPU allows them, else 8.
int accept_sampled_cluster_size(int V) {
  static std::mutex mu;  // the cache below is read and refreshed as a unit
  const std::lock_guard<std::mutex> lock(mu);
  static int cached_v = -1, cl = 8;
  if (cached_v != V) {
    cl = 8;
    cached_v = V;
    if (cudaFuncSetAttribute(accept_sampled_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(kAcceptThreads);
      const int per = (V + 15) / 16;
      cfg.dynamicSmemBytes = static_cast<size_t>(per) * 8 + static_cast<size_t>((per + 31) / 32) * 4 + 16;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 16;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int nclu = 0;
      if (cudaOccupancyMaxActiveClusters(&nclu, accept_sampled_kernel, &cfg) == cudaSuccess && nclu > 0) cl = 16;
    }
    cudaGetLastError();
  }
  return cl;
}

}  // namespace

e3_status launch_accept_sampled(const int32_t* tok, const int32_t* parent, const int32_t* node_cand, int B, int R,
                                int D, const float* logits, const float* row_max, const uint64_t* row_Q,
                                const int32_t* row_argmax, int V, const float* temp, const e3_qstat* q_stats,
                                int q_cap, const uint32_t* u_acc, const uint32_t* u_bonus, int32_t* acc_len,
                                int32_t* path, int32_t* out_tok, int32_t* status, cudaStream_t s) {
  // one-time setup (a function-local static is initialised once, thread-safely)
  static const bool attr_done =
      (cudaFuncSetAttribute(accept_sampled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024), true);
  (void)attr_done;
  const int CL = accept_sampled_cluster_size(V);
  const int per = (V + CL - 1) / CL;
  const size_t smem = static_cast<size_t>(per) * 8 + static_cast<size_t>((per + 31) / 32) * 4 + 16;
  E3_REQUIRE(smem <= 200 * 1024, E3_ERR_SHAPE, "spec_accept_sampled: V=%d too large", V);
  E3_REQUIRE(static_cast<long>(B) * CL < (1L << 31), E3_ERR_SHAPE, "spec_accept_sampled: B=%d too large", B);
  cudaError_t e = launch_pdl(accept_sampled_kernel, dim3(B * CL), dim3(kAcceptThreads), smem, s,
                             static_cast<unsigned>(CL), tok, parent, node_cand, R, D, logits, row_max, row_Q,
                             row_argmax, V, temp, q_stats, q_cap, u_acc, u_bonus, acc_len, path, out_tok, status);
  if (e != cudaSuccess) return cuda_status(e, "accept_sampled_kernel");
  return E3_OK;
}

e3_status launch_accept(const int32_t* tok, const int32_t* parent, int B, int R, int D, const float* logits,
                        const float* row_max, const uint64_t* row_Q, const int32_t* row_argmax, int V,
                        const float* temp, const uint32_t* u_acc, const uint32_t* u_bonus, int32_t* acc_len,
                        int32_t* path, int32_t* out_tok, int32_t* status, cudaStream_t s) {
  // one-time setup (a function-local static is initialised once, thread-safely)
  static const bool attr_done =
      (cudaFuncSetAttribute(accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024), true);
  (void)attr_done;
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
