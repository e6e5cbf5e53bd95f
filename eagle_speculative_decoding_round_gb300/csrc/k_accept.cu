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
// One CTA per request.  Thread 0 walks the tree (at most D+1 rows); the bonus
// draw is an inverse-CDF search over the whole vocabulary done by all threads:
// per-warp segment sums of the fixed-point masses, an exclusive scan of the
// warp sums, and a rescan of the one segment that holds the target.
#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kAcceptThreads = 1024;

__device__ __forceinline__ bool is_removed(const int* removed, int nrem, int j) {
  for (int q = 0; q < nrem; ++q)
    if (removed[q] == j) return true;
  return false;
}

__global__ void __launch_bounds__(kAcceptThreads)
accept_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ parent, int R, int D,
              const float* __restrict__ logits, const float* __restrict__ row_max,
              const uint64_t* __restrict__ row_Q, const int32_t* __restrict__ row_argmax, int V,
              const float* __restrict__ temp, const uint32_t* __restrict__ u_acc,
              const uint32_t* __restrict__ u_bonus, int32_t* acc_len, int32_t* path, int32_t* out_tok,
              int32_t* status) {
  __shared__ int s_tok[256], s_par[256];
  __shared__ int s_removed[256];
  __shared__ int s_nrem, s_u, s_acc, s_bonus, s_err;
  __shared__ unsigned long long s_x;
  __shared__ uint64_t s_scan[32];
  __shared__ int s_path[E3_MAX_DEPTH + 1];
  const int b = blockIdx.x;
  const float T = temp[b];
  const float it = inv_temp(T);
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    s_tok[i] = tok[static_cast<size_t>(b) * R + i];
    s_par[i] = parent[static_cast<size_t>(b) * R + i];
  }
  // prefetch, in parallel, everything the walk reads: each node's statistics and
  // each child's logit under its parent's row
  __shared__ float s_m[256], s_zc[256];
  __shared__ unsigned long long s_Q[256];
  __shared__ int s_am[256];
  __syncthreads();
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    const size_t row = static_cast<size_t>(b) * R + i;
    s_m[i] = row_max[row];
    s_Q[i] = row_Q[row];
    s_am[i] = row_argmax[row];
    const int p = s_par[i], t = s_tok[i];
    s_zc[i] = (i > 0 && p >= 0 && p < R && t >= 0 && t < V) ? logits[(static_cast<size_t>(b) * R + p) * V + t] : 0.0f;
  }
  if (threadIdx.x == 0) {
    s_err = 0;
    s_acc = 0;
    s_bonus = -1;
    s_path[0] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int u = 0, a = 0;
    for (;;) {
      const float m = s_m[u];
      uint64_t Rm = s_Q[u];
      const int am = s_am[u];
      if (am < 0 || !isfinite(m)) {
        s_err = E3_DEV_ERR_NONFINITE;
        break;
      }
      int nrem = 0, accepted = -1;
      for (int c = u + 1; c < R; ++c) {
        if (s_par[c] != u) continue;
        const int t = s_tok[c];
        if (T <= 0.0f) {
          if (t == am) {
            accepted = c;
            break;
          }
          continue;
        }
        if (t < 0 || t >= V) continue;
        const uint64_t q = fx_mass(__fmul_rn(s_zc[c], it), m);
        if (mulhi32(u_acc[static_cast<size_t>(b) * R + c], Rm) < q) {
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
      s_u = u;
      s_acc = a;
      s_nrem = nrem;
      if (T <= 0.0f)
        s_bonus = am;
      else
        s_x = mulhi32(u_bonus[static_cast<size_t>(b) * R + u], Rm);
      break;
    }
  }
  __syncthreads();
  const int err = s_err;
  if (!err && T > 0.0f) {
    // inverse CDF over the residual, ascending token ids.  Warp w owns the
    // contiguous segment [w*seg, (w+1)*seg) and sums it with lane-strided loads;
    // an exclusive scan of the 32 warp sums locates the segment holding x, which
    // its warp rescans 32 tokens at a time (warp scan + ballot).
    const int u = s_u, nrem = s_nrem;
    const uint64_t x = s_x;
    const size_t row = static_cast<size_t>(b) * R + u;
    const float m = row_max[row];
    const float* z = logits + row * V;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int seg = (V + nw - 1) / nw;
    const int j0 = min(V, wid * seg), j1 = min(V, j0 + seg);
    uint64_t local = 0;
#pragma unroll 8
    for (int j = j0 + lane; j < j1; j += 32) {
      const float zj = z[j];
      if (!is_removed(s_removed, nrem, j)) local += fx_mass(__fmul_rn(zj, it), m);
    }
    local = warp_reduce(local, SumU64());
    if (lane == 0) s_scan[wid] = local;
    __syncthreads();
    uint64_t excl = 0;
    for (int w = 0; w < wid; ++w) excl += s_scan[w];
    if (x >= excl && x < excl + local) {  // uniform within the warp
      uint64_t base = excl;
      for (int c0 = j0; c0 < j1; c0 += 32) {
        const int j = c0 + lane;
        uint64_t q = 0;
        if (j < j1 && !is_removed(s_removed, nrem, j)) q = fx_mass(__fmul_rn(z[j], it), m);
        uint64_t incl = q;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, base + incl > x);
        if (hit) {
          if (lane == __ffs(hit) - 1) s_bonus = j;
          break;
        }
        base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
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
}

}  // namespace

e3_status launch_accept(const int32_t* tok, const int32_t* parent, int B, int R, int D, const float* logits,
                        const float* row_max, const uint64_t* row_Q, const int32_t* row_argmax, int V,
                        const float* temp, const uint32_t* u_acc, const uint32_t* u_bonus, int32_t* acc_len,
                        int32_t* path, int32_t* out_tok, int32_t* status, cudaStream_t s) {
  accept_kernel<<<B, kAcceptThreads, 0, s>>>(tok, parent, R, D, logits, row_max, row_Q, row_argmax, V, temp,
                                            u_acc, u_bonus, acc_len, path, out_tok, status);
  E3_LAUNCH_CHECK("accept_kernel");
  return E3_OK;
}

}  // namespace e3
