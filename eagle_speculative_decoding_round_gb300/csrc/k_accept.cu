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
// builds the children lists (warp ballots) and each child's fixed-point mass in
// parallel, and its warp 0 walks the tree, testing a node's children as one warp
// (integer work only).  For the bonus draw, CTA r owns a contiguous chunk of the
// vocabulary, staged by a bulk copy (the root's row is staged speculatively while
// the tree is walked): it computes the residual masses of its chunk into shared
// memory; every CTA sends its chunk sum to all CTAs as asynchronous stores; the
// CTA whose chunk holds the target finds the token (warp sums, then one warp scan
// over per-lane pieces) and writes the request's outputs.
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

// Children lists in CSR form, children of u (the nodes c > u with parent u) in
// ascending flat order: counts by warp ballots (warp w takes nodes w, w + nw, ...),
// offsets by one warp scan, then the lists.  Every thread of the CTA calls it;
// s_par is complete and visible on entry, the lists are on return.
__device__ void build_children(int R, const int* s_par, int* s_nch, int* s_first, int* s_child) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int u = warp; u < R; u += nw) {
    int cnt = 0;
    for (int c0 = 0; c0 < R; c0 += 32) {
      const int c = c0 + lane;
      cnt += __popc(__ballot_sync(0xFFFFFFFFu, c < R && c > u && s_par[c] == u));
    }
    if (lane == 0) s_nch[u] = cnt;
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int u0 = 0; u0 < R; u0 += 32) {
      const int u = u0 + lane;
      const int v = u < R ? s_nch[u] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (u < R) s_first[u] = run + incl - v;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) s_first[R] = run;
  }
  __syncthreads();
  for (int u = warp; u < R; u += nw) {
    int base = s_first[u];
    for (int c0 = 0; c0 < R; c0 += 32) {
      const int c = c0 + lane;
      const bool is = c < R && c > u && s_par[c] == u;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, is);
      if (is) s_child[base + __popc(bal & ((1u << lane) - 1u))] = c;
      base += __popc(bal);
    }
  }
  __syncthreads();
}

// Shared-memory and cluster helpers of accept_kernel.
__device__ __forceinline__ uint32_t sh_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void acc_bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sh_addr(b)), "r"(n));
}
__device__ __forceinline__ void acc_bar_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sh_addr(b)), "r"(bytes) : "memory");
}
// bounded wait (acquire at cluster scope) for the phase of parity par of a local mbarrier
__device__ __forceinline__ bool acc_bar_wait(uint64_t* b, uint32_t par) {
  uint64_t t0 = 0;
  for (int i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(sh_addr(b)), "r"(par)
        : "memory");
    if (ok) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    if (i == 0) t0 = t;
    if (t - t0 > 1000000000ull) return false;
  }
}
// 8 bytes into CTA `rank`'s shared memory at the same offset as p, completing on
// that CTA's mbarrier at the same offset as bar (the sender does not wait)
__device__ __forceinline__ void acc_st_async64(const void* p, uint64_t v, const uint64_t* bar, uint32_t rank) {
  uint32_t a, m;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(sh_addr(p)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(m) : "r"(sh_addr(bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(a), "l"(v), "r"(m)
               : "memory");
}

// Dynamic shared memory of accept_kernel for chunks of `per` tokens: residual
// masses (u64), the bonus row's logits (fp32) and a removed-token bit per token.
size_t accept_smem_bytes(int per) {
  const size_t q = (static_cast<size_t>(per) * 8 + 15) & ~static_cast<size_t>(15);
  const size_t z = (static_cast<size_t>(per) * 4 + 15) & ~static_cast<size_t>(15);
  return q + z + static_cast<size_t>((per + 31) / 32) * 4 + 16;
}

// One cluster of CL CTAs per request; CTA r owns vocabulary chunk r.
//   1. The tree, every node's statistics and uniforms go to shared memory; each
//      child's mass under its parent's row is fetched (one load per child); the
//      children lists are built with warp ballots.  While this happens, a bulk
//      copy stages the root row's chunk (the bonus row when nothing is accepted).
//   2. Warp 0 walks the tree.  At node u the children are tested in order as one
//      warp: child c is accepted iff (u_acc[c] * Rm_c) >> 32 < q_c with Rm_c = Q_u
//      minus the masses of the valid siblings before it (they were rejected); the
//      first passing child wins, so the serial rule is reproduced exactly.
//   3. Sampled rows: the bonus row's chunk (staged, re-staged if the walk left the
//      root) becomes residual masses (removed tokens zero), summed per warp; the
//      chunk sums travel to every CTA as asynchronous stores; the CTA and warp
//      whose tokens hold x find the token.
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int per = (V + CL - 1) / CL;
  const int j0 = min(V, rank * per), j1 = min(V, j0 + per);
  const int n = j1 - j0;
  const int nwords = (per + 31) >> 5;
  extern __shared__ __align__(16) unsigned char acc_dyn[];
  unsigned long long* qbuf = reinterpret_cast<unsigned long long*>(acc_dyn);  // [per] residual masses
  float* zbuf = reinterpret_cast<float*>(acc_dyn + ((static_cast<size_t>(per) * 8 + 15) & ~static_cast<size_t>(15)));
  uint32_t* rbits = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(zbuf) +
                                                ((static_cast<size_t>(per) * 4 + 15) & ~static_cast<size_t>(15)));
  __shared__ int s_tok[kMaxR], s_par[kMaxR], s_nch[kMaxR], s_first[kMaxR + 1], s_child[kMaxR];
  __shared__ unsigned long long s_qc[kMaxR];  // mass of child c under its parent's row
  __shared__ unsigned long long s_nQ[kMaxR];
  __shared__ float s_nmax[kMaxR];
  __shared__ int s_nam[kMaxR];
  __shared__ uint32_t s_ua[kMaxR], s_ub[kMaxR];
  __shared__ int s_removed[kMaxR];
  __shared__ int s_path[E3_MAX_DEPTH + 1];
  __shared__ int s_nrem, s_u, s_acc, s_err, s_bonus;
  __shared__ unsigned long long s_x, s_sums[kMaxCluster];
  __shared__ unsigned long long s_wsum[kAcceptThreads / 32];
  __shared__ uint64_t ld_bar, sum_bar;

  if (threadIdx.x == 0) {
    acc_bar_init(&ld_bar, 1);
    acc_bar_init(&sum_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    acc_bar_expect(&sum_bar, static_cast<uint32_t>(CL) * 8u);  // every CTA's chunk sum
  }
  __syncthreads();
  // the peers' mbarriers are initialized before anyone stores to them (waited for
  // just before the first asynchronous store)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  pdl_wait();
  pdl_trigger();
  const size_t rb = static_cast<size_t>(b) * R;
  const float T = temp[b];
  const float it = inv_temp(T);
  // chunk staging: bulk copies of 16-byte multiples when the rows allow it (the last
  // n % 4 logits, or all of them otherwise, by plain loads)
  const bool bulk = (V % 4) == 0 && (per % 4) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  const uint32_t bulk_bytes = bulk ? static_cast<uint32_t>(n / 4) * 16u : 0u;
  auto stage_row = [&](int u) {  // thread 0: chunk of row u into zbuf, completing on ld_bar
    acc_bar_expect(&ld_bar, bulk_bytes);
    const unsigned char* src = reinterpret_cast<const unsigned char*>(logits + (rb + u) * V + j0);
    for (uint32_t off = 0; off < bulk_bytes; off += 32768u) {
      const uint32_t nb = min(32768u, bulk_bytes - off);
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       sh_addr(reinterpret_cast<unsigned char*>(zbuf) + off)),
                   "l"(src + off), "r"(nb), "r"(sh_addr(&ld_bar))
                   : "memory");
    }
  };
  const bool spec_root = T > 0.0f && bulk && bulk_bytes > 0;
  if (threadIdx.x == 0 && spec_root) stage_row(0);
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    s_tok[i] = tok[rb + i];
    s_par[i] = parent[rb + i];
    s_nmax[i] = row_max[rb + i];
    s_nam[i] = row_argmax[rb + i];
    s_nQ[i] = row_Q[rb + i];
    s_ua[i] = u_acc[rb + i];
    s_ub[i] = u_bonus[rb + i];
  }
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) rbits[w] = 0u;
  if (threadIdx.x == 0) {
    s_bonus = -1;
    s_path[0] = 0;
  }
  __syncthreads();
  // each child's mass under its parent's row: thread c requests its logit now (one
  // global load per child, R <= blockDim.x) and uses it after the children lists
  const int c_me = threadIdx.x;
  const int p_me = c_me < R ? s_par[c_me] : -1;
  const int t_me = c_me < R ? s_tok[c_me] : -1;
  const bool has_q = c_me > 0 && c_me < R && p_me >= 0 && p_me < c_me && T > 0.0f && t_me >= 0 && t_me < V;
  const float z_me = has_q ? logits[(rb + p_me) * V + t_me] : 0.0f;
  build_children(R, s_par, s_nch, s_first, s_child);
  if (c_me < R) s_qc[c_me] = has_q ? fx_mass(__fmul_rn(z_me, it), s_nmax[p_me]) : 0ull;
  __syncthreads();
  // the walk (warp 0 of every CTA; integer work only)
  if (warp == 0) {
    int u = 0, a = 0, nrem = 0, err = 0, bonus = -1;
    uint64_t Rm = 0;
    for (;;) {
      const float m = s_nmax[u];
      const int am = s_nam[u];
      if (am < 0 || !isfinite(m)) {
        err = E3_DEV_ERR_NONFINITE;
        break;
      }
      Rm = s_nQ[u];
      nrem = 0;
      int accepted = -1;
      const int e0 = s_first[u], ne = s_nch[u];
      for (int eb = 0; eb < ne; eb += 32) {  // the children in order, 32 at a time
        const int e = eb + lane;
        const bool in = e < ne;
        const int c = in ? s_child[e0 + e] : 0;
        const int t = in ? s_tok[c] : -1;
        bool pass, valid = false;
        uint64_t q = 0ull;
        if (T <= 0.0f) {
          pass = in && t == am;
        } else {
          valid = in && t >= 0 && t < V;
          q = valid ? s_qc[c] : 0ull;
          uint64_t incl = q;  // masses of the valid children up to this one
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
          }
          pass = valid && mulhi32(s_ua[c], Rm - (incl - q)) < q;
        }
        const unsigned pb = __ballot_sync(0xFFFFFFFFu, pass);
        const int first = pb ? __ffs(pb) - 1 : 32;
        // the valid children before the first acceptance were rejected: they leave
        // the residual
        const bool rej = valid && lane < first;
        const unsigned rb_mask = __ballot_sync(0xFFFFFFFFu, rej);
        if (rej) s_removed[nrem + __popc(rb_mask & ((1u << lane) - 1u))] = t;
        Rm -= warp_reduce(rej ? q : 0ull, SumU64());
        nrem += __popc(rb_mask);
        if (pb) {
          accepted = __shfl_sync(0xFFFFFFFFu, c, first);
          break;
        }
      }
      if (accepted >= 0 && a < D) {
        ++a;
        if (lane == 0) s_path[a] = accepted;
        u = accepted;
        continue;
      }
      if (T <= 0.0f) bonus = am;
      break;
    }
    if (lane == 0) {
      s_u = u;
      s_acc = a;
      s_nrem = nrem;
      s_err = err;
      if (bonus >= 0) s_bonus = bonus;
      s_x = (T > 0.0f) ? mulhi32(s_ub[u], Rm) : 0ull;
    }
  }
  __syncthreads();
  const int err = s_err;
  int writer = 0;  // the CTA that writes this request's outputs
  const bool sampled = !err && T > 0.0f;  // uniform across the cluster
  bool ok = true;
  if (sampled) {
    const int u = s_u;
    const uint64_t x = s_x;
    const float m = s_nmax[u];
    const int nrem = s_nrem;
    for (int i = threadIdx.x; i < nrem; i += blockDim.x) {
      const int t = s_removed[i];
      if (t >= j0 && t < j1) atomicOr(&rbits[(t - j0) >> 5], 1u << ((t - j0) & 31));
    }
    // the bonus row's chunk: the staged root row, or row u staged now
    if (bulk && bulk_bytes > 0) {
      if (threadIdx.x == 0 && u != 0) {
        ok = acc_bar_wait(&ld_bar, 0);  // the root row's copy has landed before zbuf is reused
        stage_row(u);
      }
      ok = __syncthreads_and(ok) && acc_bar_wait(&ld_bar, u != 0 ? 1u : 0u);
    }
    const float* z = logits + (rb + u) * V + j0;
    for (int j = static_cast<int>(bulk_bytes / 4) + threadIdx.x; j < n; j += blockDim.x) zbuf[j] = z[j];
    ok = __syncthreads_and(ok);
    // residual masses of warp w's contiguous segment of the chunk, two tokens at a time
    const int wseg = (n + nw - 1) / nw;
    const int a0 = min(n, warp * wseg), a1 = min(n, a0 + wseg);
    uint64_t local = 0;
    for (int j = a0 + lane; j < a1; j += 128) {  // four tokens per lane and step, two exponentials at a time
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = j + 32 * i < a1 ? __fsub_rn(__fmul_rn(zbuf[j + 32 * i], it), m) : -INFINITY;
      const float2 e01 = fx_exp_x2(make_float2(x[0], x[1])), e23 = fx_exp_x2(make_float2(x[2], x[3]));
      const float e[4] = {e01.x, e01.y, e23.x, e23.y};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int jj = j + 32 * i;
        if (jj < a1) {
          const uint64_t q = ((rbits[jj >> 5] >> (jj & 31)) & 1u) ? 0ull : fx_scale40_floor(e[i]);
          qbuf[jj] = q;
          local += q;
        }
      }
    }
    local = warp_reduce(local, SumU64());
    if (lane == 0) s_wsum[warp] = local;
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // the peers' mbarriers are initialized
    if (warp == 0) {
      uint64_t tot = lane < nw ? s_wsum[lane] : 0ull;
      tot = warp_reduce(tot, SumU64());
      if (lane < CL) acc_st_async64(&s_sums[rank], tot, &sum_bar, static_cast<uint32_t>(lane));
    }
    ok = acc_bar_wait(&sum_bar, 0) && ok;
    // the chunk sums partition [0, total): the CTA, then the warp, then the lane
    // piece whose masses hold x
    uint64_t excl = 0;
    int found = -1;
    for (int r = 0; r < CL; ++r) {
      const uint64_t sr = s_sums[r];
      if (found < 0 && x >= excl && x < excl + sr) found = r;
      excl += sr;
    }
    if (ok && found == rank) {
      uint64_t wex = 0;
      for (int r = 0; r < rank; ++r) wex += s_sums[r];
      for (int i = 0; i < warp; ++i) wex += s_wsum[i];
      if (x >= wex && x < wex + s_wsum[warp]) {  // uniform within the warp
        // lane pieces of the segment: the piece holding x by one warp scan of the
        // piece sums, then the token by one warp scan of that piece's masses (in
        // steps of 32 tokens)
        const int sub = (a1 - a0 + 31) >> 5;
        const int b0 = min(a1, a0 + lane * sub), b1 = min(a1, b0 + sub);
        uint64_t part = 0;
#pragma unroll 4
        for (int j = b0; j < b1; ++j) part += qbuf[j];
        uint64_t incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, wex + incl > x);
        if (hit) {
          const int L = __ffs(hit) - 1;
          const int pb0 = __shfl_sync(0xFFFFFFFFu, b0, L), pb1 = __shfl_sync(0xFFFFFFFFu, b1, L);
          uint64_t cum = __shfl_sync(0xFFFFFFFFu, wex + incl - part, L);  // mass before the piece
          for (int q0 = pb0; q0 < pb1; q0 += 32) {
            const int j = q0 + lane;
            const uint64_t v = j < pb1 ? qbuf[j] : 0ull;
            uint64_t ci = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, ci, o);
              if (lane >= o) ci += y;
            }
            const unsigned h2 = __ballot_sync(0xFFFFFFFFu, j < pb1 && cum + ci > x);
            if (h2) {
              if (lane == __ffs(h2) - 1) s_bonus = j0 + j;
              break;
            }
            cum += __shfl_sync(0xFFFFFFFFu, ci, 31);
          }
        }
      }
    }
    __syncthreads();
    writer = found < 0 ? 0 : found;
  } else {
    if (spec_root && threadIdx.x == 0) ok = acc_bar_wait(&ld_bar, 0);  // the root copy lands before exit
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  }
  if (rank == writer && threadIdx.x == 0) {
    const int e = err ? err : (ok ? 0 : E3_DEV_ERR_TIMEOUT);
    const int a = e ? 0 : s_acc;
    const size_t o = static_cast<size_t>(b) * (D + 1);
    for (int j = 0; j <= D; ++j) {
      path[o + j] = (!e && j <= a) ? s_path[j] : -1;
      out_tok[o + j] = -1;
    }
    if (e) {
      path[o] = 0;
    } else {
      for (int j = 1; j <= a; ++j) out_tok[o + j - 1] = s_tok[s_path[j]];
      out_tok[o + a] = s_bonus;
    }
    acc_len[b] = a;
    status[b] = e;
  }
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
  if (threadIdx.x == 0) {
    s_err = 0;
    s_bonus = -1;
    s_path[0] = 0;
    s_u = 0;
    s_a = 0;
  }
  build_children(R, s_par, s_nch, s_first, s_child);
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

// 16-CTA clusters of accept_kernel where the GPU allows them (for this vocabulary's
// shared memory), else 8.
int accept_cluster_size(int V) {
  static std::mutex mu;  // the cache below is read and refreshed as a unit
  const std::lock_guard<std::mutex> lock(mu);
  static int cached_v = -1, cl = 8;
  if (cached_v != V) {
    cl = 8;
    cached_v = V;
    if (cudaFuncSetAttribute(accept_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(kAcceptThreads);
      cfg.dynamicSmemBytes = accept_smem_bytes((V + 15) / 16);
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
  const int CL = accept_cluster_size(V);
  const size_t smem = accept_smem_bytes((V + CL - 1) / CL);
  E3_REQUIRE(smem <= 200 * 1024, E3_ERR_SHAPE, "spec_accept: V=%d too large", V);
  E3_REQUIRE(static_cast<long>(B) * CL < (1L << 31), E3_ERR_SHAPE, "spec_accept: B=%d too large", B);
  cudaError_t e = launch_pdl(accept_kernel, dim3(B * CL), dim3(kAcceptThreads), smem, s, static_cast<unsigned>(CL), tok,
                             parent, R, D, logits, row_max, row_Q, row_argmax, V, temp, u_acc, u_bonus, acc_len, path,
                             out_tok, status);
  if (e != cudaSuccess) return cuda_status(e, "accept_kernel");
  return E3_OK;
}

}  // namespace e3
