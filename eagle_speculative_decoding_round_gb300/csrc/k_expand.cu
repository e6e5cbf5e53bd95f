// k_expand.cu -- eagle3_expand: one depth of the EAGLE-2 dynamic draft tree.
//
// "EAGLE 系列与 DFlash", §二 EAGLE-2 阶段一: every frontier node keeps its top-K
// tokens as children; "论文专题讲解：EAGLE-3", Draft tree 配置: 10 nodes are
// chosen per expansion, by draft confidence.
//
// Kernel 1 (one 16- or 8-CTA cluster per frontier row): each CTA reads its part
// of the row once into shared memory and keeps, as packed (value, id) keys (ties
// go to the lower token id), only the elements that can be among its k best: those
// not below the smallest warp maximum (or, when k exceeds the warp count or too
// many qualify, the k-th largest per-thread maximum), ranked exactly.  The row
// maximum, the fixed-point mass Q and each CTA's k best are combined through
// distributed shared memory; CTA 0 ranks the lists' keys and writes the k
// children.
// Kernel 2 (one CTA per request): sort the F*k children by (score desc,
// candidate index asc) in shared memory and emit the next frontier.
//
// eagle3_expand_sampled runs kernel 1's sampled variant: the k children are
// draws without replacement from the row's draft distribution ("EAGLE 系列与
// DFlash", §四 DFlash: drafts proposed by the drafter, checked with
// min(1, p_target / p_draft)), picked as the k earliest arrivals of the
// exponential race E_j / e_j with E_j = -ln U_j from a counter-based SplitMix64
// stream; kernel 2 is unchanged.
#include <cooperative_groups.h>

#include <mutex>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kExpandThreads = 512;
constexpr int kMaxCluster = 16;  // CTAs per frontier row (at most)
constexpr uint32_t kBulkPiece = 32768;  // bytes per bulk copy of the staged chunk

// candidate-list capacity and dynamic shared memory of one CTA (CL CTAs per row).
// The exact threshold admits only elements of the k threads whose maximum reaches
// it, so k times the elements one thread holds (a float4 slot is 4 of them) bounds
// the list.
int expand_cand_cap(int V, bool vec, int k, int CL) {
  const int nvec = vec ? V / 4 : V;
  const int per = (nvec + CL - 1) / CL;
  const int per_thread = (vec ? 4 : 1) * ((per + kExpandThreads - 1) / kExpandThreads);
  return k * per_thread + 32;
}
size_t expand_smem_bytes(int V, bool vec, int k, int CL) {
  const int nvec = vec ? V / 4 : V;
  const int per = (nvec + CL - 1) / CL;
  return static_cast<size_t>(per + 1) * 16 + static_cast<size_t>(expand_cand_cap(V, vec, k, CL)) * 8 + 16;
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

__device__ __forceinline__ uint32_t cl_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return r;
}
// asynchronous store into a peer's shared memory (cluster address a), completing
// its byte count on the peer's mbarrier at cluster address bar: the sender does
// not wait for the store to land
__device__ __forceinline__ void cl_st_async64(uint32_t a, uint64_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(a), "l"(v), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cl_st_async32(uint32_t a, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(a), "r"(v), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(b))),
               "r"(n));
}
// bounded wait (acquire at cluster scope) for phase 0 of a local mbarrier
__device__ __forceinline__ bool mb_wait0(uint64_t* b) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(b));
  uint64_t t0 = 0;
  for (int i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a)
        : "memory");
    if (ok) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    if (i == 0) t0 = t;
    if (t - t0 > 1000000000ull) return false;
  }
}

// One cluster of CL CTAs per frontier row.  CTA r stages chunk r of the row (scaled
// by 1/T) in shared memory.  Its top-k: candidates are the elements not below the
// smallest of the 16 warp maxima (at least 16 >= k elements qualify, typically a
// few dozen), ranked exactly; if more than fit, the exact threshold (k-th largest
// per-thread maximum, which admits at most k * per-thread elements) is used.
// Exchanges are asynchronous stores into the peers' shared memory that complete
// on the receivers' mbarriers (st.async, transaction bytes): every CTA sends its
// maximum key and non-finite flag to every CTA (each then knows the row maximum
// m), and its mass and top-k list to CTA 0, which ranks the CL lists' keys and
// writes the k children.
//
// SAMPLED: the children are drawn from the row's draft distribution instead of
// taken as its top k.  Once the row maximum m is known, each CTA makes one pass
// over its staged values that computes the fixed-point masses and overwrites
// each s_j with minus the token's arrival time E_j / e_j (e_j = E(s_j - m),
// E_j = -ln U_j from the counter-based stream), so that the same top-k machinery
// picks the k earliest arrivals; CTA 0 re-reads s of the chosen tokens for the
// scores and records the row's draft statistics.
template <int KMAX, bool SAMPLED>
__global__ void __launch_bounds__(kExpandThreads, 2)
expand_rows_kernel(const float* __restrict__ logits, int F, int V, int k, float it,
                   const float* __restrict__ parent_score, const int32_t* __restrict__ parent_id,
                   int depth, int cand_offset, e3_cand c, int32_t* dev_err, int cand_cap, uint64_t seed,
                   e3_qstat* qs) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.x / CL;  // b * F + f
  const int b = row / F, f = row % F;
  const float* z = logits + static_cast<size_t>(row) * V;
  extern __shared__ float4 chunk4[];
  __shared__ uint64_t warp_lists[kExpandThreads / 32][E3_MAX_TOPK];
  __shared__ uint64_t s_wmax[kExpandThreads / 32];
  __shared__ uint64_t ltop[E3_MAX_TOPK];              // this CTA's best k keys
  __shared__ uint64_t top[E3_MAX_TOPK];
  __shared__ uint64_t red64[32];
  __shared__ int s_cnt;
  // written by the peers
  __shared__ uint64_t s_pmax[kMaxCluster];            // each CTA's maximum key
  __shared__ uint32_t s_pbad[kMaxCluster];            // each CTA's non-finite flag
  __shared__ uint64_t s_pQ[kMaxCluster];              // (CTA 0) each CTA's mass
  __shared__ uint64_t s_ptop[kMaxCluster * E3_MAX_TOPK];  // (CTA 0) each CTA's top-k keys
  __shared__ uint64_t mx_bar, fin_bar, ld_bar;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
  const int nvec = vec ? (V >> 2) : V;
  const int per = (nvec + CL - 1) / CL;
  const int v0 = min(nvec, rank * per), v1 = min(nvec, v0 + per);
  float* chunk = reinterpret_cast<float*>(chunk4);
  const int e0 = vec ? 4 * v0 : v0;  // token id of chunk[0]
  const int n_local = vec ? 4 * (v1 - v0) : (v1 - v0);
  pdl_wait();  // the previous depth's frontier (parent ids and scores) is complete
  // the row's parent (id and score), needed by CTA 0's writers at the end: requested now
  float ps_row = 0.0f;
  int pid_row = -1;
  if (rank == 0 && threadIdx.x < k) {
    ps_row = parent_score[row];
    pid_row = parent_id[row];
  }
  if (threadIdx.x == 0) {
    mb_init(&mx_bar, 1);  // completed by the peers' asynchronous stores: 12 bytes from each
    mb_init(&fin_bar, 1);  // (CTA 0) completed by every CTA's mass and k keys: 8 (k + 1) bytes each
    mb_init(&ld_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(&mx_bar))),
                 "r"(static_cast<uint32_t>(CL) * 12u)
                 : "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(&fin_bar))),
                 "r"(static_cast<uint32_t>(CL) * 8u * static_cast<uint32_t>(k + 1))
                 : "memory");
    if (vec) {  // the chunk: bulk copies of 16-byte aligned row pieces
      const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&ld_bar));
      const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
      for (uint32_t off = 0; off < bytes; off += kBulkPiece) {
        const uint32_t n = min(kBulkPiece, bytes - off);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                static_cast<uint32_t>(__cvta_generic_to_shared(chunk4)) + off),
            "l"(reinterpret_cast<const unsigned char*>(z + 4 * static_cast<size_t>(v0)) + off), "r"(n), "r"(bar)
            : "memory");
      }
    }
  }
  // no thread polls a barrier before thread 0 has initialized it
  __syncthreads();
  // the peers' mbarriers are initialized before anyone arrives on them (waited
  // for just before the first exchange)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // the chunk is staged by the bulk copies above (16-byte aligned rows), else by
  // plain loads; then scaled by 1/T in place, with the per-thread maximum (first occurrence of the
  // largest value, i.e. the lowest token id among ties) and the non-finite flag
  float bv = -INFINITY;
  uint32_t bid = 0xFFFFFFFFu;
  int bad = 0;
  if (vec) {
    if (!mb_wait0(&ld_bar)) bad = 1;  // (flagged as non-finite: the row is skipped)
    for (int q = threadIdx.x; q < v1 - v0; q += blockDim.x) {
      float4 v = chunk4[q];
      if (it != 1.0f) {
        v.x = __fmul_rn(v.x, it);
        v.y = __fmul_rn(v.y, it);
        v.z = __fmul_rn(v.z, it);
        v.w = __fmul_rn(v.w, it);
        chunk4[q] = v;
      }
      bad |= !isfinite(v.x) | !isfinite(v.y) | !isfinite(v.z) | !isfinite(v.w);
      const uint32_t id = static_cast<uint32_t>(e0 + 4 * q);
      if (v.x > bv) bv = v.x, bid = id;
      if (v.y > bv) bv = v.y, bid = id + 1;
      if (v.z > bv) bv = v.z, bid = id + 2;
      if (v.w > bv) bv = v.w, bid = id + 3;
    }
  } else {
#pragma unroll 4
    for (int j = v0 + threadIdx.x; j < v1; j += blockDim.x) {
      const float v = __fmul_rn(__ldg(z + j), it);
      chunk[j - v0] = v;
      bad |= !isfinite(v);
      if (v > bv) bv = v, bid = static_cast<uint32_t>(j);
    }
  }
  const uint64_t tmax = bid == 0xFFFFFFFFu ? 0ull : pack_best(bv, bid);
  // the dependent frontier kernel may be scheduled (it waits for this grid to finish)
  pdl_trigger();
  const uint64_t wmax = warp_reduce(tmax, MaxU64());
  if (lane == 0) s_wmax[warp] = wmax;
  if (threadIdx.x == 0) s_cnt = 0;
  bad = __syncthreads_or(bad);
  // send this CTA's maximum key and flag to every CTA of the cluster now; the
  // candidate selection below runs while they travel
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (threadIdx.x < CL) {
    uint64_t lbest = 0ull;
    for (int w = 0; w < kExpandThreads / 32; ++w) lbest = max(lbest, s_wmax[w]);
    const uint32_t bar = cl_addr(&mx_bar, threadIdx.x);
    cl_st_async64(cl_addr(&s_pmax[rank], threadIdx.x), lbest, bar);
    cl_st_async32(cl_addr(&s_pbad[rank], threadIdx.x), static_cast<uint32_t>(bad), bar);
  }
  // each thread visits the chunk elements it staged: float4 slots q - v0 (vec) or j - v0
  auto for_own = [&](auto&& fn) {
    if (vec) {
      for (int q = threadIdx.x; q < v1 - v0; q += blockDim.x) {
        const float4 v = chunk4[q];
        const uint32_t id = static_cast<uint32_t>(e0 + 4 * q);
        fn(v.x, id);
        fn(v.y, id + 1);
        fn(v.z, id + 2);
        fn(v.w, id + 3);
      }
    } else {
      for (int j = threadIdx.x; j < n_local; j += blockDim.x) fn(chunk[j], static_cast<uint32_t>(e0 + j));
    }
  };
  uint64_t* cand = reinterpret_cast<uint64_t*>(chunk4 + (per + 1));
  // this CTA's best k keys of the staged values -> ltop[] (s_wmax holds the warp
  // maxima of the per-thread best keys tkey, s_cnt is 0; both visible)
  auto local_topk = [&](uint64_t tkey) {
    uint64_t thr = ~0ull;
    if (k <= kExpandThreads / 32) {
      for (int w = 0; w < kExpandThreads / 32; ++w) thr = min(thr, s_wmax[w]);
      // value part of the threshold: a cheap first filter (none if some warp has no element)
      const float thr_v = thr == 0ull ? -INFINITY : unord_f32(static_cast<uint32_t>(thr >> 32));
      for_own([&](float v, uint32_t id) {
        if (v < thr_v) return;
        const uint64_t key = pack_best(v, id);
        if (key >= thr && key != 0ull) {
          const int at = atomicAdd(&s_cnt, 1);
          if (at < cand_cap) cand[at] = key;
        }
      });
    }
    __syncthreads();
    if (k > kExpandThreads / 32 || s_cnt > cand_cap) {
      // exact threshold: the k-th largest per-thread maximum
      {
        uint64_t v = tkey;
        for (int r = 0; r < k; ++r) {
          const uint64_t bst = warp_reduce(v, MaxU64());
          if (v == bst) v = 0ull;  // keys are distinct: exactly one lane (or all-zero lanes)
          if (lane == 0) warp_lists[warp][r] = bst;
        }
      }
      __syncthreads();
      if (warp == 0) {
        const int nw = blockDim.x >> 5;
        uint64_t lk[KMAX];
#pragma unroll
        for (int i = 0; i < KMAX; ++i) lk[i] = (lane < nw && i < k) ? warp_lists[lane][i] : 0ull;
        warp_merge_topk(lk, k, top);
      }
      if (threadIdx.x == 0) s_cnt = 0;
      __syncthreads();
      thr = top[k - 1];
      const float thr_v = thr == 0ull ? -INFINITY : unord_f32(static_cast<uint32_t>(thr >> 32));
      for_own([&](float v, uint32_t id) {
        if (v < thr_v) return;
        const uint64_t key = pack_best(v, id);
        if (key >= thr && key != 0ull) {
          const int at = atomicAdd(&s_cnt, 1);
          if (at < cand_cap) cand[at] = key;
        }
      });
      __syncthreads();
    }
    // (the bound above makes this unreachable; a dropped key would be a wrong child)
    if (threadIdx.x == 0 && s_cnt > cand_cap) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
    const int ncand = min(s_cnt, cand_cap);
    if (threadIdx.x < E3_MAX_TOPK) ltop[threadIdx.x] = 0ull;
    __syncthreads();
    for (int i = threadIdx.x; i < ncand; i += blockDim.x) {
      const uint64_t key = cand[i];
      int rnk = 0;
#pragma unroll 8
      for (int j = 0; j < ncand; ++j) rnk += cand[j] > key;
      if (rnk < k) ltop[rnk] = key;
    }
  };
  if constexpr (!SAMPLED) local_topk(tmax);
  const bool got = mb_wait0(&mx_bar);
  uint64_t gbest = 0ull;
  uint32_t gbad = got ? 0u : 1u;
  for (int r = 0; r < CL; ++r) {
    gbest = max(gbest, s_pmax[r]);
    gbad |= s_pbad[r];
  }
  if (!got) {
    if (threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_TIMEOUT);
    return;
  }
  if (gbad) {
    if (rank == 0 && threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_NONFINITE);
    return;  // every CTA saw the same flags; no further exchange
  }
  const float m = unord_f32(static_cast<uint32_t>(gbest >> 32));
  uint64_t Q = 0;
  if constexpr (SAMPLED) {
    // masses, and minus the arrival time of every token, in place
    const uint64_t ctr = (static_cast<uint64_t>(b) << 44) | (static_cast<uint64_t>(depth) << 36) |
                         (static_cast<uint64_t>(f) << 24);
    uint64_t tbest = 0ull;
    auto draw = [&](float sv, uint32_t id) -> float {
      const float e = fx_exp(__fsub_rn(sv, m));
      const uint64_t q = fx_scale40_floor(e);
      Q += q;
      float v = -INFINITY;  // a token of zero mass never arrives
      if (q != 0ull) {
        const uint64_t u24 = splitmix64_at(seed, ctr + id + 1) >> 40;
        const float E = __fsub_rn(0.0f, fx_ell((u24 + 1ull) << 16));
        v = __fsub_rn(0.0f, __fdiv_rn(E, e));
      }
      tbest = max(tbest, pack_best(v, id));
      return v;
    };
    __syncthreads();  // every read of s_wmax for the max exchange is done
    if (vec) {
      for (int q = threadIdx.x; q < v1 - v0; q += blockDim.x) {
        float4 v = chunk4[q];
        const uint32_t id = static_cast<uint32_t>(e0 + 4 * q);
        v.x = draw(v.x, id);
        v.y = draw(v.y, id + 1);
        v.z = draw(v.z, id + 2);
        v.w = draw(v.w, id + 3);
        chunk4[q] = v;
      }
    } else {
      for (int j = threadIdx.x; j < n_local; j += blockDim.x) chunk[j] = draw(chunk[j], static_cast<uint32_t>(e0 + j));
    }
    const uint64_t wbest = warp_reduce(tbest, MaxU64());
    if (lane == 0) s_wmax[warp] = wbest;
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    local_topk(tbest);
  } else if (vec) {
    for (int q = threadIdx.x; q < v1 - v0; q += blockDim.x) {
      const float4 v = chunk4[q];
      Q += fx_mass_x2(v.x, v.y, m) + fx_mass_x2(v.z, v.w, m);
    }
  } else {
    for_own([&](float v, uint32_t) { Q += fx_mass(v, m); });
  }
  Q = block_reduce(Q, SumU64(), red64);  // also orders ltop[] before thread 0 reads it
  // mass (thread 0) and top-k list (threads 1..k) to CTA 0, as asynchronous stores
  // completing on its fin_bar (register values: nothing of this CTA is read later)
  if (threadIdx.x <= k) {
    const uint32_t bar = cl_addr(&fin_bar, 0);
    if (threadIdx.x == 0)
      cl_st_async64(cl_addr(&s_pQ[rank], 0), Q, bar);
    else
      cl_st_async64(cl_addr(&s_ptop[rank * k + threadIdx.x - 1], 0), ltop[threadIdx.x - 1], bar);
  }
  if (rank != 0) return;  // nothing reads this CTA's shared memory any more
  const bool fin = mb_wait0(&fin_bar);
  if (!fin) {
    if (threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_TIMEOUT);
    return;
  }
  // the row's k best of the CL lists (distinct keys, zero-padded): each key's rank
  // among all CL * k of them
  if (threadIdx.x < k) top[threadIdx.x] = 0ull;
  __syncthreads();
  for (int i = threadIdx.x; i < CL * k; i += blockDim.x) {
    const uint64_t key = s_ptop[i];
    if (key == 0ull) continue;
    int rnk = 0;
#pragma unroll 8
    for (int j = 0; j < CL * k; ++j) rnk += s_ptop[j] > key;
    if (rnk < k) top[rnk] = key;
  }
  __shared__ uint64_t s_Qt;
  if (threadIdx.x == 0) {
    uint64_t t = 0;
    for (int r = 0; r < CL; ++r) t += s_pQ[r];
    s_Qt = t;
  }
  __syncthreads();
  if (SAMPLED && threadIdx.x == 0) {
    const int pid = pid_row;
    if (pid >= -1 && pid < c.cap) {
      e3_qstat st;
      st.row = z;
      st.Q = s_Qt;
      st.m = m;
      st.inv_temp = it;
      qs[static_cast<size_t>(b) * (c.cap + 1) + (pid + 1)] = st;
    }
  }
  if (threadIdx.x < k) {
    const int r = threadIdx.x;
    const float ell = fx_ell(s_Qt);
    const uint32_t t = packed_id(top[r]);
    const float sc = SAMPLED ? (t < static_cast<uint32_t>(V) ? __fmul_rn(__ldg(z + t), it) : -INFINITY)
                             : unord_f32(static_cast<uint32_t>(top[r] >> 32));
    const float ps = ps_row;
    const size_t ci = static_cast<size_t>(b) * c.cap + cand_offset + f * k + r;
    c.tok[ci] = static_cast<int32_t>(t);
    c.parent[ci] = pid_row;
    c.score[ci] = __fsub_rn(__fadd_rn(ps, __fsub_rn(sc, m)), ell);
    c.depth[ci] = depth;
  }
}

// Clusters of 16 CTAs (half the work per CTA) where every row of the call still
// fits one wave of such clusters, else clusters of 8.
template <int KMAX, bool SAMPLED>
int cluster_size_for(int rows, int V, bool vec, int k) {
  static std::mutex mu;  // the cache below is read and refreshed as a unit
  const std::lock_guard<std::mutex> lock(mu);
  static int cached_v = -1, cached_k = -1, max16 = 0;
  if (cached_v != V || cached_k != k) {
    max16 = 0;
    if (cudaFuncSetAttribute(expand_rows_kernel<KMAX, SAMPLED>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(kExpandThreads);
      cfg.dynamicSmemBytes = expand_smem_bytes(V, vec, k, 16);
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 16;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, expand_rows_kernel<KMAX, SAMPLED>, &cfg) == cudaSuccess) max16 = n;
    }
    cudaGetLastError();
    cached_v = V;
    cached_k = k;
  }
  return rows <= max16 ? 16 : 8;
}

template <int KMAX, bool SAMPLED>
e3_status launch_rows(const float* logits, int rows, int F, int V, int k, float inv_temp, const float* parent_score,
                      const int32_t* parent_id, int depth, int cand_offset, const e3_cand& c, uint64_t seed,
                      e3_qstat* qs, int32_t* dev_err, cudaStream_t s) {
  // one-time setup (a function-local static is initialised once, thread-safely)
  static const bool attr_done = (cudaFuncSetAttribute(expand_rows_kernel<KMAX, SAMPLED>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024),
                                 true);
  (void)attr_done;
  const bool vec = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  const int CL = cluster_size_for<KMAX, SAMPLED>(rows, V, vec, k);
  const int cand_cap = expand_cand_cap(V, vec, k, CL);
  const size_t smem = expand_smem_bytes(V, vec, k, CL);
  E3_REQUIRE(smem <= 200 * 1024, E3_ERR_SHAPE, "eagle3_expand: V=%d too large", V);
  const cudaError_t e = launch_pdl(expand_rows_kernel<KMAX, SAMPLED>, dim3(rows * CL), dim3(kExpandThreads), smem,
                                   s, static_cast<unsigned>(CL), logits, F, V, k, inv_temp, parent_score, parent_id,
                                   depth, cand_offset, c, dev_err, cand_cap, seed, qs);
  if (e != cudaSuccess) return cuda_status(e, "expand_rows_kernel");
  return E3_OK;
}

}  // namespace

namespace {

__global__ void __launch_bounds__(256)
expand_frontier_kernel(int n, int Wn, int cand_offset, e3_cand c, int32_t* next_id, float* next_score,
                       const int32_t* dev_err) {
  // launched as a programmatic dependent of the row kernel: wait for its results
  pdl_wait();
  pdl_trigger();
  __shared__ uint64_t keys[2048];
  __shared__ float sc[1024];
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int ci = cand_offset + i;
    const float v = c.score[static_cast<size_t>(b) * c.cap + ci];
    keys[i] = pack_best(v, static_cast<uint32_t>(ci));
    if (n <= 1024) sc[i] = v;
  }
  __syncthreads();
  if (n <= 1024) {
    // exact rank of each child among the n (distinct keys): the first Wn ranks win
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t key = keys[i];
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < n; ++j) rank += keys[j] > key;
      if (rank < Wn) {
        next_id[static_cast<size_t>(b) * Wn + rank] = static_cast<int32_t>(cand_offset + i);
        next_score[static_cast<size_t>(b) * Wn + rank] = sc[i];
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

template <bool SAMPLED>
e3_status launch_rows_k(const float* logits, int rows, int F, int V, int k, float inv_temp, const float* parent_score,
                        const int32_t* parent_id, int depth, int cand_offset, const e3_cand& c, uint64_t seed,
                        e3_qstat* qs, int32_t* dev_err, cudaStream_t s) {
  if (k <= 2)
    return launch_rows<2, SAMPLED>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c,
                                   seed, qs, dev_err, s);
  if (k <= 4)
    return launch_rows<4, SAMPLED>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c,
                                   seed, qs, dev_err, s);
  if (k <= 8)
    return launch_rows<8, SAMPLED>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c,
                                   seed, qs, dev_err, s);
  if (k <= 16)
    return launch_rows<16, SAMPLED>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c,
                                    seed, qs, dev_err, s);
  return launch_rows<32, SAMPLED>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c,
                                  seed, qs, dev_err, s);
}

}  // namespace

e3_status launch_expand(const float* logits, int B, int F, int V, int k, int W, float inv_temp,
                        const float* parent_score, const int32_t* parent_id, int depth,
                        int cand_offset, const e3_cand& c, int32_t* next_id, float* next_score, bool sampled,
                        uint64_t seed, e3_qstat* q_stats, int32_t* dev_err, cudaStream_t s) {
  const int rows = B * F;
  const e3_status st =
      sampled ? launch_rows_k<true>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c,
                                    seed, q_stats, dev_err, s)
              : launch_rows_k<false>(logits, rows, F, V, k, inv_temp, parent_score, parent_id, depth, cand_offset, c,
                                     0ull, nullptr, dev_err, s);
  if (st != E3_OK) return st;
  const int n = F * k;
  const int Wn = W < n ? W : n;
  // programmatic dependent launch: the frontier kernel is scheduled while the row
  // kernel drains and waits (griddepcontrol.wait) for its completion
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, expand_frontier_kernel, n, Wn, cand_offset, c, next_id, next_score,
                                     static_cast<const int32_t*>(dev_err));
  if (e != cudaSuccess) return cuda_status(e, "expand_frontier_kernel");
  note_launch();
  return E3_OK;
}

}  // namespace e3
