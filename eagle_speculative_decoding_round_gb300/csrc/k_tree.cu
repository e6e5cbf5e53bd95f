// k_tree.cu -- tree_build_mask: rerank, flatten, positions, ancestor bit mask.
//
// "EAGLE 系列与 DFlash", §二 EAGLE-2 阶段二: the tree is flattened to one
// sequence [x_1, x_2, x_3, x_1a, x_1b, x_1c, x_2a, ...]; 关键新增步骤① gives every
// node a position from its depth; 关键新增步骤② builds the 0/1 tree mask in which
// x_1a sees only x_1 and the root, never its cousin x_2.
// "SpecForge…", 从序列到动态草稿树: the node budget goes to the most confident
// candidates.
//
// One CTA per request.  Selection: with one key per thread (up to 1024
// candidates) each warp sorts its 32 keys (score desc, index asc) through
// shuffles, and a key's rank among all candidates is its lane plus, for every
// other warp's sorted list, a binary-searched count of the keys above it; the
// keys of rank < N are kept.  Beyond 1024 candidates a shared-memory bitonic
// sort over 1024 threads orders them.  Flattening runs depth by depth on the
// warps that hold the N kept nodes, each node on its own thread: a level's nodes
// are ranked by (parent's flat index, candidate index), and each node's mask row
// is its parent's row plus its own bit.  Optionally the candidate index of every
// flat node is written (node_cand), which is how the sampled accept finds the
// draft row a node's children were drawn from.
#include <algorithm>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kTreeThreads = 256;  // at least E3_MAX_NODES + 1 (one thread per flat row)

// Descending bitonic sort of the 32 keys of a warp, one per lane, through shuffles.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
      const bool lower = (lane & j) == 0;  // the lower lane of the pair keeps the larger key...
      const bool desc = (lane & kk) == 0;  // ...in the descending halves of the merge
      v = (lower == desc) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Number of high words above xh in a descending list of 32 keys' high words (binary
// search: those words form a prefix of the list).  Keys whose high word equals xh
// follow that prefix, ordered by their low words.
__device__ __forceinline__ int count_hi_above32(const uint32_t* H, uint32_t xh) {
  int c = H[15] > xh ? 16 : 0;
  c += H[c + 7] > xh ? 8 : 0;
  c += H[c + 3] > xh ? 4 : 0;
  c += H[c + 1] > xh ? 2 : 0;
  c += H[c] > xh ? 1 : 0;
  c += (c == 31 && H[31] > xh) ? 1 : 0;
  return c;
}

__device__ __forceinline__ void sync_first(int nthreads) {  // barrier 1 over the first nthreads threads
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

__global__ void __launch_bounds__(1024)
tree_build_kernel(e3_cand c, int n_cand, int N, const int32_t* __restrict__ root_tok,
                  const int32_t* __restrict__ kv_len, int32_t* tok, int32_t* parent, int32_t* depth,
                  int32_t* pos, uint64_t* mask, int32_t* node_cand) {
  extern __shared__ uint64_t sh[];
  __shared__ int sel[E3_MAX_NODES];               // candidate of the r-th best key
  __shared__ int lkey[E3_MAX_NODES];              // one level's (parent flat, candidate) keys
  __shared__ uint64_t rows[E3_MAX_NODES + 1][4];  // ancestor-or-self bit rows by flat index
  __shared__ int cnt[E3_MAX_DEPTH + 2];           // kept nodes per depth (1 .. E3_MAX_DEPTH)
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
  int np = 1;
  while (np < n_cand) np <<= 1;
  const bool per_thread = np <= static_cast<int>(blockDim.x);  // one key per thread
  uint64_t* keys = sh;  // [max(np, blockDim.x)]: sorted warp lists, or the whole sort
  uint32_t* whi = reinterpret_cast<uint32_t*>(keys + max(np, static_cast<int>(blockDim.x)));  // [blockDim.x] (per_thread)
  int* cdat = reinterpret_cast<int*>(whi + (per_thread ? blockDim.x : 0));  // [3][n_cand] (per_thread)
  int16_t* flat_of = reinterpret_cast<int16_t*>(cdat + (per_thread ? 3 * n_cand : 0));  // [n_cand]
  const size_t cb = static_cast<size_t>(b) * c.cap;
  for (int q = i; q < n_cand; q += blockDim.x) flat_of[q] = -1;
  if (i < E3_MAX_DEPTH + 2) cnt[i] = 0;
  const int P = kv_len[b];
  if (per_thread) {
    uint64_t v = 0ull;  // padding keys (0) rank below every candidate's key
    if (i < n_cand) {
      v = pack_best(c.score[cb + i], static_cast<uint32_t>(i));
      cdat[i] = c.depth[cb + i];
      cdat[n_cand + i] = c.parent[cb + i];
      cdat[2 * n_cand + i] = c.tok[cb + i];
    }
    v = warp_sort_desc(v);
    keys[i] = v;
    whi[i] = static_cast<uint32_t>(v >> 32);
    __syncthreads();
    // lists in order, eight searches at a time (independent chains of loads, taken
    // without branches: a search outside the lists or of the warp's own list reads a
    // valid list and counts 0); a lane stops once its rank reaches N (candidates of the
    // first depths, which hold most of the best keys, come first), the warp once all
    // its lanes have
    const int nl = (n_cand + 31) >> 5;  // warps holding candidates
    int rank = lane;
    bool live = v != 0ull && lane < N;
    const uint32_t vh = static_cast<uint32_t>(v >> 32);
    for (int q0 = 0; q0 < nl && __any_sync(0xFFFFFFFFu, live); q0 += 8) {
      if (live) {
        // counts over the high words (32-bit loads); a list whose next high word
        // equals vh holds a score tie, settled on the full keys
        int cs[8];
        bool tie = false;
#pragma unroll
        for (int u = 0; u < 8; ++u) cs[u] = count_hi_above32(whi + 32 * min(q0 + u, nl - 1), vh);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int q = q0 + u;
          const bool valid = q < nl && q != warp;
          tie |= valid && cs[u] < 32 && whi[32 * min(q, nl - 1) + min(cs[u], 31)] == vh;
        }
        if (tie) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int q = q0 + u;
            if (q < nl && q != warp)
              while (cs[u] < 32 && keys[32 * q + cs[u]] > v) ++cs[u];
          }
        }
        int add = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) add += (q0 + u < nl && q0 + u != warp) ? cs[u] : 0;
        rank += add;
        live = rank < N;
      }
    }
    if (v != 0ull && rank < N) sel[rank] = static_cast<int>(packed_id(v));
  } else {
    for (int q = i; q < np; q += blockDim.x)
      keys[q] = q < n_cand ? pack_best(c.score[cb + q], static_cast<uint32_t>(q)) : 0ull;
    __syncthreads();
    block_bitonic_desc(keys, np);
    if (i < N) sel[i] = static_cast<int>(packed_id(keys[i]));
  }
  __syncthreads();
  // from here on only the warps of the N kept nodes and the root row take part
  const int nthr = ((N + 1 + 31) >> 5) << 5;
  if (i >= nthr) return;
  int my_d = 0, lpos = 0, my_c = 0, my_p = -1, my_t = 0;
  if (i < N) {
    my_c = sel[i];
    int d;
    if (per_thread) {
      d = cdat[my_c];
      my_p = cdat[n_cand + my_c];
      my_t = cdat[2 * n_cand + my_c];
    } else {
      d = c.depth[cb + my_c];
      my_p = c.parent[cb + my_c];
      my_t = c.tok[cb + my_c];
    }
    if (my_p >= n_cand) my_p = -1;  // malformed parent: hang the node off the root
    my_d = min(max(d, 1), E3_MAX_DEPTH);
    lpos = atomicAdd(&cnt[my_d], 1);  // position within the level (any order: levels are ranked below)
  }
  sync_first(nthr);
  if (i == 0) {
    rows[0][0] = 1ull;
    rows[0][1] = rows[0][2] = rows[0][3] = 0ull;
  }
  // the level sizes (each below 2^8), packed eight to a register so that the level
  // loop reads none of them from shared memory
  uint64_t lv_lo = 0ull, lv_hi = 0ull;
  int maxd = 0;
#pragma unroll
  for (int d = 1; d <= E3_MAX_DEPTH; ++d) {
    const uint64_t n = static_cast<uint64_t>(cnt[d]);
    if (d <= 8)
      lv_lo |= n << (8 * (d - 1));
    else
      lv_hi |= n << (8 * (d - 9));
    if (n > 0) maxd = d;
  }
  sync_first(nthr);
  const int R = N + 1;
  const int words = (R + 63) >> 6;
  // flat indices level by level, each node handled by the thread that holds it:
  // rank among the level's nodes by (parent's flat index, candidate index), packed
  // into one integer key (both below 2^12); a parent not yet flattened (not kept,
  // or not at a smaller depth) counts as the root
  int base = 1;  // flat index of the level's first node
  for (int d = 1; d <= maxd; ++d) {
    const int n = static_cast<int>(((d <= 8 ? lv_lo : lv_hi) >> (8 * ((d - 1) & 7))) & 0xFFu);
    if (n == 0) continue;  // uniform across the threads taking part
    const bool mine = i < N && my_d == d;
    int pf = 0, key = 0;
    uint64_t prow[4] = {0ull, 0ull, 0ull, 0ull};
    if (mine) {
      pf = my_p < 0 ? 0 : flat_of[my_p];
      if (pf < 0) pf = 0;
      key = (pf << 12) | my_c;
      lkey[lpos] = key;
#pragma unroll
      for (int w = 0; w < 4; ++w)  // final: pf is on an earlier level
        if (w < words) prow[w] = rows[pf][w];
    }
    sync_first(nthr);
    if (mine) {
      int rank = 0;
#pragma unroll 8
      for (int q = 0; q < n; ++q) rank += lkey[q] < key;
      const int f = base + rank;
      flat_of[my_c] = static_cast<int16_t>(f);
#pragma unroll
      for (int w = 0; w < 4; ++w)
        if (w < words) rows[f][w] = prow[w] | (w == (f >> 6) ? 1ull << (f & 63) : 0ull);
      const size_t o = static_cast<size_t>(b) * R + f;
      tok[o] = my_t;
      parent[o] = pf;
      depth[o] = d;
      pos[o] = P + d;
      if (node_cand) node_cand[o] = my_c;
    }
    base += n;
    sync_first(nthr);
  }
  if (i == 0) {
    const size_t o = static_cast<size_t>(b) * R;
    tok[o] = root_tok[b];
    parent[o] = -1;
    depth[o] = 0;
    pos[o] = P;
    if (node_cand) node_cand[o] = -1;
  }
  if (i < R) {
    uint64_t* row = mask + (static_cast<size_t>(b) * R + i) * words;
    for (int w = 0; w < words; ++w) row[w] = rows[i][w];
  }
}

}  // namespace

e3_status launch_tree_build(const e3_cand& c, int B, int n_cand, int N, const int32_t* root_tok,
                            const int32_t* kv_len, int32_t* tok, int32_t* parent, int32_t* depth,
                            int32_t* pos, uint64_t* mask, int32_t* node_cand, cudaStream_t s) {
  int np = 1;
  while (np < n_cand) np <<= 1;
  // one thread per key up to 1024 keys (warp sorts and ranks), else 1024 threads
  // over a shared-memory sort
  const int threads = std::max(kTreeThreads, std::min(np, 1024));
  const bool per_thread = np <= threads;
  const size_t smem = static_cast<size_t>(std::max(np, threads)) * 8 +
                      (per_thread ? static_cast<size_t>(threads) * 4 + static_cast<size_t>(n_cand) * 12 : 0) +
                      static_cast<size_t>(n_cand) * 2 + 16;
  // the kernel's static arrays: node tables, level keys, ancestor rows, depth counts
  constexpr size_t kStatic = 2 * sizeof(int) * E3_MAX_NODES + 32 * (E3_MAX_NODES + 1) + 4 * (E3_MAX_DEPTH + 2);
  if (smem + kStatic > 48 * 1024) {
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
