// k_draft.cu -- eagle3_draft_step: the drafter's single decoder layer over the
// frontier rows of one depth of the draft tree.
//
// "论文专题讲解：EAGLE-3", 推理流程：多层特征融合 + 单层 draft decoder: one decoder
// layer; the first step reads the fused feature g and the token's embedding, a
// later step the output a of the step that proposed its token ("SpecForge…", 第二步
// 为什么没有"正确隐藏状态"可用), and a tree node attends to its ancestors only (从
// 序列到动态草稿树).  Readings where the pages leave the layer open: the two inputs
// are concatenated [e(tok); h] and projected by one linear layer, and the layer is a
// pre-norm block of the target family (RMSNorm, grouped-query attention with rotary
// positions, SwiGLU MLP); the draft logits are W_lm RMSNorm(a).
//
// A step is a chain of launches on one stream, each a programmatic dependent of the
// one before:
//   prep        slots, positions, mask rows; gathers e(tok) and h into GEMM operands
//   W_in        split-K tcgen05 GEMM over the two sources (k_tcgemm.cu)
//   norm        split-K reduction, x (fp32), RMSNorm -> y (bf16)
//   W_qkv       GEMM;  qkv: reduction, rotary, q into the attention's query rows,
//               k and v into the drafter's paged cache at the row's tree slot
//   attention   tree_verify_attn over the drafter's cache (all tree slots so far)
//   gather      the frontier rows of the attention output
//   W_o         GEMM;  norm: x += W_o o, RMSNorm -> y
//   W_gu        GEMM;  swiglu: silu(gate) * up (bf16)
//   W_down      GEMM;  norm: a = x + W_down h (fp32, kept per tree slot), RMSNorm -> y
//   LM head     lmhead_logits (tcgen05) of y: the draft logits and their statistics
// The activations between launches are a few rows (B x F) and stay in L2; the
// step's time is the weights streamed by the GEMMs and the LM head.
#include <math.h>

#include <algorithm>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kThreads = 256;

struct PrepArgs {
  int F, depth, slot_base, F_prev, slot_base_prev, R_slots, words, d, V, cap;
  const int32_t* frontier;
  const int32_t* frontier_prev;
  const int32_t* c_tok;
  const int32_t* c_parent;
  const int32_t* root_tok;
  const int32_t* kv_len;
  const __nv_bfloat16* emb;
  const __nv_bfloat16* g;
  const float* a_slots;
  uint64_t* mask;
  __nv_bfloat16* e_rows;
  __nv_bfloat16* h_rows;
  int32_t* row_slot;
  int32_t* row_pos;
  float* ones;
  int32_t* dev_err;
};

// One CTA per frontier row m = b * F + f.
__global__ void __launch_bounds__(kThreads) draft_prep_kernel(PrepArgs p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_tok, s_pslot;
  const int m = blockIdx.x, b = m / p.F, f = m - b * p.F;
  const int slot = p.slot_base + f;
  if (threadIdx.x == 0) {
    const int u = p.frontier[m];
    int tok = 0, pslot = -1;
    bool ok = true;
    if (p.depth == 1) {
      tok = p.root_tok[b];
    } else if (u >= 0 && u < p.cap) {
      tok = p.c_tok[static_cast<size_t>(b) * p.cap + u];
      const int pc = p.c_parent[static_cast<size_t>(b) * p.cap + u];
      for (int j = 0; j < p.F_prev; ++j)
        if (p.frontier_prev[static_cast<size_t>(b) * p.F_prev + j] == pc) {
          pslot = p.slot_base_prev + j;
          break;
        }
      ok = pslot >= 0;
    } else {
      ok = false;
    }
    if (tok < 0 || tok >= p.V) {
      tok = 0;
      ok = false;
    }
    if (!ok) dev_flag(p.dev_err, E3_DEV_ERR_CAPACITY);
    s_tok = tok;
    s_pslot = pslot;
    p.row_slot[m] = slot;
    p.row_pos[m] = p.kv_len[b] + p.depth - 1;
    p.ones[m] = 1.0f;
  }
  __syncthreads();
  const int tok = s_tok, pslot = s_pslot;
  uint64_t* mrow = p.mask + (static_cast<size_t>(b) * p.R_slots) * p.words;
  if (p.depth == 1) {
    // every row of the request: its own bit only (rows not yet in the tree are computed
    // by the attention call but never read)
    for (int i = threadIdx.x; i < p.R_slots * p.words; i += blockDim.x) {
      const int r = i / p.words, w = i - r * p.words;
      mrow[i] = (w == (r >> 6)) ? (1ull << (r & 63)) : 0ull;
    }
  } else if (threadIdx.x < p.words) {
    uint64_t v = pslot >= 0 ? mrow[static_cast<size_t>(pslot) * p.words + threadIdx.x] : 0ull;
    if (threadIdx.x == (slot >> 6)) v |= 1ull << (slot & 63);
    mrow[static_cast<size_t>(slot) * p.words + threadIdx.x] = v;
  }
  // GEMM operands: e(tok) and h (g at the root, the parent's a afterwards) as bf16 rows
  const uint4* esrc = reinterpret_cast<const uint4*>(p.emb + static_cast<size_t>(tok) * p.d);
  uint4* edst = reinterpret_cast<uint4*>(p.e_rows + static_cast<size_t>(m) * p.d);
  for (int i = threadIdx.x; i < p.d / 8; i += blockDim.x) edst[i] = esrc[i];
  __nv_bfloat16* hdst = p.h_rows + static_cast<size_t>(m) * p.d;
  if (p.depth == 1) {
    const uint4* gsrc = reinterpret_cast<const uint4*>(p.g + static_cast<size_t>(b) * p.d);
    for (int i = threadIdx.x; i < p.d / 8; i += blockDim.x) reinterpret_cast<uint4*>(hdst)[i] = gsrc[i];
  } else {
    const float* asrc = p.a_slots + (static_cast<size_t>(b) * p.R_slots + max(pslot, 0)) * p.d;
    for (int i = threadIdx.x; i < p.d / 2; i += blockDim.x) {
      const float2 v = reinterpret_cast<const float2*>(asrc)[i];
      reinterpret_cast<uint32_t*>(hdst)[i] = pack2_bf16(v.x, v.y);
    }
  }
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.0f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
  __syncthreads();
  return t;
}

struct NormArgs {
  const float* part;
  int splits, M, N;
  const float* resid;  // nullable: x = resid + sum of partials
  float* x_out;        // fp32 x (may alias resid)
  const float* w;      // RMSNorm weight [N]
  float eps;
  __nv_bfloat16* y;    // bf16 RMSNorm(x) * w
  float* slot_out;     // nullable: x also to slot_out[b][row_slot[m]]
  const int32_t* row_slot;
  int F, R_slots;
};

// One CTA per row: the split-K sum (in split order), the residual, RMSNorm.
__global__ void __launch_bounds__(kThreads) draft_norm_kernel(NormArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float xs[];
  __shared__ float red[kThreads / 32];
  const int m = blockIdx.x;
  const size_t plane = static_cast<size_t>(a.M) * a.N;
  float ss = 0.0f;
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const size_t e = static_cast<size_t>(m) * a.N + i;
    float v = 0.0f;
    for (int z = 0; z < a.splits; ++z) v += a.part[z * plane + e];
    if (a.resid) v += a.resid[e];
    xs[i] = v;
    ss += v * v;
  }
  const float inv = rsqrtf(block_sum(ss, red) / static_cast<float>(a.N) + a.eps);
  float* srow = a.slot_out ? a.slot_out + (static_cast<size_t>(m / a.F) * a.R_slots + a.row_slot[m]) * a.N : nullptr;
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const size_t e = static_cast<size_t>(m) * a.N + i;
    a.x_out[e] = xs[i];
    a.y[e] = __float2bfloat16_rn(xs[i] * inv * a.w[i]);
    if (srow) srow[i] = xs[i];
  }
}

struct QkvArgs {
  const float* part;
  int splits, M, H, KVH, hd;
  float rope_base;
  const int32_t* row_slot;
  const int32_t* row_pos;
  int F, R_slots;
  __nv_bfloat16* Q;  // [B][R_slots][H][hd]
  __nv_bfloat16* kc;
  __nv_bfloat16* vc;
  const int32_t* page_table;
  int max_pages, n_pages, page_size;
  const int32_t* kv_len;
  int32_t* dev_err;
};

// One CTA per row: rotary position on q and k, q into the attention's query row of
// the row's slot, k and v into the drafter's cache at logical position kv_len + slot.
__global__ void __launch_bounds__(kThreads) draft_qkv_kernel(QkvArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float cs[128], sn[128];  // cos / sin of the row's angles (hd / 2 <= 128)
  __shared__ int s_row;                // cache row of the slot (-1: no page)
  const int m = blockIdx.x, b = m / a.F;
  const int slot = a.row_slot[m], pos = a.row_pos[m];
  const int half = a.hd / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    // the angle in double precision (positions reach 10^5 and beyond), then fp32
    const double ang = static_cast<double>(pos) * pow(static_cast<double>(a.rope_base), -2.0 * i / a.hd);
    double sd, cd;
    sincos(ang, &sd, &cd);
    cs[i] = static_cast<float>(cd);
    sn[i] = static_cast<float>(sd);
  }
  if (threadIdx.x == 0) {
    const int t = a.kv_len[b] + slot;
    const int pi = t / a.page_size;
    int row = -1;
    if (t >= 0 && pi < a.max_pages) {
      const int pg = a.page_table[static_cast<size_t>(b) * a.max_pages + pi];
      if (pg >= 0 && pg < a.n_pages) row = pg * a.KVH * a.page_size + t % a.page_size;
    }
    if (row < 0) dev_flag(a.dev_err, E3_DEV_ERR_CAPACITY);
    s_row = row;
  }
  __syncthreads();
  const int N = (a.H + 2 * a.KVH) * a.hd;
  const size_t plane = static_cast<size_t>(a.M) * N;
  const float* pr = a.part + static_cast<size_t>(m) * N;
  auto col = [&](int c) {
    float v = 0.0f;
    for (int z = 0; z < a.splits; ++z) v += pr[z * plane + c];
    return v;
  };
  const int row = s_row;
  __nv_bfloat16* qrow = a.Q + (static_cast<size_t>(b) * a.R_slots + slot) * a.H * a.hd;
  for (int idx = threadIdx.x; idx < (a.H + a.KVH) * half; idx += blockDim.x) {
    const int head = idx / half, i = idx - head * half;
    const int c0 = head * a.hd + i;  // q heads first, then k heads (same layout)
    const float x0 = col(c0), x1 = col(c0 + half);
    const float r0 = x0 * cs[i] - x1 * sn[i], r1 = x0 * sn[i] + x1 * cs[i];
    if (head < a.H) {
      qrow[head * a.hd + i] = __float2bfloat16_rn(r0);
      qrow[head * a.hd + i + half] = __float2bfloat16_rn(r1);
    } else if (row >= 0) {
      __nv_bfloat16* kr = a.kc + (static_cast<size_t>(row) + static_cast<size_t>(head - a.H) * a.page_size) * a.hd;
      kr[i] = __float2bfloat16_rn(r0);
      kr[i + half] = __float2bfloat16_rn(r1);
    }
  }
  if (row >= 0)
    for (int idx = threadIdx.x; idx < a.KVH * a.hd; idx += blockDim.x) {
      const int kh = idx / a.hd, i = idx - kh * a.hd;
      a.vc[(static_cast<size_t>(row) + static_cast<size_t>(kh) * a.page_size) * a.hd + i] =
          __float2bfloat16_rn(col((a.H + a.KVH) * a.hd + idx));
    }
}

// The attention output rows of the frontier (slot rows of O) as GEMM operand rows.
__global__ void __launch_bounds__(kThreads) draft_gather_kernel(const __nv_bfloat16* O, const int32_t* row_slot, int F,
                                                                int R_slots, int width, __nv_bfloat16* out) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x, b = m / F;
  const uint4* src = reinterpret_cast<const uint4*>(O + (static_cast<size_t>(b) * R_slots + row_slot[m]) * width);
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(m) * width);
  for (int i = threadIdx.x; i < width / 8; i += blockDim.x) dst[i] = src[i];
}

// h[m][j] = silu(gate) * up, gate = columns [0, ffn), up = [ffn, 2 ffn) of the split-K sum.
__global__ void __launch_bounds__(kThreads) draft_swiglu_kernel(const float* part, int splits, int M, int ffn,
                                                                __nv_bfloat16* h) {
  pdl_wait();
  pdl_trigger();
  const size_t n = static_cast<size_t>(M) * ffn;
  const size_t plane = static_cast<size_t>(M) * 2 * ffn;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t m = i / ffn, j = i - m * ffn;
    float gt = 0.0f, up = 0.0f;
    for (int z = 0; z < splits; ++z) {
      gt += part[z * plane + m * 2 * ffn + j];
      up += part[z * plane + m * 2 * ffn + ffn + j];
    }
    h[i] = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
  }
}

// Workspace regions of one step (256-byte aligned), for M = B * F_max rows.
struct DraftWs {
  size_t e_rows, h_rows, x, y, o_rows, mlp, part, Q, O, lse, vws, row_slot, row_pos, ones, total;
  size_t vws_bytes;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

DraftWs draft_ws(const e3_drafter& w, int B, int F_max, int R_slots, int max_kv_len) {
  const int M = B * F_max;
  const int H = w.n_heads, KVH = w.n_kv_heads, hd = w.head_dim, d = w.d;
  // The largest split-K partial of any of the five GEMMs at any row count up to M.  Between
  // the row counts where the token tiling steps (16, 32, 64, 128, then multiples of 256)
  // the split count is fixed and the partial grows with the rows, so the step ends suffice.
  size_t part = 0;
  auto part_at = [&](int mm) {
    part = std::max(part, linear_partial_bytes(mm, 2 * d, d));
    part = std::max(part, linear_partial_bytes(mm, d, (H + 2 * KVH) * hd));
    part = std::max(part, linear_partial_bytes(mm, H * hd, d));
    part = std::max(part, linear_partial_bytes(mm, d, 2 * w.ffn));
    part = std::max(part, linear_partial_bytes(mm, w.ffn, d));
  };
  for (int mm : {16, 32, 64, 128}) part_at(std::min(mm, M));
  for (int mm = 256; mm < M + 256; mm += 256) part_at(std::min(mm, M));
  DraftWs r{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  r.e_rows = take(static_cast<size_t>(M) * d * 2);
  r.h_rows = take(static_cast<size_t>(M) * d * 2);
  r.x = take(static_cast<size_t>(M) * d * 4);
  r.y = take(static_cast<size_t>(M) * d * 2);
  r.o_rows = take(static_cast<size_t>(M) * H * hd * 2);
  r.mlp = take(static_cast<size_t>(M) * w.ffn * 2);
  r.part = take(part);
  r.Q = take(static_cast<size_t>(B) * R_slots * H * hd * 2);
  r.O = take(static_cast<size_t>(B) * R_slots * H * hd * 2);
  r.lse = take(static_cast<size_t>(B) * R_slots * H * 4);
  r.vws_bytes = verify_workspace_bytes(B, R_slots, H, KVH, hd, max_kv_len, verify_uses_mma(E3_BF16, hd));
  r.vws = take(r.vws_bytes);
  r.row_slot = take(static_cast<size_t>(M) * 4);
  r.row_pos = take(static_cast<size_t>(M) * 4);
  r.ones = take(static_cast<size_t>(M) * 4);
  r.total = o;
  return r;
}

e3_status check_drafter(const e3_drafter* w, const char* fn) {
  E3_REQUIRE(w != nullptr, E3_ERR_INVALID_ARG, "%s: null drafter", fn);
  E3_REQUIRE(w->emb && w->W_in && w->norm1 && w->W_qkv && w->W_o && w->norm2 && w->W_gu && w->W_down && w->norm_f &&
                 w->W_lm,
             E3_ERR_INVALID_ARG, "%s: null drafter weight", fn);
  E3_REQUIRE(w->d >= 128 && w->d % 128 == 0 && w->ffn >= 128 && w->ffn % 128 == 0 && w->V >= 1 && w->V % 4 == 0,
             E3_ERR_SHAPE, "%s: d=%d, ffn=%d must be multiples of 128, V=%d a multiple of 4", fn, w->d, w->ffn, w->V);
  E3_REQUIRE(w->n_heads >= 1 && w->n_kv_heads >= 1 && w->n_heads % w->n_kv_heads == 0, E3_ERR_SHAPE,
             "%s: heads %d / %d", fn, w->n_heads, w->n_kv_heads);
  E3_REQUIRE((w->head_dim == 64 || w->head_dim == 128) && (w->n_heads * w->head_dim) % 128 == 0, E3_ERR_SHAPE,
             "%s: head_dim %d must be 64 or 128 with H*hd a multiple of 128", fn, w->head_dim);
  E3_REQUIRE(w->rope_base > 1.0f && w->eps > 0.0f, E3_ERR_INVALID_ARG, "%s: rope_base > 1 and eps > 0", fn);
  return E3_OK;
}

}  // namespace

}  // namespace e3

using namespace e3;

extern "C" {

E3_API size_t eagle3_draft_workspace_bytes(const e3_drafter* drafter, int B, int F_max, int R_slots, int max_kv_len) {
  if (check_drafter(drafter, "eagle3_draft_workspace_bytes") != E3_OK) return 0;
  if (B < 1 || F_max < 1 || B * F_max > 1024 || R_slots < 1 || R_slots > E3_MAX_NODES + 1 || max_kv_len < 0) return 0;
  return draft_ws(*drafter, B, F_max, R_slots, max_kv_len).total;
}

E3_API e3_status eagle3_draft_step(const e3_drafter* drafter, const e3_kv_layer* kv, const int32_t* kv_len,
                                   int max_kv_len, int B, int depth, int F, const int32_t* frontier, int slot_base,
                                   int F_prev, const int32_t* frontier_prev, int slot_base_prev, int R_slots,
                                   const e3_cand* cands, const int32_t* root_tok, const void* g, float* a_slots,
                                   uint64_t* mask, float* logits, float* row_max, uint64_t* row_Q,
                                   int32_t* row_argmax, void* ws, size_t ws_bytes, int32_t* dev_err,
                                   e3_stream_t stream) {
  clear_error();
  const char* fn = "eagle3_draft_step";
  e3_status st = check_drafter(drafter, fn);
  if (st != E3_OK) return st;
  const e3_drafter& w = *drafter;
  E3_REQUIRE(kv && kv_len && frontier && cands && root_tok && g && a_slots && mask && logits && row_max && row_Q &&
                 row_argmax && ws,
             E3_ERR_INVALID_ARG, "%s: null pointer", fn);
  E3_REQUIRE(kv->k && kv->v && kv->page_table && kv->dt == E3_BF16 && kv->head_dim == w.head_dim &&
                 kv->n_kv_heads == w.n_kv_heads && kv->page_size > 0 && kv->max_pages > 0 && kv->n_pages > 0,
             E3_ERR_SHAPE, "%s: the drafter's cache must be bf16 with the drafter's head_dim and KV heads", fn);
  E3_REQUIRE((kv->flags & ~(E3_KV_PREFIX_STABLE | E3_KV_SELFTEST_STALL)) == 0, E3_ERR_INVALID_ARG,
             "%s: unknown kv flags", fn);
  E3_REQUIRE(B >= 1 && F >= 1 && B * F <= 1024, E3_ERR_SHAPE, "%s: B=%d F=%d", fn, B, F);
  E3_REQUIRE(depth >= 1 && depth <= E3_MAX_DEPTH, E3_ERR_SHAPE, "%s: depth %d", fn, depth);
  E3_REQUIRE(depth > 1 || (F == 1 && slot_base == 0), E3_ERR_SHAPE, "%s: depth 1 expands the root only (slot 0)", fn);
  E3_REQUIRE(depth == 1 || (frontier_prev && F_prev >= 1 && slot_base_prev >= 0 && slot_base_prev + F_prev <= slot_base),
             E3_ERR_SHAPE, "%s: previous frontier (F_prev=%d at slot %d) must precede slot %d", fn, F_prev,
             slot_base_prev, slot_base);
  E3_REQUIRE(R_slots >= 1 && R_slots <= E3_MAX_NODES + 1 && slot_base >= 0 && slot_base + F <= R_slots, E3_ERR_SHAPE,
             "%s: slots [%d, %d) outside R_slots=%d", fn, slot_base, slot_base + F, R_slots);
  E3_REQUIRE(cands->tok && cands->parent && cands->cap >= 1, E3_ERR_INVALID_ARG, "%s: bad candidate arrays", fn);
  E3_REQUIRE(max_kv_len >= 0 && static_cast<long>(max_kv_len) + R_slots <= static_cast<long>(kv->max_pages) * kv->page_size,
             E3_ERR_CAPACITY, "%s: max_kv_len + R_slots exceeds the drafter cache's pages", fn);
  const DraftWs L = draft_ws(w, B, F, R_slots, max_kv_len);
  E3_REQUIRE(ws_bytes >= L.total, E3_ERR_CAPACITY, "%s: workspace of %zu bytes needed, %zu given", fn, L.total,
             ws_bytes);
  E3_REQUIRE(aligned16(ws) && aligned16(g) && aligned16(w.emb) && aligned16(a_slots) && aligned16(logits), E3_ERR_INVALID_ARG,
             "%s: ws, g, emb, a_slots, logits must be 16-byte aligned", fn);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(ws);
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(base + off); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
  auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(base + off); };
  const int M = B * F, d = w.d, H = w.n_heads, KVH = w.n_kv_heads, hd = w.head_dim;
  const int words = (R_slots + 63) / 64;
  float* part = f32(L.part);
  int splits = 1;

  PrepArgs pa{F, depth, slot_base, F_prev, slot_base_prev, R_slots, words, d, w.V, cands->cap, frontier,
              frontier_prev, cands->tok, cands->parent, root_tok, kv_len,
              static_cast<const __nv_bfloat16*>(w.emb), static_cast<const __nv_bfloat16*>(g), a_slots, mask,
              bf(L.e_rows), bf(L.h_rows), i32(L.row_slot), i32(L.row_pos), f32(L.ones), dev_err};
  cudaError_t e = launch_pdl(draft_prep_kernel, dim3(M), dim3(kThreads), 0, s, 1, pa);
  if (e != cudaSuccess) return cuda_status(e, "draft_prep_kernel");

  auto norm = [&](const float* resid, const float* wn, float* slot_out) {
    NormArgs na{part, splits, M, d, resid, f32(L.x), wn, w.eps, bf(L.y), slot_out, i32(L.row_slot), F, R_slots};
    const cudaError_t e2 = launch_pdl(draft_norm_kernel, dim3(M), dim3(kThreads), static_cast<size_t>(d) * 4, s, 1, na);
    return e2 == cudaSuccess ? E3_OK : cuda_status(e2, "draft_norm_kernel");
  };
  // x = W_in [e(tok); h];  y = RMSNorm(x) norm1
  const void* in_src[2] = {bf(L.e_rows), bf(L.h_rows)};
  st = launch_linear_tc(w.W_in, in_src, 2, d, M, d, part, &splits, dev_err, s);
  if (st != E3_OK) return st;
  if ((st = norm(nullptr, w.norm1, nullptr)) != E3_OK) return st;
  // q, k, v with rotary positions; k, v into the cache at the rows' tree slots
  const void* y_src[1] = {bf(L.y)};
  st = launch_linear_tc(w.W_qkv, y_src, 1, d, M, (H + 2 * KVH) * hd, part, &splits, dev_err, s);
  if (st != E3_OK) return st;
  QkvArgs qa{part, splits, M, H, KVH, hd, w.rope_base, i32(L.row_slot), i32(L.row_pos), F, R_slots, bf(L.Q),
             static_cast<__nv_bfloat16*>(kv->k), static_cast<__nv_bfloat16*>(kv->v), kv->page_table, kv->max_pages,
             kv->n_pages, kv->page_size, kv_len, dev_err};
  e = launch_pdl(draft_qkv_kernel, dim3(M), dim3(kThreads), 0, s, 1, qa);
  if (e != cudaSuccess) return cuda_status(e, "draft_qkv_kernel");
  // attention over the drafter's cache: prefix + the tree slots on each row's mask
  st = launch_verify(bf(L.Q), *kv, kv_len, mask, B, R_slots, H, max_kv_len, 1.0f / sqrtf(static_cast<float>(hd)),
                     bf(L.O), f32(L.lse), dev_err, base + L.vws, L.vws_bytes, s);
  if (st != E3_OK) return st;
  e = launch_pdl(draft_gather_kernel, dim3(M), dim3(kThreads), 0, s, 1, static_cast<const __nv_bfloat16*>(bf(L.O)),
                 static_cast<const int32_t*>(i32(L.row_slot)), F, R_slots, H * hd, bf(L.o_rows));
  if (e != cudaSuccess) return cuda_status(e, "draft_gather_kernel");
  // x += W_o o;  y = RMSNorm(x) norm2
  const void* o_src[1] = {bf(L.o_rows)};
  st = launch_linear_tc(w.W_o, o_src, 1, H * hd, M, d, part, &splits, dev_err, s);
  if (st != E3_OK) return st;
  if ((st = norm(f32(L.x), w.norm2, nullptr)) != E3_OK) return st;
  // SwiGLU MLP
  st = launch_linear_tc(w.W_gu, y_src, 1, d, M, 2 * w.ffn, part, &splits, dev_err, s);
  if (st != E3_OK) return st;
  {
    const size_t n = static_cast<size_t>(M) * w.ffn;
    const int blocks = static_cast<int>(std::min<size_t>((n + kThreads - 1) / kThreads, 2048));
    e = launch_pdl(draft_swiglu_kernel, dim3(blocks), dim3(kThreads), 0, s, 1, static_cast<const float*>(part),
                   splits, M, w.ffn, bf(L.mlp));
    if (e != cudaSuccess) return cuda_status(e, "draft_swiglu_kernel");
  }
  // a = x + W_down h (kept per tree slot for the children's steps);  y = RMSNorm(a) norm_f
  const void* m_src[1] = {bf(L.mlp)};
  st = launch_linear_tc(w.W_down, m_src, 1, w.ffn, M, d, part, &splits, dev_err, s);
  if (st != E3_OK) return st;
  if ((st = norm(f32(L.x), w.norm_f, a_slots)) != E3_OK) return st;
  // draft logits and their statistics (temperature 1)
  return launch_lmhead_tc(bf(L.y), w.W_lm, M, d, w.V, f32(L.ones), logits, row_max, row_Q, row_argmax, dev_err, s);
}

}  // extern "C"
