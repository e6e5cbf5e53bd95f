// k_verify.cu -- tree_verify_attn: one tree-masked attention layer of the verify pass.
//
// "EAGLE 系列与 DFlash", §二 阶段三: the flattened tree goes through the target in
// ONE forward pass; 关键新增步骤②: node i attends to the KV prefix, its ancestors
// and itself only.  "EAGLE-3 投机解码与 USP 长序列训练优化", USP 核心设计：三步走:
// a heavy main segment and a light branch segment are computed apart and merged
// with a streaming softmax on their log-sum-exp; here the main segment is the
// KV prefix (split across CTAs) and the branch is the tree.
//
// Layout: the work of one KV head of one request is a set of key segments
//   s < n_pre : prefix keys [s*chunk, min((s+1)*chunk, P))
//   s = n_pre : the R tree slots P..P+R-1, masked per query row
// and a set of query rows r = i*G + g (node i, head h = kvh*G + g, G = H/KVH).
// Each CTA computes, for its segment and its rows, a partial (o, m, l) in the
// log2 domain into the workspace; a merge kernel combines the segments.
#include <math.h>

#include <atomic>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMmaRows = 128;  // query rows per CTA of the tensor-core kernel

struct VerifyGeom {
  int B, R, H, KVH, G, hd;
  int n_pre, S, chunk, RG;
  int max_kv_len;
  int fold;  // 1: S prefix segments, the last one also holding the tree slots
};

__device__ __forceinline__ bool kv_capacity_ok(const e3_kv_layer& kv, int P, int R, int max_kv_len) {
  const long need = static_cast<long>(P) + R;
  return P >= 0 && P <= max_kv_len && need <= static_cast<long>(kv.max_pages) * kv.page_size;
}

// Address of element 0 of logical token t (head kvh) of request b, or nullptr if
// its page id is out of range.
template <typename T>
__device__ __forceinline__ const T* kv_row(const T* base, const e3_kv_layer& kv, int b, int kvh, int t) {
  const int page = kv.page_table[static_cast<size_t>(b) * kv.max_pages + t / kv.page_size];
  if (page < 0 || page >= kv.n_pages) return nullptr;
  const size_t off = ((static_cast<size_t>(page) * kv.n_kv_heads + kvh) * kv.page_size + t % kv.page_size) *
                     static_cast<size_t>(kv.head_dim);
  return base + off;
}

// ---------------------------------------------------------------------------
// SIMT kernel (fp32 and generic head dims): one warp per query row.
// ---------------------------------------------------------------------------
template <typename T, int HD>
__global__ void __launch_bounds__(256)
verify_simt_kernel(const T* __restrict__ Q, e3_kv_layer kv, const int32_t* __restrict__ kv_len,
                   const uint64_t* __restrict__ mask, VerifyGeom g, float sm_scale,
                   float* __restrict__ ws_o, float2* __restrict__ ws_ml, int32_t* dev_err) {
  constexpr int PER = HD / 32;
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int P = kv_len[b];
  if (!kv_capacity_ok(kv, P, g.R, g.max_kv_len)) {
    if (threadIdx.x == 0 && s == 0 && kvh == 0) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
    return;
  }
  const T* Kb = static_cast<const T*>(kv.k);
  const T* Vb = static_cast<const T*>(kv.v);
  const bool tree = (s == g.n_pre);
  int k0 = 0, k1 = 0;
  if (tree) {
    k0 = 0;
    k1 = g.R;
  } else {
    k0 = s * g.chunk;
    k1 = min(P, k0 + g.chunk);
  }
  const int words = (g.R + 63) >> 6;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const float c2 = sm_scale * kLog2e;
  for (int r = warp; r < g.G * g.R; r += nwarp) {
    const int i = r / g.G, h = kvh * g.G + r % g.G;
    const T* q = Q + ((static_cast<size_t>(b) * g.R + i) * g.H + h) * HD;
    float qv[PER], acc[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      qv[u] = ld_elem(q, lane + 32 * u);
      acc[u] = 0.0f;
    }
    float m = -INFINITY, l = 0.0f;
    const uint64_t* mrow = mask + (static_cast<size_t>(b) * g.R + i) * words;
    // keys in groups of kGrp: the group's K and V rows are loaded before any of its
    // dot products is reduced, so that the loads overlap; the online-softmax updates
    // then run in key order
    constexpr int kGrp = 8;
    for (int kb = k0; kb < k1; kb += kGrp) {
      float kvals[kGrp][PER], vvals[kGrp][PER];
      bool use[kGrp];
#pragma unroll
      for (int j = 0; j < kGrp; ++j) {
        const int kk = kb + j;
        use[j] = kk < k1;
        int t = kk;
        if (use[j] && tree) {
          use[j] = (mrow[kk >> 6] >> (kk & 63)) & 1ull;
          t = P + kk;
        }
        const T* kr = use[j] ? kv_row(Kb, kv, b, kvh, t) : nullptr;
        const T* vr = use[j] ? kv_row(Vb, kv, b, kvh, t) : nullptr;
        if (use[j] && (!kr || !vr)) {
          if (lane == 0) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
          use[j] = false;
        }
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          kvals[j][u] = use[j] ? ld_elem(kr, lane + 32 * u) : 0.0f;
          vvals[j][u] = use[j] ? ld_elem(vr, lane + 32 * u) : 0.0f;
        }
      }
      float d[kGrp];
#pragma unroll
      for (int j = 0; j < kGrp; ++j) {
        d[j] = 0.0f;
#pragma unroll
        for (int u = 0; u < PER; ++u) d[j] = fmaf(qv[u], kvals[j][u], d[j]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < kGrp; ++j) d[j] += __shfl_xor_sync(0xFFFFFFFFu, d[j], o);
#pragma unroll
      for (int j = 0; j < kGrp; ++j) {
        if (!use[j]) continue;
        const float sc = d[j] * c2;
        const float mn = fmaxf(m, sc);
        const float corr = exp2f(m - mn);  // m = -inf -> 0
        const float p = exp2f(sc - mn);
        l = l * corr + p;
#pragma unroll
        for (int u = 0; u < PER; ++u) acc[u] = fmaf(p, vvals[j][u], acc[u] * corr);
        m = mn;
      }
    }
    const size_t rec = ((static_cast<size_t>(b) * g.S + s) * g.R + i) * g.H + h;
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
    for (int u = 0; u < PER; ++u) ws_o[rec * HD + lane + 32 * u] = acc[u] * inv;
    if (lane == 0) ws_ml[rec] = make_float2(m, l);
  }
}

// ---------------------------------------------------------------------------
// Tensor-core kernel (bf16): mma.sync m16n8k16, one 16-row tile per warp,
// 32-key blocks double-buffered in shared memory with cp.async, online softmax
// in registers (FlashAttention-2 register layout).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int HD>
struct MmaCfg {
  static constexpr int KB = 32;               // keys per block
  static constexpr int PITCH = HD + 8;        // bf16 elements per smem row (16-byte skew)
  static constexpr int TILE = KB * PITCH;     // elements per K or V block
  static constexpr int SMEM = 2 * 2 * TILE * 2;  // 2 stages x (K, V) x bytes
};

template <int HD>
__global__ void __launch_bounds__(256)
verify_mma_kernel(const __nv_bfloat16* __restrict__ Q, e3_kv_layer kv, const int32_t* __restrict__ kv_len,
                  const uint64_t* __restrict__ mask, VerifyGeom g, float sm_scale, float* __restrict__ ws_o,
                  float2* __restrict__ ws_ml, int32_t* dev_err) {
  using C = MmaCfg<HD>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [2][KB][PITCH]
  __nv_bfloat16* sV = sK + 2 * C::TILE;                            // [2][KB][PITCH]

  const int rg = blockIdx.x % g.RG, s = blockIdx.x / g.RG;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int P = kv_len[b];
  if (!kv_capacity_ok(kv, P, g.R, g.max_kv_len)) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
    return;
  }
  const bool tree = (s == g.n_pre);
  const int k0 = tree ? 0 : s * g.chunk;
  const int k1 = tree ? g.R : min(P, k0 + g.chunk);
  const int nkeys = max(0, k1 - k0);
  const int nblk = (nkeys + C::KB - 1) / C::KB;
  const __nv_bfloat16* Kb = static_cast<const __nv_bfloat16*>(kv.k);
  const __nv_bfloat16* Vb = static_cast<const __nv_bfloat16*>(kv.v);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  const int rows = g.G * g.R;
  const int tile0 = rg * kMmaRows + warp * 16;
  const bool warp_active = tile0 < rows;

  // ---- issue loads of one key block -------------------------------------
  auto load_block = [&](int blk, int stage) {
    constexpr int CH = HD / 8;  // 16-byte chunks per row
    for (int idx = threadIdx.x; idx < C::KB * CH * 2; idx += blockDim.x) {
      const int which = idx / (C::KB * CH);  // 0 = K, 1 = V
      const int rem = idx % (C::KB * CH);
      const int key = rem / CH, ch = rem % CH;
      const int kk = k0 + blk * C::KB + key;
      const __nv_bfloat16* base = which ? Vb : Kb;
      const __nv_bfloat16* src = base;
      int bytes = 0;
      if (kk < k1) {
        const int t = tree ? P + kk : kk;
        const __nv_bfloat16* row = kv_row(base, kv, b, kvh, t);
        if (row) {
          src = row + ch * 8;
          bytes = 16;
        } else {
          dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
        }
      }
      __nv_bfloat16* dst = (which ? sV : sK) + stage * C::TILE + key * C::PITCH + ch * 8;
      cp_async16(smem_u32(dst), src, bytes);
    }
    cp_async_commit();
  };

  // ---- Q fragments of this warp's 16 rows ---------------------------------
  uint32_t qa[HD / 16][4];
  int rowi[2] = {0, 0};
  bool rowv[2] = {false, false};
#pragma unroll
  for (int hrow = 0; hrow < 2; ++hrow) {
    const int r = tile0 + gq + hrow * 8;
    rowv[hrow] = warp_active && r < rows;
    rowi[hrow] = rowv[hrow] ? r / g.G : 0;
  }
  {
    const __nv_bfloat16* qp[2];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int r = tile0 + gq + hrow * 8;
      const int h = kvh * g.G + (rowv[hrow] ? r % g.G : 0);
      qp[hrow] = Q + ((static_cast<size_t>(b) * g.R + rowi[hrow]) * g.H + h) * HD;
    }
#pragma unroll
    for (int kc = 0; kc < HD / 16; ++kc) {
      const int c0 = kc * 16 + 2 * tq;
      qa[kc][0] = rowv[0] ? *reinterpret_cast<const uint32_t*>(qp[0] + c0) : 0u;
      qa[kc][1] = rowv[1] ? *reinterpret_cast<const uint32_t*>(qp[1] + c0) : 0u;
      qa[kc][2] = rowv[0] ? *reinterpret_cast<const uint32_t*>(qp[0] + c0 + 8) : 0u;
      qa[kc][3] = rowv[1] ? *reinterpret_cast<const uint32_t*>(qp[1] + c0 + 8) : 0u;
    }
  }
  const int words = (g.R + 63) >> 6;
  const uint64_t* mrow0 = mask + (static_cast<size_t>(b) * g.R + rowi[0]) * words;
  const uint64_t* mrow1 = mask + (static_cast<size_t>(b) * g.R + rowi[1]) * words;

  float o[HD / 8][4];
#pragma unroll
  for (int dt = 0; dt < HD / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  const float c2 = sm_scale * kLog2e;

  if (nblk > 0) load_block(0, 0);
  for (int blk = 0; blk < nblk; ++blk) {
    const int stage = blk & 1;
    if (blk + 1 < nblk) {
      load_block(blk + 1, stage ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (warp_active) {
      const __nv_bfloat16* k_s = sK + stage * C::TILE;
      const __nv_bfloat16* v_s = sV + stage * C::TILE;
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
      // S = Q K^T for 32 keys: pairs of n8 tiles
#pragma unroll
      for (int np2 = 0; np2 < 2; ++np2) {
#pragma unroll
        for (int kc = 0; kc < HD / 16; ++kc) {
          const int mi = lane >> 3;
          const int key = np2 * 16 + (mi >> 1) * 8 + (lane & 7);
          const int col = kc * 16 + (mi & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(k_s + key * C::PITCH + col), b0, b1, b2, b3);
          mma_bf16(sc[2 * np2], qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b0, b1);
          mma_bf16(sc[2 * np2 + 1], qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b2, b3);
        }
      }
      // scale, mask, running max
      const int kbase = blk * C::KB;  // key offset inside the segment
      uint64_t w0 = 0, w1 = 0;
      if (tree) {
        w0 = mrow0[(k0 + kbase) >> 6];
        w1 = mrow1[(k0 + kbase) >> 6];
      }
      float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = k0 + kbase + nt * 8 + 2 * tq + e;
          bool ok0 = kk < k1, ok1 = kk < k1;
          if (tree) {
            ok0 = ok0 && ((w0 >> (kk & 63)) & 1ull);
            ok1 = ok1 && ((w1 >> (kk & 63)) & 1ull);
          }
          sc[nt][e] = ok0 ? sc[nt][e] * c2 : -INFINITY;
          sc[nt][2 + e] = ok1 ? sc[nt][2 + e] * c2 : -INFINITY;
          bm0 = fmaxf(bm0, sc[nt][e]);
          bm1 = fmaxf(bm1, sc[nt][2 + e]);
        }
      }
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xFFFFFFFFu, bm0, 1));
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xFFFFFFFFu, bm0, 2));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xFFFFFFFFu, bm1, 1));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xFFFFFFFFu, bm1, 2));
      const float nm0 = fmaxf(m0, bm0), nm1 = fmaxf(m1, bm1);
      const float corr0 = (nm0 == -INFINITY) ? 1.0f : exp2f(m0 - nm0);
      const float corr1 = (nm1 == -INFINITY) ? 1.0f : exp2f(m1 - nm1);
      const float sub0 = (nm0 == -INFINITY) ? 0.0f : nm0;
      const float sub1 = (nm1 == -INFINITY) ? 0.0f : nm1;
      m0 = nm0;
      m1 = nm1;
      float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - sub0);
        sc[nt][1] = exp2f(sc[nt][1] - sub0);
        sc[nt][2] = exp2f(sc[nt][2] - sub1);
        sc[nt][3] = exp2f(sc[nt][3] - sub1);
        rs0 += sc[nt][0] + sc[nt][1];
        rs1 += sc[nt][2] + sc[nt][3];
      }
      l0 = l0 * corr0 + rs0;
      l1 = l1 * corr1 + rs1;
#pragma unroll
      for (int dt = 0; dt < HD / 8; ++dt) {
        o[dt][0] *= corr0;
        o[dt][1] *= corr0;
        o[dt][2] *= corr1;
        o[dt][3] *= corr1;
      }
      // O += P V
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        const uint32_t a0 = pack_bf16(sc[2 * pc][0], sc[2 * pc][1]);
        const uint32_t a1 = pack_bf16(sc[2 * pc][2], sc[2 * pc][3]);
        const uint32_t a2 = pack_bf16(sc[2 * pc + 1][0], sc[2 * pc + 1][1]);
        const uint32_t a3 = pack_bf16(sc[2 * pc + 1][2], sc[2 * pc + 1][3]);
#pragma unroll
        for (int dt = 0; dt < HD / 8; dt += 2) {
          const int mi = lane >> 3;
          const int key = pc * 16 + (mi & 1) * 8 + (lane & 7);
          const int col = (dt + (mi >> 1)) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(v_s + key * C::PITCH + col), b0, b1, b2, b3);
          mma_bf16(o[dt], a0, a1, a2, a3, b0, b1);
          mma_bf16(o[dt + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  if (!warp_active) return;
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
#pragma unroll
  for (int hrow = 0; hrow < 2; ++hrow) {
    if (!rowv[hrow]) continue;
    const int r = tile0 + gq + hrow * 8;
    const int i = r / g.G, h = kvh * g.G + r % g.G;
    const size_t rec = ((static_cast<size_t>(b) * g.S + s) * g.R + i) * g.H + h;
    const float l = hrow ? l1 : l0;
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    float* dst = ws_o + rec * HD;
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
      float2 v = make_float2(o[dt][2 * hrow] * inv, o[dt][2 * hrow + 1] * inv);
      *reinterpret_cast<float2*>(dst + dt * 8 + 2 * tq) = v;
    }
    if (tq == 0) ws_ml[rec] = make_float2(hrow ? m1 : m0, l);
  }
}

// ---------------------------------------------------------------------------
// Merge of the segments: one warp per (b, i, h) row.  Lanes load the segments'
// (m, l) in parallel; each lane owns HD/32 consecutive output dims and adds the
// weighted partial vectors with independent loads.
// ---------------------------------------------------------------------------
template <typename T, int HD>
__global__ void __launch_bounds__(256)
verify_merge_kernel(e3_kv_layer kv, const int32_t* __restrict__ kv_len, VerifyGeom g,
                    const float* __restrict__ ws_o, const float2* __restrict__ ws_ml, T* __restrict__ O,
                    float* __restrict__ lse) {
  constexpr int PER = HD / 32;
  pdl_wait();  // the segment kernel's partial records are complete
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long row = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long nrows = static_cast<long>(g.B) * g.R * g.H;
  if (row >= nrows) return;
  const int b = static_cast<int>(row / (static_cast<long>(g.R) * g.H));
  const int ih = static_cast<int>(row % (static_cast<long>(g.R) * g.H));
  const int P = kv_len[b];
  if (!kv_capacity_ok(kv, P, g.R, g.max_kv_len)) return;
  // segments that hold keys: the prefix segments up to P and the tree segment, or
  // (tree folded into the last prefix segment) every segment
  const int n_pre_b = g.fold ? g.S : (P + g.chunk - 1) / g.chunk;
  const int nseg = g.fold ? g.S : n_pre_b + 1;
  const size_t stride = static_cast<size_t>(g.R) * g.H;
  const size_t base = static_cast<size_t>(b) * g.S * stride + ih;
  auto seg_id = [&](int q) { return q < n_pre_b ? q : g.n_pre; };
  float M = -INFINITY;
  for (int q0 = 0; q0 < nseg; q0 += 32) {
    const int q = q0 + lane;
    if (q < nseg) {
      const float2 ml = ws_ml[base + seg_id(q) * stride];
      if (ml.y > 0.0f) M = fmaxf(M, ml.x);
    }
  }
  M = warp_reduce(M, MaxF());
  float acc[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) acc[u] = 0.0f;
  float den = 0.0f;
  for (int q0 = 0; q0 < nseg; q0 += 32) {
    const int q = q0 + lane;
    float w = 0.0f;
    if (q < nseg) {
      const float2 ml = ws_ml[base + seg_id(q) * stride];
      w = ml.y > 0.0f ? ml.y * exp2f(ml.x - M) : 0.0f;
    }
    den += w;
    const int nq = min(32, nseg - q0);
#pragma unroll 4
    for (int j = 0; j < nq; ++j) {
      const float wj = __shfl_sync(0xFFFFFFFFu, w, j);
      const float* src = ws_o + (base + seg_id(q0 + j) * stride) * HD + lane * PER;
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[u] = fmaf(wj, src[u], acc[u]);
    }
  }
  den = warp_reduce(den, [](float a, float c) { return a + c; });
  const float inv = den > 0.0f ? 1.0f / den : 0.0f;
  T* out = O + static_cast<size_t>(row) * HD + lane * PER;
#pragma unroll
  for (int u = 0; u < PER; ++u) st_elem(out, u, acc[u] * inv);
  if (lane == 0) lse[row] = (M + log2f(den)) * kLn2;
}

int num_sms() {
  static const int n_once = [] {  // queried once, thread-safely (152 on GB300 if the query fails)
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    return n;
  }();
  return n_once;
}

VerifyGeom make_geom(int B, int R, int H, int KVH, int hd, int max_kv_len, bool mma) {
  VerifyGeom g{};
  g.B = B;
  g.R = R;
  g.H = H;
  g.KVH = KVH;
  g.G = H / KVH;
  g.hd = hd;
  g.max_kv_len = max_kv_len;
  g.RG = mma ? (g.G * R + kMmaRows - 1) / kMmaRows : 1;
  const long natural = static_cast<long>(B) * KVH * g.RG;
  const long target = 2L * num_sms();
  long splits = (target + natural - 1) / natural;
  if (splits < 1) splits = 1;
  long chunk = (max_kv_len + splits - 1) / splits;
  chunk = ((chunk + 63) / 64) * 64;
  if (chunk < 64) chunk = 64;
  if (mma && chunk < 256) chunk = 256;  // two 128-key tiles per tensor-core CTA at least
  if (mma) {                            // at most 15 prefix segments (+ tree) per cluster
    const long cap = ((static_cast<long>(max_kv_len) + 14) / 15 + 127) / 128 * 128;
    if (chunk < cap) chunk = cap;
  }
  g.chunk = static_cast<int>(chunk);
  g.n_pre = static_cast<int>((max_kv_len + chunk - 1) / chunk);
  g.S = g.n_pre + 1;
  return g;
}

}  // namespace

size_t verify_workspace_bytes(int B, int R, int H, int KVH, int hd, int max_kv_len, bool mma) {
  VerifyGeom g = make_geom(B, R, H, KVH, hd, max_kv_len, mma);
  const size_t recs = static_cast<size_t>(B) * g.S * R * H;
  return recs * hd * sizeof(float) + recs * sizeof(float2) + 256;
}

bool verify_uses_mma(e3_dtype dt, int hd) { return dt == E3_BF16 && (hd == 64 || hd == 128); }

e3_status launch_verify(const void* Q, const e3_kv_layer& kv, const int32_t* kv_len, const uint64_t* mask,
                        int B, int R, int H, int max_kv_len, float sm_scale, void* O, float* lse,
                        int32_t* dev_err, void* ws, size_t ws_bytes, cudaStream_t s) {
  const int hd = kv.head_dim;
  const bool mma = verify_uses_mma(kv.dt, hd);
  VerifyGeom g = make_geom(B, R, H, kv.n_kv_heads, hd, max_kv_len, mma);
  const size_t need = verify_workspace_bytes(B, R, H, kv.n_kv_heads, hd, max_kv_len, mma);
  E3_REQUIRE(ws != nullptr && ws_bytes >= need, E3_ERR_CAPACITY,
             "tree_verify_attn: workspace of %zu bytes needed, %zu given", need, ws_bytes);
  const size_t recs = static_cast<size_t>(B) * g.S * R * H;
  float* ws_o = static_cast<float*>(ws);
  uintptr_t ml_addr = reinterpret_cast<uintptr_t>(ws_o + recs * hd);
  ml_addr = (ml_addr + 15) & ~static_cast<uintptr_t>(15);
  float2* ws_ml = reinterpret_cast<float2*>(ml_addr);

  if (mma && verify_tc_supported(kv, H)) {
    bool merged = false;
    VerifySplit sp{g.n_pre, g.S, g.chunk, 0};
    e3_status st = launch_verify_tc(Q, kv, kv_len, mask, B, R, H, max_kv_len, sm_scale, &sp, ws_o, ws_ml, O, lse,
                                    &merged, dev_err, s);
    if (st != E3_OK) return st;
    if (merged) return E3_OK;  // segments merged inside the cluster
    g.n_pre = sp.n_pre;
    g.S = sp.S;
    g.chunk = sp.chunk;
    g.fold = sp.fold;
  } else if (mma) {
    dim3 grid(g.RG * g.S, kv.n_kv_heads, B);
#define E3_MMA_CASE(HDV)                                                                           \
  do {                                                                                             \
    const int smem = MmaCfg<HDV>::SMEM;                                                            \
    static std::atomic<bool> attr_done{false};                                                     \
    if (!attr_done.load(std::memory_order_acquire)) {                                              \
      cudaFuncSetAttribute(verify_mma_kernel<HDV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); \
      attr_done.store(true, std::memory_order_release);                                            \
    }                                                                                              \
    verify_mma_kernel<HDV><<<grid, 256, smem, s>>>(static_cast<const __nv_bfloat16*>(Q), kv, kv_len, \
                                                   mask, g, sm_scale, ws_o, ws_ml, dev_err);       \
  } while (0)
    if (hd == 128)
      E3_MMA_CASE(128);
    else
      E3_MMA_CASE(64);
#undef E3_MMA_CASE
    E3_LAUNCH_CHECK("tree_verify_attn segment kernel");
  } else {
    dim3 grid(g.S, kv.n_kv_heads, B);
#define E3_SIMT_CASE(TT, HDV)                                                                  \
  verify_simt_kernel<TT, HDV><<<grid, 256, 0, s>>>(static_cast<const TT*>(Q), kv, kv_len, mask, g, \
                                                   sm_scale, ws_o, ws_ml, dev_err)
    if (kv.dt == E3_F32) {
      switch (hd) {
        case 32: E3_SIMT_CASE(float, 32); break;
        case 64: E3_SIMT_CASE(float, 64); break;
        case 96: E3_SIMT_CASE(float, 96); break;
        case 128: E3_SIMT_CASE(float, 128); break;
        case 160: E3_SIMT_CASE(float, 160); break;
        case 192: E3_SIMT_CASE(float, 192); break;
        case 224: E3_SIMT_CASE(float, 224); break;
        default: E3_SIMT_CASE(float, 256); break;
      }
    } else {
      switch (hd) {
        case 32: E3_SIMT_CASE(__nv_bfloat16, 32); break;
        case 96: E3_SIMT_CASE(__nv_bfloat16, 96); break;
        case 160: E3_SIMT_CASE(__nv_bfloat16, 160); break;
        case 192: E3_SIMT_CASE(__nv_bfloat16, 192); break;
        case 224: E3_SIMT_CASE(__nv_bfloat16, 224); break;
        default: E3_SIMT_CASE(__nv_bfloat16, 256); break;
      }
    }
#undef E3_SIMT_CASE
    E3_LAUNCH_CHECK("tree_verify_attn segment kernel");
  }
  const long nrows = static_cast<long>(B) * R * H;
  const int blocks = static_cast<int>((nrows + 7) / 8);
  cudaError_t me = cudaSuccess;
#define E3_MERGE_CASE(TT, HDV)                                                                               \
  me = launch_pdl(verify_merge_kernel<TT, HDV>, dim3(blocks), dim3(256), 0, s, 1, kv, kv_len, g,                    \
                  static_cast<const float*>(ws_o), static_cast<const float2*>(ws_ml), static_cast<TT*>(O), lse)
  if (kv.dt == E3_F32) {
    switch (hd) {
      case 32: E3_MERGE_CASE(float, 32); break;
      case 64: E3_MERGE_CASE(float, 64); break;
      case 96: E3_MERGE_CASE(float, 96); break;
      case 128: E3_MERGE_CASE(float, 128); break;
      case 160: E3_MERGE_CASE(float, 160); break;
      case 192: E3_MERGE_CASE(float, 192); break;
      case 224: E3_MERGE_CASE(float, 224); break;
      default: E3_MERGE_CASE(float, 256); break;
    }
  } else {
    switch (hd) {
      case 32: E3_MERGE_CASE(__nv_bfloat16, 32); break;
      case 64: E3_MERGE_CASE(__nv_bfloat16, 64); break;
      case 96: E3_MERGE_CASE(__nv_bfloat16, 96); break;
      case 128: E3_MERGE_CASE(__nv_bfloat16, 128); break;
      case 160: E3_MERGE_CASE(__nv_bfloat16, 160); break;
      case 192: E3_MERGE_CASE(__nv_bfloat16, 192); break;
      case 224: E3_MERGE_CASE(__nv_bfloat16, 224); break;
      default: E3_MERGE_CASE(__nv_bfloat16, 256); break;
    }
  }
#undef E3_MERGE_CASE
  if (me != cudaSuccess) return cuda_status(me, "tree_verify_attn merge kernel");
  return E3_OK;
}

}  // namespace e3
