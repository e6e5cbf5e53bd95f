// k_gemm.cu -- SIMT GEMM for eagle3_fuse / lmhead_logits (fp32 inputs and the
// general case) and the per-row softmax statistics of lmhead_logits.
//
// Fusion ("SpecForge…", 多层特征融合到底融合了什么): g = W_f [h_low; h_mid; h_high];
// the concatenation is never materialised -- the K loop switches source
// pointer at d and 2d.
// LM head ("SpecForge…", 先看 checkpoint 最终要参与什么计算): the target computes
// the true distribution of every tree node.
#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

// Few rows (M <= kSkinnyRows): one warp per output column n, the lanes striding
// over k (coalesced rows of W and of A), one accumulator per row, then a warp
// reduction.  Same definition as gemm_simt_kernel below.
constexpr int kSkinnyRows = 16;
template <typename T, typename TO>
__global__ void __launch_bounds__(256)
gemm_skinny_kernel(const T* __restrict__ a0, const T* __restrict__ a1, const T* __restrict__ a2, int dseg,
                   const T* __restrict__ W, const float* __restrict__ bias, TO* __restrict__ out, int M, int N,
                   int K) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (n >= N) return;
  float acc[kSkinnyRows];
#pragma unroll
  for (int m = 0; m < kSkinnyRows; ++m) acc[m] = 0.0f;
  const T* wrow = W + static_cast<size_t>(n) * K;
  for (int seg = 0; seg * dseg < K; ++seg) {
    const T* src = seg == 0 ? a0 : (seg == 1 ? a1 : a2);
    const int klen = min(dseg, K - seg * dseg);
    for (int kin = lane; kin < klen; kin += 32) {
      const float w = ld_elem(wrow, static_cast<size_t>(seg) * dseg + kin);
#pragma unroll
      for (int m = 0; m < kSkinnyRows; ++m)
        if (m < M) acc[m] = fmaf(ld_elem(src, static_cast<size_t>(m) * dseg + kin), w, acc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < kSkinnyRows; ++m) {
    float v = acc[m];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0 && m < M) {
      if (bias) v += bias[n];
      st_elem(out, static_cast<size_t>(m) * N + n, v);
    }
  }
}

// out[m][n] = sum_k A(m, k) * W[n][k]  (+ bias[n]); A(m, k) reads segment k / dseg.
template <typename T, typename TO>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const T* __restrict__ a0, const T* __restrict__ a1, const T* __restrict__ a2, int dseg,
                 const T* __restrict__ W, const float* __restrict__ bias, TO* __restrict__ out, int M, int N,
                 int K) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Ws[BK][BN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int idx = threadIdx.x; idx < BM * BK; idx += 256) {
      const int mm = idx / BK, kk = idx % BK;
      const int m = m0 + mm, k = k0 + kk;
      float v = 0.0f;
      if (m < M && k < K) {
        const int sgi = k / dseg, kin = k % dseg;
        const T* src = sgi == 0 ? a0 : (sgi == 1 ? a1 : a2);
        v = ld_elem(src, static_cast<size_t>(m) * dseg + kin);
      }
      As[kk][mm] = v;
    }
    for (int idx = threadIdx.x; idx < BN * BK; idx += 256) {
      const int nn = idx / BK, kk = idx % BK;
      const int n = n0 + nn, k = k0 + kk;
      Ws[kk][nn] = (n < N && k < K) ? ld_elem(W, static_cast<size_t>(n) * K + k) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        av[u] = As[kk][ty * 4 + u];
        wv[u] = Ws[kk][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], wv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + ty * 4 + u;
    if (m >= M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int n = n0 + tx * 4 + v;
      if (n >= N) continue;
      float r = acc[u][v];
      if (bias) r += bias[n];
      st_elem(out, static_cast<size_t>(m) * N + n, r);
    }
  }
}

// Softmax statistics of one logit row per CTA (see lmhead_logits in eagle3.h).
__global__ void __launch_bounds__(1024)
row_stats_kernel(const float* __restrict__ logits, int V, const float* __restrict__ temp,
                 float* __restrict__ row_max, uint64_t* __restrict__ row_Q, int32_t* __restrict__ row_argmax,
                 int32_t* dev_err) {
  __shared__ uint64_t red64[32];
  __shared__ int redi[32];
  const int m = blockIdx.x;
  const float* z = logits + static_cast<size_t>(m) * V;
  const float it = inv_temp(temp[m]);
  uint64_t best = 0ull;
  int bad = 0;
  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    for (int q = threadIdx.x; q < (V >> 2); q += blockDim.x) {
      float4 v = z4[q];
      float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        bad |= !isfinite(e[u]);
        uint64_t key = pack_best(__fmul_rn(e[u], it), static_cast<uint32_t>(4 * q + u));
        best = key > best ? key : best;
      }
    }
  } else {
    for (int j = threadIdx.x; j < V; j += blockDim.x) {
      const float v = z[j];
      bad |= !isfinite(v);
      uint64_t key = pack_best(__fmul_rn(v, it), static_cast<uint32_t>(j));
      best = key > best ? key : best;
    }
  }
  bad = block_reduce(bad, OrI(), redi);
  best = block_reduce(best, MaxU64(), red64);
  if (bad) {
    if (threadIdx.x == 0) {
      dev_flag(dev_err, E3_DEV_ERR_NONFINITE);
      row_max[m] = __int_as_float(0x7FC00000);
      row_Q[m] = 0ull;
      row_argmax[m] = -1;
    }
    return;
  }
  const float mx = unord_f32(static_cast<uint32_t>(best >> 32));
  uint64_t Q = 0;
  if (vec) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    for (int q = threadIdx.x; q < (V >> 2); q += blockDim.x) {
      float4 v = z4[q];
      Q += fx_mass(__fmul_rn(v.x, it), mx) + fx_mass(__fmul_rn(v.y, it), mx) +
           fx_mass(__fmul_rn(v.z, it), mx) + fx_mass(__fmul_rn(v.w, it), mx);
    }
  } else {
    for (int j = threadIdx.x; j < V; j += blockDim.x) Q += fx_mass(__fmul_rn(z[j], it), mx);
  }
  Q = block_reduce(Q, SumU64(), red64);
  if (threadIdx.x == 0) {
    row_max[m] = mx;
    row_Q[m] = Q;
    row_argmax[m] = static_cast<int32_t>(packed_id(best));
  }
}

}  // namespace

e3_status launch_gemm_simt(const void* a0, const void* a1, const void* a2, int dseg, const void* W,
                           const float* bias, void* out, bool out_f32, int M, int N, int K, e3_dtype dt,
                           cudaStream_t s) {
  if (M <= kSkinnyRows) {
    const dim3 sg((N + 7) / 8);
    if (dt == E3_F32) {
      if (!out_f32) return E3_ERR_UNSUPPORTED;
      gemm_skinny_kernel<float, float><<<sg, 256, 0, s>>>(
          static_cast<const float*>(a0), static_cast<const float*>(a1), static_cast<const float*>(a2), dseg,
          static_cast<const float*>(W), bias, static_cast<float*>(out), M, N, K);
    } else {
      using B16 = __nv_bfloat16;
      if (out_f32)
        gemm_skinny_kernel<B16, float><<<sg, 256, 0, s>>>(
            static_cast<const B16*>(a0), static_cast<const B16*>(a1), static_cast<const B16*>(a2), dseg,
            static_cast<const B16*>(W), bias, static_cast<float*>(out), M, N, K);
      else
        gemm_skinny_kernel<B16, B16><<<sg, 256, 0, s>>>(
            static_cast<const B16*>(a0), static_cast<const B16*>(a1), static_cast<const B16*>(a2), dseg,
            static_cast<const B16*>(W), bias, static_cast<B16*>(out), M, N, K);
    }
    E3_LAUNCH_CHECK("gemm_skinny_kernel");
    return E3_OK;
  }
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  if (dt == E3_F32) {
    if (out_f32)
      gemm_simt_kernel<float, float><<<grid, 256, 0, s>>>(
          static_cast<const float*>(a0), static_cast<const float*>(a1), static_cast<const float*>(a2), dseg,
          static_cast<const float*>(W), bias, static_cast<float*>(out), M, N, K);
    else
      return E3_ERR_UNSUPPORTED;
  } else {
    using B16 = __nv_bfloat16;
    if (out_f32)
      gemm_simt_kernel<B16, float><<<grid, 256, 0, s>>>(
          static_cast<const B16*>(a0), static_cast<const B16*>(a1), static_cast<const B16*>(a2), dseg,
          static_cast<const B16*>(W), bias, static_cast<float*>(out), M, N, K);
    else
      gemm_simt_kernel<B16, B16><<<grid, 256, 0, s>>>(
          static_cast<const B16*>(a0), static_cast<const B16*>(a1), static_cast<const B16*>(a2), dseg,
          static_cast<const B16*>(W), bias, static_cast<B16*>(out), M, N, K);
  }
  E3_LAUNCH_CHECK("gemm_simt_kernel");
  return E3_OK;
}

e3_status launch_row_stats(const float* logits, int M, int V, const float* temp, float* row_max,
                           uint64_t* row_Q, int32_t* row_argmax, int32_t* dev_err, cudaStream_t s) {
  row_stats_kernel<<<M, 1024, 0, s>>>(logits, V, temp, row_max, row_Q, row_argmax, dev_err);
  E3_LAUNCH_CHECK("row_stats_kernel");
  return E3_OK;
}

}  // namespace e3
