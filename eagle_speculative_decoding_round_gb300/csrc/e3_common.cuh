// e3_common.cuh -- shared device helpers of libeagle3 (CUDA, sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <utility>
#include <stdint.h>

#include "../../include/eagle3.h"

namespace e3 {

// ---------------------------------------------------------------------------
// host-side error reporting
// ---------------------------------------------------------------------------
void set_error(const char* fmt, ...);
// Empties the calling thread's error message (every entry point starts with it).
void clear_error();
e3_status cuda_status(cudaError_t e, const char* what);

#define E3_REQUIRE(cond, code, ...)   \
  do {                                \
    if (!(cond)) {                    \
      ::e3::set_error(__VA_ARGS__);   \
      return code;                    \
    }                                 \
  } while (0)

// Host-side count of the library's kernel launches (eagle3_launch_count).
void note_launch();

// After one kernel launch: report a launch error, else count the launch.
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization and calls pdl_wait() before its first access
// to global memory, which returns once the preceding kernel has completed and its
// writes are visible; so only the launch itself (and setup in shared or tensor
// memory) overlaps the predecessor, never work on its results.  pdl_trigger()
// lets the next kernel be scheduled early (it waits the same way).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// cudaLaunchKernelEx with programmatic stream serialization and, for cluster_x > 1,
// clusters of cluster_x CTAs along x.  Counts the launch when it succeeds.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) note_launch();
  return e;
}

#define E3_LAUNCH_CHECK(what)                                   \
  do {                                                          \
    cudaError_t _e = cudaGetLastError();                        \
    if (_e != cudaSuccess) return ::e3::cuda_status(_e, what);  \
    ::e3::note_launch();                                        \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// device error word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dev_flag(int32_t* dev_err, int bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// ---------------------------------------------------------------------------
// element loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ld_elem(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_elem(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------------------
// Fixed-point softmax decision arithmetic (fp32, every operation explicitly
// rounded so that no contraction changes a result).
//   E(x), x <= 0:  Cody-Waite reduction x = n ln2 + r (ln2 split into a 16-bit
//   high part and a low part), Taylor polynomial of exp(r) to degree 7 with
//   coefficients 1/k! rounded to fp32, Horner with fused multiply-add, then an
//   exact scaling by 2^n.  E(x) = 0 for x < -32.
//   mass(s, m) = floor(2^40 E(s - m)).
//   ell(Q) = ln(Q 2^-40): Q -> fp32 (nearest), exponent extraction, mantissa
//   folded into [sqrt(1/2), sqrt(2)], ln f = 2 atanh(t), t = (f-1)/(f+1), series
//   to t^11, plus (e - 40) ln2 (split).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fx_exp(float x) {
  if (x < -32.0f) return 0.0f;
  const float kLog2e = 0x1.715476p+0f;
  const float kLn2Hi = 0x1.62e4p-1f;
  const float kLn2Lo = 0x1.7f7d1cp-20f;
  float t = __fmul_rn(x, kLog2e);
  // n = rint(t) (ties to even) and its integer value, from t + 1.5 * 2^23: the sum
  // rounds t to an integer exactly as rint does for |t| < 2^22, and its low
  // mantissa bits are that integer (for larger |t| the result is zeroed below)
  const float tm = __fadd_rn(t, 0x1.8p23f);
  const float n = __fsub_rn(tm, 0x1.8p23f);
  const int ni = static_cast<int>(__float_as_uint(tm) - 0x4B400000u);
  float r = __fmaf_rn(-n, kLn2Hi, x);
  r = __fmaf_rn(-n, kLn2Lo, r);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  float scale = __uint_as_float(static_cast<uint32_t>(ni + 127) << 23);
  return __fmul_rn(p, scale);
}

// floor(e * 2^40) for 0 <= e <= 1, from the bits of e: e = 1.f x 2^E, so the
// product is the 24-bit significand shifted by sh = E + 17 <= 17.  The two 32-bit
// words of the result come from funnel shifts (a right shift by -sh > 31 and the
// zero and denormal encodings give 0), so no 64-bit shift and no float -> 64-bit
// integer conversion is needed; exact over every float in [0, 1] (checked against
// the 64-bit shift form on the GPU, all 1,065,353,217 encodings).
__device__ __forceinline__ uint64_t fx_scale40_floor(float e) {
  const uint32_t b = __float_as_uint(e);
  const int sh = static_cast<int>(b >> 23) - 110;
  const uint32_t mant = (b & 0x7FFFFFu) | 0x800000u;
  const uint32_t hi = __funnelshift_lc(mant, 0u, static_cast<unsigned>(max(sh, 0)));
  const uint32_t lo = sh >= 0 ? (mant << sh) : __funnelshift_rc(mant, 0u, static_cast<unsigned>(-sh));
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t fx_mass(float s, float m) {
  return fx_scale40_floor(fx_exp(__fsub_rn(s, m)));
}

// Two lanes of fx_exp at once with the packed fp32x2 operations (each lane is
// rounded exactly as the scalar operation it replaces, so the results are
// bit-identical to fx_exp on each lane).
__device__ __forceinline__ float2 fx_exp_x2(float2 x) {
  const float2 kLog2e = make_float2(0x1.715476p+0f, 0x1.715476p+0f);
  const float2 kLn2Hi = make_float2(0x1.62e4p-1f, 0x1.62e4p-1f);
  const float2 kLn2Lo = make_float2(0x1.7f7d1cp-20f, 0x1.7f7d1cp-20f);
  const float2 t = __fmul2_rn(x, kLog2e);
  // rint(t) and its integer value per lane, as in fx_exp (scalar adds: a paired
  // add may be contracted with the paired multiply above into one fused operation)
  const float2 tm = make_float2(__fadd_rn(t.x, 0x1.8p23f), __fadd_rn(t.y, 0x1.8p23f));
  const float2 nn = make_float2(__fsub_rn(0x1.8p23f, tm.x), __fsub_rn(0x1.8p23f, tm.y));  // -n
  const int nix = static_cast<int>(__float_as_uint(tm.x) - 0x4B400000u);
  const int niy = static_cast<int>(__float_as_uint(tm.y) - 0x4B400000u);
  float2 r = __ffma2_rn(nn, kLn2Hi, x);
  r = __ffma2_rn(nn, kLn2Lo, r);
  float2 p = make_float2(0x1.a01a02p-13f, 0x1.a01a02p-13f);
  p = __ffma2_rn(p, r, make_float2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
  p = __ffma2_rn(p, r, make_float2(0x1.111112p-7f, 0x1.111112p-7f));
  p = __ffma2_rn(p, r, make_float2(0x1.555556p-5f, 0x1.555556p-5f));
  p = __ffma2_rn(p, r, make_float2(0x1.555556p-3f, 0x1.555556p-3f));
  p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
  p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
  const float2 scale = make_float2(__uint_as_float(static_cast<uint32_t>(nix + 127) << 23),
                                   __uint_as_float(static_cast<uint32_t>(niy + 127) << 23));
  float2 e = __fmul2_rn(p, scale);
  if (x.x < -32.0f) e.x = 0.0f;
  if (x.y < -32.0f) e.y = 0.0f;
  return e;
}

// fx_mass(a, m) + fx_mass(b, m)
__device__ __forceinline__ uint64_t fx_mass_x2(float a, float b, float m) {
  const float2 e = fx_exp_x2(make_float2(__fsub_rn(a, m), __fsub_rn(b, m)));
  return fx_scale40_floor(e.x) + fx_scale40_floor(e.y);
}

__device__ __forceinline__ float fx_ell(uint64_t Q) {
  const float kLn2Hi = 0x1.62e4p-1f;
  const float kLn2Lo = 0x1.7f7d1cp-20f;
  float y = __ull2float_rn(Q);
  uint32_t b = __float_as_uint(y);
  int e = static_cast<int>(b >> 23) - 127;
  float f = __uint_as_float((b & 0x7FFFFFu) | 0x3F800000u);
  if (f > 0x1.6a09e6p+0f) {
    f = __fmul_rn(f, 0.5f);
    e += 1;
  }
  float t = __fdiv_rn(__fsub_rn(f, 1.0f), __fadd_rn(f, 1.0f));
  float t2 = __fmul_rn(t, t);
  float P = 0x1.745d18p-4f;
  P = __fmaf_rn(P, t2, 0x1.c71c72p-4f);
  P = __fmaf_rn(P, t2, 0x1.24924ap-3f);
  P = __fmaf_rn(P, t2, 0x1.99999ap-3f);
  P = __fmaf_rn(P, t2, 0x1.555556p-2f);
  P = __fmaf_rn(P, t2, 1.0f);
  float lnf = __fmul_rn(__fmul_rn(t, P), 2.0f);
  float k = static_cast<float>(e - 40);
  return __fmaf_rn(k, kLn2Hi, __fmaf_rn(k, kLn2Lo, lnf));
}

// 1/T for T > 0, else 1 (greedy rows keep s = z).
__device__ __forceinline__ float inv_temp(float T) {
  return T > 0.0f ? __fdiv_rn(1.0f, T) : 1.0f;
}

// (u * R) >> 32 for a uint32 uniform and a mass R < 2^57, exact.
__device__ __forceinline__ uint64_t mulhi32(uint32_t u, uint64_t R) {
  uint64_t lo = static_cast<uint64_t>(u) * R;  // low 64 bits of the product
  uint64_t hi = __umul64hi(static_cast<uint64_t>(u), R);
  return (hi << 32) | (lo >> 32);
}

// floor(a * b / c) for many a < 2^63 with b and c > 0 fixed, without a division
// per a: b / c = I + bm / c (I = floor(b / c), bm = b mod c) and
// rf = floor(bm 2^64 / c), so that t = floor(a rf / 2^64) is floor(a bm / c) or
// one less (a rf / 2^64 > a bm / c - a / 2^64 > a bm / c - 1); one exact
// comparison of (t + 1) c with a bm, as 128-bit (high, low) word pairs, settles
// it.  Exact whenever the result fits 64 bits.
struct FracMul {
  uint64_t I, bm, rf, c;
};
__device__ __forceinline__ FracMul frac_mul_prep(uint64_t b, uint64_t c) {
  FracMul f;
  f.c = c;
  f.I = b / c;
  f.bm = b - f.I * c;
  f.rf = static_cast<uint64_t>((static_cast<unsigned __int128>(f.bm) << 64) / c);
  return f;
}
__device__ __forceinline__ uint64_t frac_mul(const FracMul& f, uint64_t a) {
  const uint64_t t = __umul64hi(a, f.rf), t1 = t + 1;
  const uint64_t n_hi = __umul64hi(a, f.bm), n_lo = a * f.bm;
  const uint64_t m_hi = __umul64hi(t1, f.c), m_lo = t1 * f.c;
  const bool up = (m_hi < n_hi) || (m_hi == n_hi && m_lo <= n_lo);
  return a * f.I + (up ? t1 : t);
}

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): output number i >= 1 of the
// stream started at `seed` is mix(seed + i * 0x9E3779B97F4A7C15).
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
  uint64_t z = seed + i * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Order-preserving map of a finite float to uint32 (-0 folded onto +0).
__device__ __forceinline__ uint32_t ord_f32(float f) {
  f = __fadd_rn(f, 0.0f);
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(uint32_t o) {
  uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}

// Two floats -> packed bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// (value desc, id asc) packed so that a larger key is better.
__device__ __forceinline__ uint64_t pack_best(float v, uint32_t id) {
  return (static_cast<uint64_t>(ord_f32(v)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - id);
}
__device__ __forceinline__ uint32_t packed_id(uint64_t k) {
  return 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull);
}

// ---------------------------------------------------------------------------
// block reductions (blockDim.x a multiple of 32, <= 1024)
// ---------------------------------------------------------------------------
template <typename T, typename Op>
__device__ __forceinline__ T warp_reduce(T v, Op op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

template <typename T, typename Op>
__device__ T block_reduce(T v, Op op, T* smem32 /* >= 32 */) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_reduce(v, op);
  __syncthreads();
  if (lane == 0) smem32[wid] = v;
  __syncthreads();
  T r = smem32[0];
  for (int i = 1; i < nw; ++i) r = op(r, smem32[i]);
  return r;
}

struct MaxU64 {
  __device__ __forceinline__ uint64_t operator()(uint64_t a, uint64_t b) const { return a > b ? a : b; }
};
struct SumU64 {
  __device__ __forceinline__ uint64_t operator()(uint64_t a, uint64_t b) const { return a + b; }
};
struct MaxF {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct OrI {
  __device__ __forceinline__ int operator()(int a, int b) const { return a | b; }
};

// Block-wide bitonic sort of n (power of two) uint64 keys in shared memory,
// descending.
__device__ __forceinline__ void block_bitonic_desc(uint64_t* s, int n) {
  for (int kk = 2; kk <= n; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int ixj = i ^ j;
        if (ixj > i) {
          uint64_t a = s[i], b = s[ixj];
          bool first_half = (i & kk) == 0;
          if (first_half ? (a < b) : (a > b)) {
            s[i] = b;
            s[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace e3
