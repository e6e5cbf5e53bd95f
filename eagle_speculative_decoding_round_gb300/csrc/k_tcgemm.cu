// k_tcgemm.cu -- tcgen05 / TMEM / TMA GEMM for the two dense contractions of the
// round (bf16 in, fp32 accumulate):
//   LM head  ("SpecForge…", 先看 checkpoint 最终要参与什么计算): logits[m][v] = h[m] . W_lm[v]
//   fusion   ("SpecForge…", 多层特征融合到底融合了什么): g[m][o] = W_f[o] . [h_low; h_mid; h_high][m]
//
// Few tokens, many weight rows: the weight rows are the MMA's M side (128 per
// tile) and the tokens its N side (16..256), so one tile streams a 128-row slab
// of the weight through shared memory while the token tile stays L2-resident.
// Operands are K-major 128-byte-swizzled tiles loaded by TMA; the accumulator
// lives in tensor memory; one thread issues tcgen05.mma.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warps 2..5 epilogue (each reads the 32 TMEM lanes its warp may access).
// The LM head runs persistently (one CTA per SM, tiles round-robin) with the
// accumulator double-buffered in tensor memory, so that a tile's epilogue (the
// logits store and the per-token best key) overlaps the next tile's K loop.
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA sets
// E3_DEV_ERR_TIMEOUT, stops issuing, frees its TMEM and returns.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int A_BYTES = BM * BK * 2;
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; returns false (and raises *abort) if the phase did not complete.
// mbarrier.try_wait suspends in hardware; the clock is checked every 64 probes.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitNs) {
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_ss(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int BN>
struct TcCfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN <= 64 ? 4 : (BN <= 128 ? 5 : 4);
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int SMEM = 1024 /*align slack*/ + STAGES * STAGE + 512 /*barriers*/;
};

enum { kModePartial = 1 };

// out (kModePartial): split-K partial [Mx][Nw] fp32 of split blockIdx.z.
template <int BN, int MODE>
__global__ void __launch_bounds__(192, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2, int Nw, int Mx,
               int kb_per_src, int kb_total, int kb_per_split, float* __restrict__ out, int32_t* dev_err) {
  using C = TcCfg<BN>;
  pdl_wait();
  pdl_trigger();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* accum = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, tile_m = blockIdx.y, split = blockIdx.z;
  const int kb0 = split * kb_per_split;
  const int kb1 = min(kb_total, kb0 + kb_per_split);
  const int nkb = max(0, kb1 - kb0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      for (int it = 0; it < nkb; ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, abort)) break;
        unsigned char* a_s = smem + s * C::STAGE;
        unsigned char* b_s = a_s + A_BYTES;
        mbar_expect_tx(&full[s], C::STAGE);
        const int kb = kb0 + it;
        tma_load_2d(a_s, &tmA, kb * BK, tile_m * BM, &full[s]);
        const int src = kb / kb_per_src, kl = kb % kb_per_src;
        const CUtensorMap* mb = src == 0 ? &tmB0 : (src == 1 ? &tmB1 : &tmB2);
        tma_load_2d(b_s, mb, kl * BK, tile_n * BN, &full[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(BM, BN);
      const uint64_t desc0 = smem_desc(su32(smem));  // stage / K-slice offsets add to its address field
      for (int it = 0; it < nkb; ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&full[s], ph, abort)) break;
        tc_fence_after();
        const uint64_t da = desc0 + static_cast<uint64_t>((s * C::STAGE) >> 4);
        const uint64_t db = da + static_cast<uint64_t>(A_BYTES >> 4);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          mma_bf16_ss(tmem, da + 2 * k, db + 2 * k, idesc, (it | k) != 0);  // +32 bytes per K slice
        mma_commit(&empty[s]);  // frees the stage once these MMAs have read it
      }
      mma_commit(accum);  // accumulator complete (or nothing issued)
    }
  } else {
    // epilogue: warps 2..5 -> TMEM lane quarter (warp % 4)
    const int q = warp & 3;
    const int row = tile_m * BM + q * 32 + lane;
    bool ok = mbar_wait(accum, 0, abort);
    tc_fence_after();
    if (ok && nkb > 0) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, v);
        float* o = out + static_cast<size_t>(split) * Mx * Nw;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int m = tile_n * BN + c0 + j;
          if (m < Mx && row < Nw) o[static_cast<size_t>(m) * Nw + row] = v[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
  }
}

// g[m][o] = bf16(sum_z part[z][m][o] + bias[o])
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int Mx, int Nw,
                                     const float* __restrict__ bias, __nv_bfloat16* __restrict__ g) {
  pdl_wait();
  pdl_trigger();
  const size_t n = static_cast<size_t>(Mx) * Nw;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float acc = 0.0f;
    for (int z = 0; z < splits; ++z) acc += part[static_cast<size_t>(z) * n + i];
    if (bias) acc += bias[i % Nw];
    g[i] = __float2bfloat16_rn(acc);
  }
}

// ---------------------------------------------------------------------------
// LM head (persistent)
// ---------------------------------------------------------------------------
constexpr int kSmemCap = 227 * 1024;
constexpr int kXposeBytes = 4 * 32 * 33 * 8;  // per epilogue warp: 32 x 33 u64 (padded transpose)

template <int BN>
struct LmCfg {
  static_assert(BN % 32 == 0, "the epilogue reads 32 accumulator columns at a time");
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
  static constexpr int FIXED = 1024 /*align slack*/ + 256 /*barriers*/ + kXposeBytes + 4 * BN * 8 /*warp bests*/ +
                               BN * 4 /*inverse temperatures*/;
  static constexpr int FIT = (kSmemCap - FIXED) / STAGE;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int SMEM = FIXED + STAGES * STAGE;
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}

// logits[m][v] = h[m] . W[v] for every (128-row vocabulary tile, BN-token tile),
// tiles taken round-robin by a grid of at most one CTA per SM.  best[m] receives
// (atomic max) the packed key (z[m][v] / T_m, -v) of every tile, for the
// statistics pass that follows.
template <int BN>
__global__ void __launch_bounds__(192, 1)
lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int V, int M,
              int kb_total, int n_mt, int n_tiles, float* __restrict__ logits, unsigned long long* __restrict__ best,
              const float* __restrict__ temp, int32_t* dev_err) {
  using C = LmCfg<BN>;
  pdl_wait();
  pdl_trigger();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;   // [2] MMAs of the buffer's tile done
  uint64_t* acc_empty = acc_full + 2;       // [2] epilogue done reading the buffer
  uint64_t* ep_sync = acc_empty + 2;        // [2] epilogue-internal syncs (128 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ep_sync + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* xpose = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE + 256);  // [4][32][33]
  uint64_t* wbest = xpose + 4 * 32 * 33;                                                // [4][BN]
  float* s_it = reinterpret_cast<float*>(wbest + 4 * BN);                               // [BN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
      mbar_init(&ep_sync[a], 128);
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer: the K loop of every tile through one ring
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        const int vt = tile / n_mt, mt = tile % n_mt;
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait(&empty[st], ((it / C::STAGES) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          unsigned char* a_s = smem + st * C::STAGE;
          mbar_expect_tx(&full[st], C::STAGE);
          tma_load_2d(a_s, &tmA, kb * BK, vt * BM, &full[st]);
          tma_load_2d(a_s + A_BYTES, &tmB, kb * BK, mt * BN, &full[st]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = instr_desc(BM, BN);
      // descriptors built once: a stage or a K slice only adds its byte offset / 16 to
      // the start-address field (shared addresses stay below 256 KB: no carry)
      const uint64_t desc0 = smem_desc(su32(smem));
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++local) {
        const int a = local & 1;
        if (!mbar_wait(&acc_empty[a], ((local >> 1) & 1) ^ 1, abort)) break;
        tc_fence_after();
        const uint32_t d = tmem + a * BN;
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait(&full[st], (it / C::STAGES) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = desc0 + static_cast<uint64_t>((st * C::STAGE) >> 4);
          const uint64_t db = da + static_cast<uint64_t>(A_BYTES >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16_ss(d, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);  // +32 bytes per K slice
          mma_commit(&empty[st]);
        }
        if (ok) mma_commit(&acc_full[a]);
      }
    }
  } else {
    // epilogue warps 2..5: TMEM lane quarter q = warp % 4 (vocabulary rows 32q..32q+31 of the tile)
    const int q = warp & 3;
    const int et = threadIdx.x - 64;  // 0..127
    uint64_t* xp = xpose + q * 32 * 33;
    int bad = 0, local = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
      const int vt = tile / n_mt, mt = tile % n_mt;
      const int a = local & 1;
      for (int j = et; j < BN; j += 128) {
        const int m = mt * BN + j;
        s_it[j] = m < M ? inv_temp(temp[m]) : 1.0f;
      }
      mbar_arrive(&ep_sync[0]);
      if (!mbar_wait(&ep_sync[0], local & 1, abort)) break;
      if (!mbar_wait(&acc_full[a], (local >> 1) & 1, abort)) break;
      tc_fence_after();
      const int vrow = vt * BM + q * 32 + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + a * BN + (static_cast<uint32_t>(q * 32) << 16) + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int m = mt * BN + c0 + j;
          uint64_t key = 0ull;
          if (m < M) {
            const float z = v[j];
            bad |= !isfinite(z);
            if (vrow < V) {
              logits[static_cast<size_t>(m) * V + vrow] = z;
              key = pack_best(__fmul_rn(z, s_it[c0 + j]), static_cast<uint32_t>(vrow));
            }
          }
          xp[lane * 33 + j] = key;
        }
        __syncwarp();
        uint64_t kbest = 0ull;  // column c0 + lane: best of this warp's 32 rows
#pragma unroll 8
        for (int r = 0; r < 32; ++r) kbest = max(kbest, static_cast<uint64_t>(xp[r * 33 + lane]));
        if (c0 + lane < BN) wbest[q * BN + c0 + lane] = kbest;
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[a]);  // the accumulator buffer may take the tile after next
      mbar_arrive(&ep_sync[1]);
      if (!mbar_wait(&ep_sync[1], local & 1, abort)) break;
      for (int j = et; j < BN; j += 128) {  // one atomic per token column per tile
        const int m = mt * BN + j;
        if (m >= M) continue;
        uint64_t k = wbest[j];
        for (int qq = 1; qq < 4; ++qq) k = max(k, static_cast<uint64_t>(wbest[qq * BN + j]));
        if (k != 0ull) atomicMax(&best[m], static_cast<unsigned long long>(k));
      }
    }
    if (bad) dev_flag(dev_err, E3_DEV_ERR_NONFINITE);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
  }
}

// Second pass of the LM-head softmax statistics, one cluster of kRowQCluster CTAs
// per row: row_Q[m] holds the packed row maximum (from the GEMM epilogue); each
// CTA sums the fixed-point masses of its part of the row, CTA 0 adds the parts
// and publishes row_max, row_argmax and row_Q (row_Q doubles as the packed-
// maximum scratch; every CTA has read it before the first cluster barrier).
constexpr int kRowQCluster = 8;
constexpr int kRowQThreads = 256;

__global__ void __launch_bounds__(kRowQThreads)
row_q_kernel(const float* __restrict__ logits, int V, const float* __restrict__ temp, float* __restrict__ row_max,
             uint64_t* __restrict__ row_Q, int32_t* __restrict__ row_argmax) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ uint64_t red64[32];
  __shared__ int redi[32];
  __shared__ uint64_t part_Q;
  __shared__ int part_bad;
  const int rank = static_cast<int>(cluster.block_rank());
  const int m = blockIdx.x / kRowQCluster;
  pdl_wait();
  pdl_trigger();
  const float4* z4 = reinterpret_cast<const float4*>(logits + static_cast<size_t>(m) * V);
  const float it = inv_temp(temp[m]);
  const uint64_t best = row_Q[m];
  const float mx = unord_f32(static_cast<uint32_t>(best >> 32));
  const int nv4 = V >> 2;
  const int per = (nv4 + kRowQCluster - 1) / kRowQCluster;
  const int q0 = min(nv4, rank * per), q1 = min(nv4, q0 + per);
  uint64_t Q = 0;
  // non-finite logits on the fused multiply-add pipe (the masses keep the integer
  // pipe busy): z * 0 + acc stays 0 for finite z and turns NaN for an infinity or NaN
  float2 nf = make_float2(0.0f, 0.0f);
  const float2 zero2 = make_float2(0.0f, 0.0f);
  auto add4 = [&](const float4& v) {
    nf = __ffma2_rn(make_float2(v.x, v.y), zero2, nf);
    nf = __ffma2_rn(make_float2(v.z, v.w), zero2, nf);
    Q += fx_mass_x2(__fmul_rn(v.x, it), __fmul_rn(v.y, it), mx) + fx_mass_x2(__fmul_rn(v.z, it), __fmul_rn(v.w, it), mx);
  };
  // eight loads in flight per thread, then the masses of those inside the chunk
  for (int q8 = q0 + threadIdx.x; q8 < q1; q8 += 8 * kRowQThreads) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q8 + u * kRowQThreads;
      v[u] = q < q1 ? z4[q] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (q8 + u * kRowQThreads < q1) add4(v[u]);
  }
  int bad = (nf.x != nf.x) | (nf.y != nf.y);
  Q = block_reduce(Q, SumU64(), red64);
  bad = block_reduce(bad, OrI(), redi);
  if (threadIdx.x == 0) {
    part_Q = Q;
    part_bad = bad;
  }
  cluster.sync();  // every part is published; every CTA has read row_Q[m]
  if (rank == 0 && threadIdx.x < 32) {
    uint64_t v = 0ull;
    int bd = 0;
    if (threadIdx.x < kRowQCluster) {
      v = *cluster.map_shared_rank(&part_Q, threadIdx.x);
      bd = *cluster.map_shared_rank(&part_bad, threadIdx.x);
    }
    v = warp_reduce(v, SumU64());
    bd = warp_reduce(bd, OrI());
    if (threadIdx.x == 0) {
      row_max[m] = bd ? __int_as_float(0x7FC00000) : mx;
      row_argmax[m] = bd ? -1 : static_cast<int32_t>(packed_id(best));
      row_Q[m] = bd ? 0ull : v;
    }
  }
  cluster.sync();  // CTA 0 is done reading the others' shared memory
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// The driver's tensor-map encoder, looked up through the runtime so that the
// library does not link libcuda (it must load on machines without a driver).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {  // looked up once, thread-safely
    PFN_cuTensorMapEncodeTiled_v12000 found = nullptr;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      found = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return found;
  }();
  return fn;
}

bool make_map(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN>
e3_status launch_fuse_bn(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& b2,
                         int Nw, int Mx, int kb_per_src, int kb_total, int splits, float* out, int32_t* dev_err,
                         cudaStream_t s) {
  using C = TcCfg<BN>;
  static std::atomic<bool> attr_done{false};
  if (!attr_done.load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN, kModePartial>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return cuda_status(e, "tc_gemm_kernel smem attribute");
    attr_done.store(true, std::memory_order_release);
  }
  const int kb_per_split = (kb_total + splits - 1) / splits;  // callers pass splits with no empty split
  dim3 grid((Mx + BN - 1) / BN, (Nw + BM - 1) / BM, splits);
  const cudaError_t e = launch_pdl(tc_gemm_kernel<BN, kModePartial>, grid, dim3(192), C::SMEM, s, 1, a, b0, b1, b2, Nw,
                                   Mx, kb_per_src, kb_total, kb_per_split, out, dev_err);
  if (e != cudaSuccess) return cuda_status(e, "tc_gemm_kernel");
  return E3_OK;
}

e3_status dispatch_fuse(int bn, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const CUtensorMap& b2, int Nw, int Mx, int kb_per_src, int kb_total, int splits, float* out,
                        int32_t* dev_err, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_fuse_bn<16>(a, b0, b1, b2, Nw, Mx, kb_per_src, kb_total, splits, out, dev_err, s);
    case 32: return launch_fuse_bn<32>(a, b0, b1, b2, Nw, Mx, kb_per_src, kb_total, splits, out, dev_err, s);
    case 64: return launch_fuse_bn<64>(a, b0, b1, b2, Nw, Mx, kb_per_src, kb_total, splits, out, dev_err, s);
    case 128: return launch_fuse_bn<128>(a, b0, b1, b2, Nw, Mx, kb_per_src, kb_total, splits, out, dev_err, s);
    default: return launch_fuse_bn<256>(a, b0, b1, b2, Nw, Mx, kb_per_src, kb_total, splits, out, dev_err, s);
  }
}

int pick_bn(int Mx) {
  if (Mx <= 16) return 16;
  if (Mx <= 32) return 32;
  if (Mx <= 64) return 64;
  if (Mx <= 128) return 128;
  return 256;
}

// Splits of the K loop: about two CTAs per SM over the (token tile, weight tile) grid,
// at least four k-blocks per split, at most 16 splits, none empty.
int linear_splits_impl(int M, int K_total, int N) {
  const int tiles = ((M + pick_bn(M) - 1) / pick_bn(M)) * ((N + BM - 1) / BM);
  const int kb_total = K_total / BK;
  int splits = (2 * 148 + tiles - 1) / tiles;  // about two CTAs per SM
  if (splits > kb_total / 4) splits = kb_total / 4;
  if (splits < 1) splits = 1;
  if (splits > 16) splits = 16;
  const int per = (kb_total + splits - 1) / splits;
  return (kb_total + per - 1) / per;  // every split owns at least one k-block
}

int fuse_splits(int M, int d, int d_out) { return linear_splits_impl(M, 3 * d, d_out); }

}  // namespace

int linear_splits(int M, int K_total, int N) { return linear_splits_impl(M, K_total, N); }

size_t linear_partial_bytes(int M, int K_total, int N) {
  return static_cast<size_t>(linear_splits_impl(M, K_total, N)) * M * N * sizeof(float);
}

e3_status launch_linear_tc(const void* W, const void* const* src, int n_src, int K, int M, int N, float* part,
                           int* splits, int32_t* dev_err, cudaStream_t s) {
  E3_REQUIRE(n_src >= 1 && n_src <= 3 && K % BK == 0 && K >= BK && M >= 1 && N >= 1, E3_ERR_SHAPE,
             "linear: n_src=%d K=%d M=%d N=%d", n_src, K, M, N);
  const int bn = pick_bn(M);
  CUtensorMap a, b[3];
  bool ok = make_map(&a, W, N, n_src * K, BM);
  for (int i = 0; i < n_src; ++i) ok = ok && make_map(&b[i], src[i], M, K, bn);
  E3_REQUIRE(ok, E3_ERR_INVALID_ARG, "linear: cuTensorMapEncodeTiled rejected an operand");
  for (int i = n_src; i < 3; ++i) b[i] = b[0];
  *splits = linear_splits_impl(M, n_src * K, N);
  return dispatch_fuse(bn, a, b[0], b[1], b[2], N, M, K / BK, n_src * K / BK, *splits, part, dev_err, s);
}

bool tc_gemm_supported(int d_k, int n_rows) { return d_k % BK == 0 && n_rows >= 1; }

size_t tc_fuse_workspace_bytes(int M, int d, int d_out) {
  return static_cast<size_t>(fuse_splits(M, d, d_out)) * M * d_out * sizeof(float) + 256;
}

e3_status launch_fuse_tc(const void* h_low, const void* h_mid, const void* h_high, const void* W_f, const float* bias,
                         void* g, int M, int d, int d_out, void* ws, size_t ws_bytes, int32_t* dev_err,
                         cudaStream_t s) {
  const size_t need = tc_fuse_workspace_bytes(M, d, d_out);
  E3_REQUIRE(ws && ws_bytes >= need, E3_ERR_CAPACITY, "eagle3_fuse: workspace of %zu bytes needed, %zu given", need,
             ws_bytes);
  const int bn = pick_bn(M);
  CUtensorMap a, b0, b1, b2;
  E3_REQUIRE(make_map(&a, W_f, d_out, 3 * d, BM) && make_map(&b0, h_low, M, d, bn) && make_map(&b1, h_mid, M, d, bn) &&
                 make_map(&b2, h_high, M, d, bn),
             E3_ERR_INVALID_ARG, "eagle3_fuse: cuTensorMapEncodeTiled rejected an operand");
  const int splits = fuse_splits(M, d, d_out);
  float* part = static_cast<float*>(ws);
  e3_status st = dispatch_fuse(bn, a, b0, b1, b2, d_out, M, d / BK, 3 * d / BK, splits, part, dev_err, s);
  if (st != E3_OK) return st;
  const size_t n = static_cast<size_t>(M) * d_out;
  const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
  const cudaError_t e = launch_pdl(splitk_reduce_kernel, dim3(blocks), dim3(256), 0, s, 1,
                                   static_cast<const float*>(part), splits, M, d_out, bias,
                                   static_cast<__nv_bfloat16*>(g));
  if (e != cudaSuccess) return cuda_status(e, "splitk_reduce_kernel");
  return E3_OK;
}

template <int BN>
e3_status launch_lmhead_bn(const CUtensorMap& a, const CUtensorMap& b, int V, int M, int kb_total, float* logits,
                           unsigned long long* best, const float* temp, int32_t* dev_err, cudaStream_t s) {
  using C = LmCfg<BN>;
  static_assert(C::STAGES >= 2, "LM-head ring too small");
  static std::atomic<bool> attr_done{false};
  static std::atomic<int> n_sm{0};
  if (!attr_done.load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(lmhead_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return cuda_status(e, "lmhead_kernel smem attribute");
    int dev = 0;
    cudaGetDevice(&dev);
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    n_sm.store(n < 1 ? 1 : n, std::memory_order_relaxed);
    attr_done.store(true, std::memory_order_release);
  }
  const int n_mt = (M + BN - 1) / BN;
  const int n_vt = (V + BM - 1) / BM;
  const long n_tiles = static_cast<long>(n_mt) * n_vt;
  E3_REQUIRE(n_tiles < (1L << 31), E3_ERR_SHAPE, "lmhead_logits: %ld tiles", n_tiles);
  const int grid = static_cast<int>(std::min<long>(n_tiles, n_sm.load(std::memory_order_relaxed)));
  const cudaError_t e = launch_pdl(lmhead_kernel<BN>, dim3(grid), dim3(192), C::SMEM, s, 1, a, b, V, M, kb_total, n_mt,
                                   static_cast<int>(n_tiles), logits, best, temp, dev_err);
  if (e != cudaSuccess) return cuda_status(e, "lmhead_kernel");
  return E3_OK;
}

e3_status launch_lmhead_tc(const void* h, const void* W_lm, int M, int d, int V, const float* temp, float* logits,
                           float* row_max, uint64_t* row_Q, int32_t* row_argmax, int32_t* dev_err, cudaStream_t s) {
  const int bn = std::max(32, pick_bn(M));  // the epilogue reads the accumulator 32 columns at a time
  CUtensorMap a, b;
  E3_REQUIRE(make_map(&a, W_lm, V, d, BM) && make_map(&b, h, M, d, bn), E3_ERR_INVALID_ARG,
             "lmhead_logits: cuTensorMapEncodeTiled rejected an operand");
  cudaError_t e = cudaMemsetAsync(row_Q, 0, static_cast<size_t>(M) * sizeof(uint64_t), s);
  if (e != cudaSuccess) return cuda_status(e, "lmhead_logits memset");
  unsigned long long* best = reinterpret_cast<unsigned long long*>(row_Q);
  const int kb = d / BK;
  e3_status st;
  switch (bn) {
    case 32: st = launch_lmhead_bn<32>(a, b, V, M, kb, logits, best, temp, dev_err, s); break;
    case 64: st = launch_lmhead_bn<64>(a, b, V, M, kb, logits, best, temp, dev_err, s); break;
    case 128: st = launch_lmhead_bn<128>(a, b, V, M, kb, logits, best, temp, dev_err, s); break;
    default: st = launch_lmhead_bn<256>(a, b, V, M, kb, logits, best, temp, dev_err, s); break;
  }
  if (st != E3_OK) return st;
  e = launch_pdl(row_q_kernel, dim3(static_cast<unsigned>(M) * kRowQCluster), dim3(kRowQThreads), 0, s,
                 static_cast<unsigned>(kRowQCluster), static_cast<const float*>(logits), V, temp, row_max, row_Q,
                 row_argmax);
  if (e != cudaSuccess) return cuda_status(e, "row_q_kernel");
  return E3_OK;
}

}  // namespace e3
