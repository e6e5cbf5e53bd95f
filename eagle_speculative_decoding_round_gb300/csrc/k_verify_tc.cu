// k_verify_tc.cu -- tree_verify_attn on the 5th-generation tensor cores (bf16,
// head_dim 128, pages of a multiple of 64 tokens).
//
// Same segment decomposition as the mma.sync kernel in k_verify.cu ("EAGLE-3 投机
// 解码与 USP 长序列训练优化", USP 核心设计：三步走: the prefix is the main segment,
// split across CTAs, the tree is the branch segment; all are merged by their
// log-sum-exp).  The mask is the ancestor-only tree mask of "EAGLE 系列与 DFlash",
// §二 关键新增步骤②.
//
// One CTA = (segment, 128-query-row group) of one KV head of one request.  The
// 128 rows are the G query heads of 128/G consecutive tree nodes (a 3-D TMA box
// over Q[B*R][H][hd]).  Keys stream in tiles of 128 (two 64-token page boxes per
// operand):
//   S = Q K^T    tcgen05.mma, M = 128 rows, N = 128 keys, K = head_dim (K-major),
//                into one of two S buffers in TMEM
//   softmax      the kParts threads of a query row read its TMEM lane (kPK keys
//                each); running max and sum in registers; P (bf16) is written
//                back over S in TMEM
//   O += P V     tcgen05.mma with A (P) from TMEM, N = head_dim, K = keys; V is
//                used in place as an MN-major operand.  O stays in TMEM for the
//                whole key range: its exponent base moves only when a tile's
//                maximum exceeds it by more than 2^8, and then the softmax warps
//                rescale it in place.
// Warps: 0 K loads (TMA), 1 TMEM owner + MMA issuer, 2 .. kVWarp-1 softmax and
// epilogue (kParts warps per TMEM lane quarter, each owning kPK keys of a tile and
// kPD head dims of O), kVWarp V loads (TMA).
//
// Segments are combined in one of three ways.  A row group that is not split (S =
// 1) writes O and lse directly.  CLUSTER with S > 1: the S segments of one row
// group form a thread-block cluster; every CTA stores its partial (o, m, l) rows
// into the owning CTA's receive area with distributed-shared-memory stores, and
// after one cluster barrier each CTA merges and writes its rows.  Otherwise
// (prefixes long enough to fill the GPU with independent CTAs) the partial records
// go to a workspace and verify_merge_kernel combines them.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr int kRows = 128;      // query rows per CTA
constexpr int kKeys = 128;      // keys per tile
constexpr int kHD = 128;        // head dim
constexpr int kHalf = 64;       // head-dim (or key) elements per 128-byte row
constexpr int kBox = kHalf * kHalf * 2;        // 64 x 64 bf16 = 8 KB
constexpr int kQBytes = kRows * kHD * 2;       // 32 KB (two 16 KB halves)
constexpr int kKVBytes = kKeys * kHD * 2;      // 32 KB per operand per tile
constexpr int kRowCache = 128;       // KV block rows looked up ahead
constexpr int kParts = 2;             // parts of a query row (warps per TMEM lane quarter)
constexpr int kPK = kKeys / kParts;   // keys of a part per tile
constexpr int kPD = kHD / kParts;     // head dims of a part
constexpr int kSoftmaxThreads = 128 * kParts;
constexpr int kVWarp = 2 + 4 * kParts;  // warp 0 K loads, warp 1 MMA, softmax warps, then the V-load warp
constexpr int kThreads = 32 * (kVWarp + 1);
static_assert(kParts >= 1 && kParts <= 4 && kKeys % (32 * kParts) == 0, "parts of 32-key multiples, at most four");
// Cluster merge receive area: (128 + 15) rows (the most a CTA owns times 16 segments)
// of bf16 partial o and float2 (m, l), written by every CTA of the cluster.
constexpr int kRecvRows = kRows + 15;
constexpr int kRecvBytes = kRecvRows * (kHD * 2 + 8);
constexpr int kSmem = 1024 + kQBytes + 4 * kKVBytes + 256 + 12 * 128 * 4 + 4 * kRowCache + 64 + kRecvBytes + 16;
constexpr float kLog2e = 1.4426950408889634f;
static_assert(kQBytes == kKVBytes, "Q and K halves share the slice offsets");
constexpr float kLazy = 8.0f;  // log2 headroom before the exponent base moves
constexpr unsigned long long kWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void bar_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
               : "=r"(ok)
               : "r"(su32(b)), "r"(par)
               : "memory");
  return ok != 0;
}
// Bounded wait: mbarrier.try_wait suspends the thread in hardware until the phase
// completes or a short system-dependent limit passes; the clock and the abort flag
// are checked every 64 probes.
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t par, volatile int* abort) {
  if (bar_try(b, par)) return true;
  const uint64_t t0 = gtimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (bar_try(b, par)) return true;
    if (*abort) return false;
    if (gtimer() - t0 > kWaitNs) {
      *abort = 1;
      return false;
    }
  }
}
// Wait bounded by time only (for copies that are in flight whatever the abort flag says).
__device__ __forceinline__ bool bar_wait_timed(uint64_t* b, uint32_t par) {
  if (bar_try(b, par)) return true;
  const uint64_t t0 = gtimer();
  while (gtimer() - t0 < kWaitNs)
    if (bar_try(b, par)) return true;
  return false;
}
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* b) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
                   "r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(su32(b))
               : "memory");
}
__device__ __forceinline__ void tma3d(void* dst, const CUtensorMap* m, int x, int y, int z, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(su32(b))
      : "memory");
}
// 128-byte-swizzled smem descriptor; lbo/sbo in bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// kind::f16 instruction descriptor: bf16 x bf16 -> f32, M x N, operand majors.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::
                   "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc));
}
// D = A(TMEM) * B(smem): A is M x K with row i in TMEM lane i and two 16-bit
// K elements per 32-bit column (the lower half is the lower K index).
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::
                   "r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b)) : "memory");
}
// 64 consecutive 32-bit TMEM columns of this thread's lane as 32 register pairs,
// one load instruction and one wait
__device__ __forceinline__ void tmem_ld64p(uint32_t taddr, float (&v)[64]) {
  unsigned long long q[32];
  asm volatile(
      "{\n .reg .b32 t<64>;\n"
      " tcgen05.ld.sync.aligned.32x32b.x64.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15,t16,t17,t18,t19,t20,t21,t22,t23,t24,t25,t26,t27,t28,t29,t30,t31,t32,t33,t34,t35,t36,t37,t38,t39,t40,t41,t42,t43,t44,t45,t46,t47,t48,t49,t50,t51,t52,t53,t54,t55,t56,t57,t58,t59,t60,t61,t62,t63}, [%32];\n"
      " tcgen05.wait::ld.sync.aligned;\n"
      " mov.b64 %0, {t0, t1};\n"
      " mov.b64 %1, {t2, t3};\n"
      " mov.b64 %2, {t4, t5};\n"
      " mov.b64 %3, {t6, t7};\n"
      " mov.b64 %4, {t8, t9};\n"
      " mov.b64 %5, {t10, t11};\n"
      " mov.b64 %6, {t12, t13};\n"
      " mov.b64 %7, {t14, t15};\n"
      " mov.b64 %8, {t16, t17};\n"
      " mov.b64 %9, {t18, t19};\n"
      " mov.b64 %10, {t20, t21};\n"
      " mov.b64 %11, {t22, t23};\n"
      " mov.b64 %12, {t24, t25};\n"
      " mov.b64 %13, {t26, t27};\n"
      " mov.b64 %14, {t28, t29};\n"
      " mov.b64 %15, {t30, t31};\n"
      " mov.b64 %16, {t32, t33};\n"
      " mov.b64 %17, {t34, t35};\n"
      " mov.b64 %18, {t36, t37};\n"
      " mov.b64 %19, {t38, t39};\n"
      " mov.b64 %20, {t40, t41};\n"
      " mov.b64 %21, {t42, t43};\n"
      " mov.b64 %22, {t44, t45};\n"
      " mov.b64 %23, {t46, t47};\n"
      " mov.b64 %24, {t48, t49};\n"
      " mov.b64 %25, {t50, t51};\n"
      " mov.b64 %26, {t52, t53};\n"
      " mov.b64 %27, {t54, t55};\n"
      " mov.b64 %28, {t56, t57};\n"
      " mov.b64 %29, {t58, t59};\n"
      " mov.b64 %30, {t60, t61};\n"
      " mov.b64 %31, {t62, t63};\n"
      "}\n"
      : "=l"(q[0]), "=l"(q[1]), "=l"(q[2]), "=l"(q[3]), "=l"(q[4]), "=l"(q[5]), "=l"(q[6]), "=l"(q[7]), "=l"(q[8]), "=l"(q[9]), "=l"(q[10]), "=l"(q[11]), "=l"(q[12]), "=l"(q[13]), "=l"(q[14]), "=l"(q[15]), "=l"(q[16]), "=l"(q[17]), "=l"(q[18]), "=l"(q[19]), "=l"(q[20]), "=l"(q[21]), "=l"(q[22]), "=l"(q[23]), "=l"(q[24]), "=l"(q[25]), "=l"(q[26]), "=l"(q[27]), "=l"(q[28]), "=l"(q[29]), "=l"(q[30]), "=l"(q[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[2 * i] = __uint_as_float(static_cast<uint32_t>(q[i]));
    v[2 * i + 1] = __uint_as_float(static_cast<uint32_t>(q[i] >> 32));
  }
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 consecutive 32-bit TMEM columns of this thread's lane, as floats (load / store)
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]));
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// 16 bytes / 8 bytes into (possibly another CTA's) shared memory at a shared::cluster address
__device__ __forceinline__ void st_cluster_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ void st_cluster_v2f(uint32_t a, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// bit j set iff lo <= T0 + j < hi (j < 32)
__device__ __forceinline__ uint32_t range_bits32(int T0, int lo, int hi) {
  const int a = max(lo - T0, 0), e = min(hi - T0, 32);
  if (e <= a) return 0u;
  const uint32_t upto = e >= 32 ? 0xFFFFFFFFu : ((1u << e) - 1u);
  return upto & ~((1u << a) - 1u);
}
// bit j = mask bit (j0 + j) of an ancestor row of `words` uint64 words, 0 outside it
__device__ __forceinline__ uint32_t mask_bits32(const uint64_t* row, int words, int j0) {
  uint32_t out = 0;
  const int w0 = j0 >> 6;  // floor division (j0 may be negative)
  for (int w = w0; w <= w0 + 1; ++w) {
    if (w < 0 || w >= words) continue;
    const uint64_t bits = row[w];
    const int sh = w * 64 - j0;  // position of word bit 0 in the output
    if (sh >= 0) {
      if (sh < 32) out |= static_cast<uint32_t>(bits << sh);
    } else if (-sh < 64) {
      out |= static_cast<uint32_t>(bits >> (-sh));
    }
  }
  return out;
}

struct TcGeom {
  int B, R, H, KVH, G, n_pre, S, chunk, RG, max_kv_len;
  int prefix_stable;  // E3_KV_PREFIX_STABLE: prefix K/V, lengths and pages may be read before the wait
  int stall;          // E3_KV_SELFTEST_STALL: the MMA thread waits on a barrier nothing arrives on
  int fold_tree;  // 1: segment S-1 also processes the tree slots (no separate tree segment)
  int page_size, max_pages, n_pages;
  const int32_t* page_table;
};

__device__ __forceinline__ int page_of(const TcGeom& g, int b, int t, bool* ok) {
  const int pi = t / g.page_size;
  if (pi < 0 || pi >= g.max_pages) {
    *ok = false;
    return 0;
  }
  const int p = g.page_table[static_cast<size_t>(b) * g.max_pages + pi];
  if (p < 0 || p >= g.n_pages) {
    *ok = false;
    return 0;
  }
  return p;
}

// CLUSTER: the S segments of one (row group, KV head, request) form one cluster;
// after their tile loops each CTA pushes its partial (o, m, l) rows into the
// shared memory of the CTA that owns those rows, and each CTA merges and writes
// the final O and lse of its slice.  Otherwise partial records go to the
// workspace for verify_merge_kernel.
template <bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, TcGeom g, const int32_t* __restrict__ kv_len,
                 const uint64_t* __restrict__ mask, float sm_scale, float* __restrict__ ws_o,
                 float2* __restrict__ ws_ml, __nv_bfloat16* __restrict__ O, float* __restrict__ lse,
                 int32_t* dev_err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // Tile t uses K stage, V stage and TMEM S/O buffer t % 2.  K(t) is released as
  // soon as S(t) has been computed and V(t) once PV(t) has run, so the next tiles'
  // loads start early.  P(t) is written (bf16) over S(t) in tensor memory.
  unsigned char* sQ = sm;                                  // [2 halves][128 rows][128 B]
  unsigned char* sK = sQ + kQBytes;                        // [2 stages][2 hd halves][128 keys][128 B]
  unsigned char* sV = sK + 2 * kKVBytes;                   // [2 stages][2 hd halves][128 keys][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + 2 * kKVBytes);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* k_empty = bars + 3;    // [2]
  uint64_t* v_full = bars + 5;     // [2]
  uint64_t* v_empty = bars + 7;    // [2]
  uint64_t* s_full = bars + 9;     // [2]
  uint64_t* p_full = bars + 11;    // [2]
  uint64_t* o_done = bars + 13;    // PV(t) completed (once per tile); bars + 19 unused
  uint64_t* stall_bar = bars + 14; // (self-test) never arrived on
  uint64_t* xch = bars + 15;       // [4] exchange among the parts of a row, per lane quarter
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ int s_kv_last[4];  // last tile loaded into K stage 0/1 and V stage 0/1 (-1: none)
  float* s_max = reinterpret_cast<float*>(tmem_slot + 4);  // [2 parities][kParts <= 4][128 rows]
  float* s_l = s_max + 8 * kRows;                           // [kParts <= 4][128 rows]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = CLUSTER ? blockIdx.x / g.S : blockIdx.x % g.RG;
  const int s = CLUSTER ? blockIdx.x % g.S : blockIdx.x / g.RG;
  const int kvh = blockIdx.y;
  const int nodes_per_tile = kRows / g.G;
  const int i0 = rg * nodes_per_tile;  // first node of this row group
  if (threadIdx.x == 0) {  // barriers first: they depend on nothing in global memory
    bar_init(q_full, 1);
    for (int bb = 0; bb < 2; ++bb) {
      bar_init(&k_full[bb], 1);
      bar_init(&k_empty[bb], 1);
      bar_init(&v_full[bb], 1);
      bar_init(&v_empty[bb], 1);
      bar_init(&s_full[bb], 1);
      bar_init(&p_full[bb], kSoftmaxThreads / 32);  // one arrival per softmax warp
    }
    for (int qq = 0; qq < 4; ++qq) bar_init(&xch[qq], kParts);  // one arrival per part (warp) of a lane quarter
    bar_init(o_done, 1);
    bar_init(stall_bar, 1);
    for (int i = 0; i < 4; ++i) s_kv_last[i] = -1;
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)), "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // Launched as a programmatic dependent: everything above touches only this CTA's
  // shared and tensor memory.  Without the prefix-stable promise nothing in global
  // memory is read before the preceding kernel has completed.  With it (the prefix
  // K/V, kv_len and the page table are not written by that kernel), the request
  // lengths and page-table rows are read and the first prefix tiles' K/V loads are
  // issued before the wait; Q, the mask and the tree slots only after it, and
  // nothing is written to global memory before it.
  if (!g.prefix_stable) asm volatile("griddepcontrol.wait;" ::: "memory");
  auto issue_q = [&](int bq) {
    bar_expect(q_full, kQBytes);
    for (int h = 0; h < 2; ++h) tma3d(sQ + h * (kQBytes / 2), &tmQ, h * kHalf, kvh * g.G, bq * g.R + i0, q_full);
  };
  // Requests are taken in order of decreasing length (ties: lower index first): the
  // CTAs of blockIdx.z = j serve the request of rank j, so that the longest requests
  // are launched first and the short ones fill the last wave.
  int b = blockIdx.z;
  if (gridDim.z > 1) {
    __shared__ int s_req;
    const int nb = static_cast<int>(gridDim.z);
    for (int c = threadIdx.x; c < nb; c += blockDim.x) {
      const int Pc = kv_len[c];
      int rank = 0;
      for (int o = 0; o < nb; ++o) {
        const int Po = kv_len[o];
        rank += (Po > Pc) || (Po == Pc && o < c);
      }
      if (rank == static_cast<int>(blockIdx.z)) s_req = c;
    }
    __syncthreads();
    b = s_req;
  }
  if (!g.prefix_stable && threadIdx.x == 0) issue_q(b);  // Q may be read now: it overlaps the length reads
  // Warp 0 loads, together with the request's length, the page-table entries of
  // this segment's first prefix blocks as they are if the prefix covers the whole
  // segment; after the length is known they are kept where that guess holds.
  const int spec_base = (g.fold_tree || s < g.n_pre) ? s * g.chunk : -1;
  int spec[kRowCache / 32];
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < kRowCache / 32; ++k) {
      const int pi = (spec_base + (lane + 32 * k) * kHalf) / g.page_size;
      spec[k] = (spec_base >= 0 && pi < g.max_pages) ? g.page_table[static_cast<size_t>(b) * g.max_pages + pi] : -1;
    }
  }
  const int P = kv_len[b];
  const long need = static_cast<long>(P) + g.R;
  if (P < 0 || P > g.max_kv_len || need > static_cast<long>(g.max_pages) * g.page_size) {
    if (g.prefix_stable) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
      if (blockIdx.x == 0 && kvh == 0) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
      if (!g.prefix_stable) bar_wait_timed(q_full, 0);  // the Q load lands before the CTA leaves
    }
    // the tensor memory allocated above is released (uniform across the CTA: same request)
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tmem_slot), "r"(512));
    return;  // uniform across the cluster (same request)
  }
  // key ranges of this CTA: a prefix range [pk0, pk1) and, for the tree segment
  // (or the last segment when the tree is folded in), the tree slots [P, P + R)
  int pk0 = 0, pk1 = 0;
  bool has_tree;
  if (g.fold_tree) {
    pk0 = min(P, s * g.chunk);
    pk1 = min(P, pk0 + g.chunk);
    has_tree = (s == g.S - 1);
  } else if (s == g.n_pre) {
    has_tree = true;
  } else {
    pk0 = min(P, s * g.chunk);
    pk1 = min(P, pk0 + g.chunk);
    has_tree = false;
  }
  const int tA = pk0 & ~(kHalf - 1);
  const int ntA = pk1 > pk0 ? (pk1 - tA + kKeys - 1) / kKeys : 0;
  const int tB = P & ~(kHalf - 1);
  const int ntB = has_tree ? (P + g.R - tB + kKeys - 1) / kKeys : 0;
  const int ntile = ntA + ntB;
  auto tile_T0 = [&](int t) { return t < ntA ? tA + t * kKeys : tB + (t - ntA) * kKeys; };
  auto tile_lo = [&](int t) { return t < ntA ? pk0 : P; };
  auto tile_hi = [&](int t) { return t < ntA ? pk1 : P + g.R; };

  // rows of the first kRowCache 64-key blocks, looked up by warp 0's lanes in parallel
  int* s_rows = reinterpret_cast<int*>(s_l + 4 * kRows);  // [kRowCache], -1 = bad page
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < kRowCache / 32; ++k) {
      const int i = lane + 32 * k;
      if (i < 2 * ntile) {
        const int T = tile_T0(i >> 1) + (i & 1) * kHalf;
        const int pi = T / g.page_size;
        int p = spec[k];
        if (T != spec_base + i * kHalf || spec_base < 0)
          p = pi < g.max_pages ? g.page_table[static_cast<size_t>(b) * g.max_pages + pi] : -1;
        const bool ok = pi < g.max_pages && p >= 0 && p < g.n_pages;
        s_rows[i] = (ok || T >= P + g.R) ? ((ok ? p : 0) * g.KVH + kvh) * g.page_size + (ok ? T % g.page_size : 0) : -1;
      }
    }
    __syncwarp();
  }
  auto block_row = [&](int i, bool* okp) {  // cache row of 64-key block i
    if (i < kRowCache) {
      const int row = s_rows[i];
      if (row < 0) {
        *okp = false;
        return 0;
      }
      return row;
    }
    const int T = tile_T0(i >> 1) + (i & 1) * kHalf;
    bool ok = true;
    const int page = page_of(g, b, T, &ok);
    const int slot = ok ? T % g.page_size : 0;
    if (!ok && T < P + g.R) *okp = false;
    return (page * g.KVH + kvh) * g.page_size + slot;
  };
  // load tile t's K (which = 0) or V (which = 1) into stage t % 2
  auto issue_kv = [&](int t, int which, bool* okp) {
    const int st = t & 1;
    unsigned char* base = (which ? sV : sK) + st * kKVBytes;
    uint64_t* bar = which ? &v_full[st] : &k_full[st];
    const CUtensorMap* map = which ? &tmV : &tmK;
    bar_expect(bar, kKVBytes);
    for (int blk = 0; blk < 2; ++blk) {
      const int row = block_row(2 * t + blk, okp);
      for (int h = 0; h < 2; ++h) tma2d(base + h * (kKVBytes / 2) + blk * kBox, map, h * kHalf, row, bar);
    }
    s_kv_last[which * 2 + st] = t;  // (written by the issuing thread only; read after the final barrier)
  };
  // The first two tiles' K and V.  Under the prefix-stable promise the prefix
  // tiles (t < ntA) are requested before the wait: their slots hold the committed
  // prefix (slots of the tree, which the preceding kernel may be writing, can share
  // a 64-key block with the prefix's last keys; they are outside [pk0, pk1), so
  // their scores are never used and their V rows are zeroed below).
  const int n_first = min(ntile, 2);
  const int n_early = g.prefix_stable ? min(n_first, ntA) : 0;
  bool okp0 = true;
  if (threadIdx.x == 0)
    for (int t = 0; t < n_early; ++t) {
      issue_kv(t, 0, &okp0);
      issue_kv(t, 1, &okp0);
    }
  if (g.prefix_stable) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    if (g.prefix_stable) issue_q(b);
    for (int t = n_early; t < n_first; ++t) {
      issue_kv(t, 0, &okp0);
      issue_kv(t, 1, &okp0);
    }
    if (!okp0) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM: S buffers at columns [0,128) and [128,256), O buffers at [256,384), [384,512)
  auto tS = [&](int bb) { return tmem + bb * kKeys; };
  const uint32_t tO = tmem + 2 * kKeys;  // the O accumulator

  if (warp == 0 || warp == kVWarp) {
    // warp 0 streams K, warp kVWarp streams V: each producer waits on its own
    // stage releases in a warp of its own, so neither wait delays the other's loads
    const int which = warp == 0 ? 0 : 1;
    if (lane == 0 && ntile > 2) {
      bool okp = true;
      for (int t = 2; t < ntile; ++t) {
        uint64_t* empty = which == 0 ? &k_empty[t & 1] : &v_empty[t & 1];
        if (!bar_wait(empty, ((t >> 1) & 1) ^ 1, abort)) break;
        issue_kv(t, which, &okp);
      }
      if (!okp) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
    }
  } else if (warp == 1) {
    if (lane == 0 && ntile > 0) {
      constexpr uint32_t idS = idesc_bf16(kRows, kKeys, 0, 0);
      constexpr uint32_t idO = idesc_bf16(kRows, kHD, 0, 1);
      // Descriptors are built once; a K slice or a stage only adds its byte offset / 16
      // to the start-address field (all addresses stay below 256 KB, so the 14-bit
      // field never carries into the others).  Issuing is then a few instructions per
      // MMA, so the tensor core, not the issuing thread, sets the pace.
      const uint64_t q_desc = desc_sw128(su32(sQ), 16, 1024);
      const uint64_t k_desc = desc_sw128(su32(sK), 16, 1024);
      const uint64_t v_desc = desc_sw128(su32(sV), kKVBytes / 2, 1024);
      auto issue_S = [&](int t) {  // S(t) = Q K(t)^T into S buffer t % 2; frees K stage t % 2
        const int bb = t & 1;
        const uint64_t kd = k_desc + static_cast<uint64_t>((bb * kKVBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          constexpr int kHalfBytes = kKVBytes / 2;  // == kQBytes / 2
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          umma(tS(bb), q_desc + off, kd + off, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[bb]);
        umma_commit(&k_empty[bb]);
      };
      // (self-test: a barrier nothing arrives on, so the bounded wait runs out)
      bool ok = g.stall ? bar_wait(stall_bar, 0, abort) : bar_wait(q_full, 0, abort);
      for (int t = 0; ok && t < ntile && t < 2; ++t) {
        if (!bar_wait(&k_full[t], 0, abort)) {
          ok = false;
          break;
        }
        fence_after();
        issue_S(t);
      }
      for (int t = 0; ok && t < ntile; ++t) {
        const int bb = t & 1;
        if (!bar_wait(&p_full[bb], (t >> 1) & 1, abort)) break;
        if (!bar_wait(&v_full[bb], (t >> 1) & 1, abort)) break;
        fence_after();
        const uint64_t vd = v_desc + static_cast<uint64_t>((bb * kKVBytes) >> 4);
        const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)  // O (+)= P(t) V(t) over keys; P from TMEM; 16 keys = 16 rows of 128 B
          umma_ts(tO, tS(bb) + kk * 8, vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), idO, kk > 0 ? 1u : acc0);
        umma_commit(o_done);  // O holds tiles 0..t; V stage t % 2 is free
        umma_commit(&v_empty[bb]);
        if (t + 2 < ntile) {
          // S(t+2) overwrites P(t): PV(t) must have completed
          if (!bar_wait(o_done, t & 1, abort)) break;
          if (!bar_wait(&k_full[bb], ((t + 2) >> 1) & 1, abort)) break;
          fence_after();
          issue_S(t + 2);
        }
      }
    }
  }
  // softmax warps 2..(2 + 4 kParts - 1): warp w reads TMEM lane quarter q = w % 4
  // (query rows 32q..32q+31) and owns part pp of the row: keys [kPK pp, kPK (pp+1))
  // of S and head dims [kPD pp, kPD (pp+1)) of O.  The parts of a row exchange maxima
  // and sums through shared memory, ordered by a per-quarter mbarrier (bounded wait).
  const bool softmax = warp >= 2 && warp < kVWarp;
  const int q = warp & 3;
  const int pp = softmax ? (warp - 2) >> 2 : 0;
  const int r = q * 32 + lane;
  const int gr = rg * kRows + r;  // row within the KV head's G*R rows
  const bool row_ok = softmax && gr < g.G * g.R;
  const int node = row_ok ? gr / g.G : 0;
  const int head = kvh * g.G + (row_ok ? gr % g.G : 0);
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  float m = -INFINITY, lt = 0.0f;  // exponent base (moved lazily) and the row's total sum
  bool live = true;
  if (softmax) {
    const int words = (g.R + 63) >> 6;
    const uint64_t* mrow = mask + (static_cast<size_t>(b) * g.R + node) * words;
    const float c2 = sm_scale * kLog2e;
    const int tid_sm = threadIdx.x - 64;  // 0 .. kSoftmaxThreads - 1
    float l = 0.0f;
    for (int t = 0; t < ntile; ++t) {
      const int T0 = tile_T0(t);
      const int k0 = tile_lo(t), k1 = tile_hi(t);
      const bool tree = t >= ntA;
      const int bb = t & 1;
      if (!bar_wait(&s_full[bb], (t >> 1) & 1, abort)) {
        live = false;
        break;
      }
      fence_after();
      static_assert(kPK == 64, "one 64-column load per part");
      float v[kPK];
      tmem_ld64p(tS(bb) + lane_base + pp * kPK, v);  // this part's scores
      uint32_t valid[kPK / 32];
      bool full = true;
#pragma unroll
      for (int c = 0; c < kPK / 32; ++c) {
        const int Tc = T0 + pp * kPK + 32 * c;
        valid[c] = range_bits32(Tc, k0, k1);
        if (tree) valid[c] &= mask_bits32(mrow, words, Tc - P);
        full = full && valid[c] == 0xFFFFFFFFu;  // interior chunk: no per-element tests
      }
      float pmax = -INFINITY;
      if (full) {
        float a0 = fmax3f(v[0], v[1], v[2]), a1 = fmax3f(v[3], v[4], v[5]);
        float a2 = fmax3f(v[6], v[7], v[8]), a3 = fmax3f(v[9], v[10], v[11]);
#pragma unroll
        for (int j = 12; j + 8 <= kPK - 4; j += 8) {
          a0 = fmax3f(a0, v[j], v[j + 1]);
          a1 = fmax3f(a1, v[j + 2], v[j + 3]);
          a2 = fmax3f(a2, v[j + 4], v[j + 5]);
          a3 = fmax3f(a3, v[j + 6], v[j + 7]);
        }
        a0 = fmax3f(a0, v[kPK - 4], v[kPK - 3]);
        a1 = fmax3f(a1, v[kPK - 2], v[kPK - 1]);
        pmax = fmax3f(a0, a1, fmaxf(a2, a3)) * c2;
      } else {
#pragma unroll
        for (int j = 0; j < kPK; ++j)
          if ((valid[j >> 5] >> (j & 31)) & 1u) pmax = fmaxf(pmax, v[j] * c2);
      }
      s_max[((t & 1) * kParts + pp) * kRows + r] = pmax;
      fence_before();  // this part's S loads are done before the others overwrite S with P
      __syncwarp();    // the warp's s_max writes, then one arrival for the warp
      if (lane == 0) bar_arrive(&xch[q]);
      // probabilities of this part's keys against base -nsub, packed to bf16 pairs
      uint32_t pk[kPK / 2];
      float rs = 0.0f;
      auto probs = [&](float nsub) {
        const float2 c2v = make_float2(c2, c2), nv = make_float2(nsub, nsub);
        float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                         make_float2(0.0f, 0.0f)};  // four independent sum chains
        if (full) {
#pragma unroll
          for (int j = 0; j < kPK; j += 2) {
            const float2 a = __ffma2_rn(make_float2(v[j], v[j + 1]), c2v, nv);
            const float e0 = fast_exp2(a.x), e1 = fast_exp2(a.y);
            acc[(j >> 1) & 3] = __fadd2_rn(acc[(j >> 1) & 3], make_float2(e0, e1));
            pk[j >> 1] = pack2_bf16(e0, e1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < kPK; j += 2) {
            const uint32_t vb = valid[j >> 5];
            const float2 a = __ffma2_rn(make_float2(v[j], v[j + 1]), c2v, nv);
            const float e0 = ((vb >> (j & 31)) & 1u) ? fast_exp2(a.x) : 0.0f;
            const float e1 = ((vb >> ((j + 1) & 31)) & 1u) ? fast_exp2(a.y) : 0.0f;
            acc[(j >> 1) & 3] = __fadd2_rn(acc[(j >> 1) & 3], make_float2(e0, e1));
            pk[j >> 1] = pack2_bf16(e0, e1);
          }
        }
        const float2 s01 = __fadd2_rn(acc[0], acc[1]), s23 = __fadd2_rn(acc[2], acc[3]);
        const float2 st = __fadd2_rn(s01, s23);
        rs = st.x + st.y;
      };
      // While the other parts' maxima arrive, the probabilities are computed against
      // the current base.  They are final unless some part of the row exceeds the base
      // by more than 2^kLazy (the first tile always does); then the tile is redone
      // below against the moved base.
      const bool spec = __all_sync(0xFFFFFFFFu, m != -INFINITY);
      if (spec) probs(-m);
      if (!bar_wait(&xch[q], t & 1, abort)) {
        live = false;
        break;
      }
      fence_after();
      float tmax = s_max[((t & 1) * kParts) * kRows + r];
#pragma unroll
      for (int x = 1; x < kParts; ++x) tmax = fmaxf(tmax, s_max[((t & 1) * kParts + x) * kRows + r]);
      // The base moves only when the tile's maximum exceeds it by more than 2^8; then
      // O (tiles 0..t-1, which needs PV(t-1) completed) is rescaled in TMEM, warp-
      // wide (lanes whose base stays multiply by 1).  Each thread waits every phase
      // of o_done in order: PV(t-1) here or before posting P(t).
      const bool move = tmax > m + kLazy;  // (also the first tile with a valid key)
      float corr = 1.0f;
      if (move) {
        corr = m == -INFINITY ? 0.0f : fast_exp2(m - tmax);
        l *= corr;
        m = tmax;
      }
      const bool any_move = __any_sync(0xFFFFFFFFu, move);
      bool waited_prev = false;
      if (t > 0 && any_move) {
        if (!bar_wait(o_done, (t - 1) & 1, abort)) {
          live = false;
          break;
        }
        waited_prev = true;
        fence_after();
#pragma unroll 1
        for (int h = 0; h < kPD / 16; ++h) {  // in 16-column steps, to keep register pressure low
          float ov[16];
          tmem_ld16f(tO + lane_base + pp * kPD + h * 16, ov);
#pragma unroll
          for (int j = 0; j < 16; ++j) ov[j] *= corr;
          tmem_st16f(tO + lane_base + pp * kPD + h * 16, ov);
        }
      }
      if (!spec || any_move) probs((m == -INFINITY) ? 0.0f : -m);
      l += rs;
      if (t > 0 && !waited_prev && !bar_wait(o_done, (t - 1) & 1, abort)) {
        live = false;
        break;
      }
      // P(t) over this part's S columns: keys [kPK pp, kPK (pp+1)) -> columns
      // [kPK/2 pp, kPK/2 (pp+1)) of the S buffer (all parts have read their scores:
      // the exchange above)
#pragma unroll
      for (int c = 0; c < kPK / 32; ++c)
        tmem_st16(tS(bb) + lane_base + pp * (kPK / 2) + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * c]));
      // V rows of keys outside the range are zeroed so that masked keys add exactly 0
      bool zeroed = false;
      if (tid_sm < kKeys) {
        const int T = T0 + tid_sm;
        if (T < k0 || T >= k1) {
          if (!bar_wait(&v_full[bb], (t >> 1) & 1, abort)) {
            live = false;
            break;
          }
          unsigned char* vst = sV + bb * kKVBytes;
          const uint4 z = make_uint4(0, 0, 0, 0);
          for (int h = 0; h < 2; ++h) {
            uint4* rowp = reinterpret_cast<uint4*>(vst + h * (kKVBytes / 2) + tid_sm * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) rowp[c] = z;
          }
          zeroed = true;
        }
      }
      if (zeroed) fence_async_smem();  // generic-proxy writes -> tensor core
      fence_before();                  // order the tcgen05.st before the arrival
      __syncwarp();
      if (lane == 0) bar_arrive(&p_full[bb]);
    }
    // total of the parts' sums
    s_l[pp * kRows + r] = l;
    __syncwarp();
    if (lane == 0) bar_arrive(&xch[q]);
    bar_wait(&xch[q], ntile & 1, abort);
    lt = 0.0f;
#pragma unroll
    for (int x = 0; x < kParts; ++x) lt += s_l[x * kRows + r];
  }
  // this part's kPD columns of O, from TMEM once the last PV has completed (zero
  // where no tile was processed); warp-uniform, as the TMEM loads are warp-wide
  float o[kPD];
  {
    bool o_ready = false;
    if (softmax && live && ntile > 0) {
      o_ready = bar_wait(o_done, (ntile - 1) & 1, abort);
      fence_after();
    }
    o_ready = __all_sync(0xFFFFFFFFu, o_ready);
#pragma unroll
    for (int c = 0; c < kPD / 32; ++c) {
      if (o_ready) {
        tmem_ld32(tO + lane_base + pp * kPD + 32 * c, *reinterpret_cast<float(*)[32]>(&o[32 * c]));
      } else {
#pragma unroll
        for (int d = 0; d < 32; ++d) o[32 * c + d] = 0.0f;
      }
    }
  }
  if (!CLUSTER && row_ok && !*abort) {
    const size_t rec = ((static_cast<size_t>(b) * g.S + s) * g.R + node) * g.H + head;
    const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
    float4* dst = reinterpret_cast<float4*>(ws_o + rec * kHD + pp * kPD);
#pragma unroll
    for (int d = 0; d < kPD / 4; ++d)
      dst[d] = make_float4(o[4 * d] * inv, o[4 * d + 1] * inv, o[4 * d + 2] * inv, o[4 * d + 3] * inv);
    if (pp == 0) ws_ml[rec] = make_float2(m, lt);
  }
  // Cluster merge.  Row r of the group is owned (merged and written) by CTA r / rpc
  // of the cluster.  Every CTA stores its normalized partial rows (bf16) and their
  // (m, l) straight into the owners' receive areas -- a region of its own in each
  // CTA's shared memory, so no CTA has to wait for another's tile loop before the
  // stores -- then one cluster barrier publishes them and each CTA merges its rows.
  const int rpc = CLUSTER ? (kRows + g.S - 1) / g.S : kRows;  // rows owned per CTA
  unsigned char* recv = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(s_rows + kRowCache) + 15) & ~static_cast<uintptr_t>(15));
  __nv_bfloat16* recv_o = reinterpret_cast<__nv_bfloat16*>(recv);         // [S][rpc][128]
  float2* recv_ml = reinterpret_cast<float2*>(recv + kRecvRows * kHD * 2);  // [S][rpc]
  if (CLUSTER && softmax && g.S == 1) {
    // the row group is not split: this part of the row is final
    if (row_ok && !*abort) {
      const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
      const size_t orow = (static_cast<size_t>(b) * g.R + node) * g.H + head;
      uint4* dst = reinterpret_cast<uint4*>(O + orow * kHD + pp * kPD);
#pragma unroll
      for (int k = 0; k < kPD / 8; ++k)
        dst[k] = make_uint4(pack2_bf16(o[8 * k] * inv, o[8 * k + 1] * inv), pack2_bf16(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                            pack2_bf16(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                            pack2_bf16(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
      if (pp == 0) lse[orow] = (m + __log2f(lt)) * 0.6931471805599453f;
    }
  } else if (CLUSTER && softmax) {
    const bool ok = row_ok && !*abort;
    const float inv = (ok && lt > 0.0f) ? 1.0f / lt : 0.0f;
    const int ow = r / rpc, li = r - ow * rpc;
    // this part's kPD head dims = 16-byte chunks of the row (8 bf16 each), XOR-swizzled
    // by the owner-local row so that the 32 lanes' stores spread over the banks
    const uint32_t row = cluster_addr(su32(recv_o + static_cast<size_t>(s * rpc + li) * kHD), ow);
#pragma unroll
    for (int k = 0; k < kPD / 8; ++k) {
      const int slot = ((kPD / 8) * pp + k) ^ (li & 7);
      st_cluster_v4(row + slot * 16, pack2_bf16(o[8 * k] * inv, o[8 * k + 1] * inv),
                    pack2_bf16(o[8 * k + 2] * inv, o[8 * k + 3] * inv), pack2_bf16(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                    pack2_bf16(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
    }
    if (pp == 0) st_cluster_v2f(cluster_addr(su32(recv_ml + s * rpc + li), ow), m, ok ? lt : 0.0f);
  }
  // the next kernel may be scheduled (it waits for this grid's completion before
  // touching global memory)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the Q load has landed (also where no tile was processed) before the CTA's
  // shared memory is reused or released
  if (threadIdx.x == 0 && !bar_wait_timed(q_full, 0)) *abort = 1;
  fence_before();
  if (__syncthreads_or(*abort != 0)) {
    // After an abort some K/V loads may never have been consumed: every load this CTA
    // issued lands (bounded by time) before its shared memory is reused or released.
    // Without an abort every load was waited on by its consumer.
    if (threadIdx.x == 0)
      for (int i = 0; i < 4; ++i) {
        const int t = s_kv_last[i];
        if (t >= 0) bar_wait_timed(i < 2 ? &k_full[i & 1] : &v_full[i & 1], (t >> 1) & 1);
      }
    __syncthreads();
  }
  if (*abort && threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_TIMEOUT);
  if (CLUSTER && g.S > 1) {
    const int S = g.S;
    const int n_own = max(0, min(rpc, kRows - s * rpc));
    __syncwarp();
    cluster_arrive_release();  // publishes the stores above to the owners
    cluster_wait();
    // merge: 16 threads per owned row, each with 8 head dims (one swizzled chunk)
    for (int it = threadIdx.x; it < n_own * 16; it += kThreads) {
      const int li = it >> 4, c = it & 15;
      const int rr = s * rpc + li;
      const int grr = rg * kRows + rr;
      if (grr < g.G * g.R) {
        const int nd = grr / g.G, hh = kvh * g.G + grr % g.G;
        const int slot = c ^ (li & 7);
        float M = -INFINITY;
        for (int sg = 0; sg < S; ++sg) {
          const float2 ml = recv_ml[sg * rpc + li];
          if (ml.y > 0.0f) M = fmaxf(M, ml.x);
        }
        float den = 0.0f;
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = 0.0f;
        for (int sg = 0; sg < S; ++sg) {
          const float2 ml = recv_ml[sg * rpc + li];
          const float w = ml.y > 0.0f ? ml.y * fast_exp2(ml.x - M) : 0.0f;
          den += w;
          const uint4 raw = reinterpret_cast<const uint4*>(recv_o + static_cast<size_t>(sg * rpc + li) * kHD)[slot];
          const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            a[2 * j] = fmaf(w, __uint_as_float(wd[j] << 16), a[2 * j]);
            a[2 * j + 1] = fmaf(w, __uint_as_float(wd[j] & 0xFFFF0000u), a[2 * j + 1]);
          }
        }
        const float inv = den > 0.0f ? 1.0f / den : 0.0f;
        const size_t orow = (static_cast<size_t>(b) * g.R + nd) * g.H + hh;
        uint4 pk;
        pk.x = pack2_bf16(a[0] * inv, a[1] * inv);
        pk.y = pack2_bf16(a[2] * inv, a[3] * inv);
        pk.z = pack2_bf16(a[4] * inv, a[5] * inv);
        pk.w = pack2_bf16(a[6] * inv, a[7] * inv);
        *reinterpret_cast<uint4*>(O + orow * kHD + c * 8) = pk;
        if (c == 0) lse[orow] = (M + __log2f(den)) * 0.6931471805599453f;
      }
    }
  }
  if (warp == 1) {
    __syncwarp();
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// How many clusters of S verify CTAs (one per SM) can be resident at once
// (0 if such clusters cannot be launched).
int max_active_clusters(int S) {
  static std::atomic<int> cache[17];  // 0: not yet known, -1: not launchable (idempotent entries)
  if (S < 1 || S > 16) return 0;
  if (cache[S].load(std::memory_order_relaxed) == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = S;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    cache[S].store((cudaOccupancyMaxActiveClusters(&n, verify_tc_kernel<true>, &cfg) == cudaSuccess && n > 0) ? n : -1,
                   std::memory_order_relaxed);
    cudaGetLastError();
  }
  const int v = cache[S].load(std::memory_order_relaxed);
  return v > 0 ? v : 0;
}

// Segments per cluster: the largest S (<= 16) whose clusters all fit in one wave
// and still give every CTA at least two 128-key tiles; 1 when the groups alone
// fill the GPU; 0 if no cluster can be launched.
int pick_cluster_segments(int groups, int max_kv_len) {
  if (max_active_clusters(1) == 0) return 0;
  if (groups >= max_active_clusters(1)) return 1;
  for (int S = 16; S >= 2; --S) {
    const int n = max_active_clusters(S);
    if (n >= groups && (max_kv_len + S - 1) / S >= 2 * kKeys) return S;
  }
  return 1;
}

}  // namespace

bool verify_tc_supported(const e3_kv_layer& kv, int H) {
  const int G = H / kv.n_kv_heads;
  return kv.dt == E3_BF16 && kv.head_dim == kHD && kv.page_size % kHalf == 0 && G >= 1 && G <= 16 &&
         (kRows % G) == 0;
}

e3_status launch_verify_tc(const void* Q, const e3_kv_layer& kv, const int32_t* kv_len, const uint64_t* mask, int B,
                           int R, int H, int max_kv_len, float sm_scale, VerifySplit* split, float* ws_o,
                           float2* ws_ml, void* O, float* lse, bool* merged, int32_t* dev_err, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  E3_REQUIRE(enc != nullptr, E3_ERR_CUDA, "tree_verify_attn: tensor-map encoder unavailable");
  const int G = H / kv.n_kv_heads;
  CUtensorMap mq, mk, mv;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B) * R};
    cuuint64_t str[2] = {static_cast<cuuint64_t>(kHD) * 2, static_cast<cuuint64_t>(H) * kHD * 2};
    cuuint32_t box[3] = {kHalf, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kRows / G)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(Q), dims, str, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    E3_REQUIRE(r == CUDA_SUCCESS, E3_ERR_INVALID_ARG, "tree_verify_attn: Q tensor map rejected (%d)", (int)r);
  }
  const cuuint64_t rows = static_cast<cuuint64_t>(kv.n_pages) * kv.n_kv_heads * kv.page_size;
  for (int w = 0; w < 2; ++w) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHD), rows};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(kHD) * 2};
    cuuint32_t box[2] = {kHalf, kHalf};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(w ? &mv : &mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w ? kv.v : kv.k, dims, str, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    E3_REQUIRE(r == CUDA_SUCCESS, E3_ERR_INVALID_ARG, "tree_verify_attn: KV tensor map rejected (%d)", (int)r);
  }
  TcGeom g;
  g.B = B;
  g.R = R;
  g.H = H;
  g.KVH = kv.n_kv_heads;
  g.G = G;
  g.n_pre = split->n_pre;
  g.S = split->S;
  g.chunk = split->chunk;
  g.RG = (G * R + kRows - 1) / kRows;
  g.max_kv_len = max_kv_len;
  g.page_size = kv.page_size;
  g.max_pages = kv.max_pages;
  g.n_pages = kv.n_pages;
  g.page_table = kv.page_table;
  g.fold_tree = 0;
  g.prefix_stable = (kv.flags & E3_KV_PREFIX_STABLE) ? 1 : 0;
  g.stall = (kv.flags & E3_KV_SELFTEST_STALL) ? 1 : 0;
  static std::atomic<bool> attr_done{false};
  if (!attr_done.load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(verify_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return cuda_status(e, "verify_tc_kernel smem attribute");
    cudaFuncSetAttribute(verify_tc_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaGetLastError();
    attr_done.store(true, std::memory_order_release);
  }
  *merged = false;
  const int groups = g.RG * kv.n_kv_heads * B;
  const int Sc = pick_cluster_segments(groups, max_kv_len);
  // The alternative: one wave of independent CTAs (as many segments as fit the
  // SMs and the workspace, tree folded into the last) and the separate merge
  // kernel.  It costs a few microseconds more in fixed latency, so it is taken
  // only where it saves at least four 128-key tiles per CTA.
  const int Sn = std::max(1, std::min(split->S, max_active_clusters(1) / std::max(1, groups)));
  auto tiles = [&](int Sx) { return ((max_kv_len + Sx - 1) / Sx + kKeys - 1) / kKeys; };
  const bool use_cluster = Sc >= 1 && (Sn <= Sc || tiles(Sc) - tiles(Sn) < 4);
  if (use_cluster) {
    // cluster mode: Sc prefix segments, the tree folded into the last one
    const int S = Sc;
    g.S = Sc;
    g.n_pre = Sc;
    g.fold_tree = 1;
    g.chunk = ((max_kv_len + Sc - 1) / Sc + kHalf - 1) / kHalf * kHalf;
    if (g.chunk < kHalf) g.chunk = kHalf;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.RG * S, kv.n_kv_heads, B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // programmatic dependent launch
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, verify_tc_kernel<true>, mq, mk, mv, g, kv_len, mask, sm_scale, ws_o,
                                       ws_ml, static_cast<__nv_bfloat16*>(O), lse, dev_err);
    if (e != cudaSuccess) return cuda_status(e, "verify_tc_kernel (cluster)");
    note_launch();
    *merged = true;
    return E3_OK;
  }
  if (Sn > 1 && Sn <= split->S) {  // one wave, tree folded into the last segment
    g.S = Sn;
    g.n_pre = Sn;
    g.fold_tree = 1;
    g.chunk = std::max(kHalf, ((max_kv_len + Sn - 1) / Sn + kHalf - 1) / kHalf * kHalf);
    *split = VerifySplit{Sn, Sn, g.chunk, 1};
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.RG * g.S, kv.n_kv_heads, B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;  // programmatic dependent launch
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, verify_tc_kernel<false>, mq, mk, mv, g, kv_len, mask, sm_scale, ws_o, ws_ml,
                                     static_cast<__nv_bfloat16*>(O), lse, dev_err);
  if (e != cudaSuccess) return cuda_status(e, "verify_tc_kernel");
  note_launch();
  return E3_OK;
}

}  // namespace e3
