// k_compact.cu -- kv_compact: commit only the accepted path's KV.
//
// "Thinking Budget 与 EAGLE-3", 一棵候选树怎样被验证, step 5: only the KV on the
// accepted path is committed and the other branches are released;
// "EAGLE 系列与 DFlash", §二 阶段三: decoding rolls back to the last accepted node.
//
// One CTA per (layer, KV head, request) slice.  The accepted nodes' rows are
// loaded into shared memory before any row is stored: path [0, 3, 4, 5] reads
// slot P+3 for element 1 while element 3 writes slot P+3.
#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

__device__ __forceinline__ char* kv_row_bytes(void* base, const e3_kv_layer& kv, int esz, int b, int kvh, int t,
                                             bool* ok) {
  const int pi = t / kv.page_size;
  if (t < 0 || pi >= kv.max_pages) {
    *ok = false;
    return nullptr;
  }
  const int page = kv.page_table[static_cast<size_t>(b) * kv.max_pages + pi];
  if (page < 0 || page >= kv.n_pages) {
    *ok = false;
    return nullptr;
  }
  const size_t row = (static_cast<size_t>(page) * kv.n_kv_heads + kvh) * kv.page_size + t % kv.page_size;
  return static_cast<char*>(base) + row * kv.head_dim * esz;
}

__global__ void __launch_bounds__(128)
compact_kernel(CompactLayers layers, e3_kv_layer geo, int D, const int32_t* __restrict__ path,
               const int32_t* __restrict__ acc_len, const int32_t* __restrict__ kv_len, int32_t* dev_err) {
  __shared__ __align__(16) uint4 buf[2 * E3_MAX_DEPTH * 64];  // up to 2 x 16 rows x 1 KiB
  pdl_wait();
  pdl_trigger();
  const int l = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int a = acc_len[b];
  if (a <= 0) return;
  if (a > D) {
    if (threadIdx.x == 0) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
    return;
  }
  const int P = kv_len[b];
  const int esz = geo.dt == E3_F32 ? 4 : 2;
  const int vec_per_row = geo.head_dim * esz / 16;
  geo.k = layers.k[l];
  geo.v = layers.v[l];
  bool ok = true;
  // load every source row (K and V) first
  for (int idx = threadIdx.x; idx < 2 * a * vec_per_row; idx += blockDim.x) {
    const int which = idx / (a * vec_per_row);
    const int rem = idx % (a * vec_per_row);
    const int j = rem / vec_per_row + 1, q = rem % vec_per_row;
    const int src = P + path[static_cast<size_t>(b) * (D + 1) + j];
    bool rok = true;
    const char* p = kv_row_bytes(which ? geo.v : geo.k, geo, esz, b, kvh, src, &rok);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (rok)
      v = reinterpret_cast<const uint4*>(p)[q];
    else
      ok = false;
    buf[(which * E3_MAX_DEPTH + (j - 1)) * 64 + q] = v;
  }
  if (!ok) dev_flag(dev_err, E3_DEV_ERR_CAPACITY);
  __syncthreads();
  for (int idx = threadIdx.x; idx < 2 * a * vec_per_row; idx += blockDim.x) {
    const int which = idx / (a * vec_per_row);
    const int rem = idx % (a * vec_per_row);
    const int j = rem / vec_per_row + 1, q = rem % vec_per_row;
    bool rok = true;
    char* p = kv_row_bytes(which ? geo.v : geo.k, geo, esz, b, kvh, P + j, &rok);
    if (rok) reinterpret_cast<uint4*>(p)[q] = buf[(which * E3_MAX_DEPTH + (j - 1)) * 64 + q];
  }
}

__global__ void kv_len_update_kernel(int B, const int32_t* __restrict__ acc_len, int32_t* kv_len) {
  pdl_wait();  // compact_kernel has read kv_len
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) kv_len[b] += 1 + acc_len[b];
}

}  // namespace

e3_status launch_compact(const CompactLayers& layers, const e3_kv_layer& geo, int L, int B, const int32_t* path,
                         const int32_t* acc_len, int D, int32_t* kv_len, int32_t* dev_err, cudaStream_t s) {
  cudaError_t e = launch_pdl(compact_kernel, dim3(L, geo.n_kv_heads, B), dim3(128), 0, s, 1, layers, geo, D, path,
                             acc_len, static_cast<const int32_t*>(kv_len), dev_err);
  if (e != cudaSuccess) return cuda_status(e, "compact_kernel");
  e = launch_pdl(kv_len_update_kernel, dim3((B + 255) / 256), dim3(256), 0, s, 1, B, acc_len, kv_len);
  if (e != cudaSuccess) return cuda_status(e, "kv_len_update_kernel");
  return E3_OK;
}

}  // namespace e3
