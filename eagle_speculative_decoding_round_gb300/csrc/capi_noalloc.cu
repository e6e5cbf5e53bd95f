// capi_noalloc.cu -- eagle3_fuse_noalloc: feature fusion for callers that cannot
// allocate device memory.
//
// eagle3_fuse needs caller-provided device scratch for its split-K partial sums.
// Some callers cannot provide it: they must not call cudaMalloc (or any routine
// that allocates, torch's caching allocator included) where they run the fusion
// -- a serving loop that must never block on or fragment the allocator, an
// embedder that has no device allocator of its own, or code running under a
// policy that forbids allocation at that point.  This entry point takes the same
// inputs and outputs but keeps its scratch in a fixed array inside the library.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes (4 MiB);
// every GPU that loads the library holds it until the process exits.  In host
// code its name is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current -- the
// first call on each device does this lookup, so make that first call before any
// stream capture.  (The library as a whole serves one device per process: its
// kernels' one-time attribute setup is per process; only this lookup is kept per
// device.)  All calls share the one array: calls that overlap on the GPU
// (different streams, or several host threads) race on it and must be ordered by
// the caller.  Each call overwrites every scratch element it later reads, so
// nothing has to start at zero.
#include <mutex>

#include "e3_common.cuh"
#include "e3_kernels.h"

namespace e3 {

namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fuse_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fuse_scratch on the current device (looked up once).
e3_status scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "eagle3_fuse_noalloc: cudaGetDevice");
  E3_REQUIRE(dev >= 0 && dev < kMaxDevices, E3_ERR_UNSUPPORTED, "eagle3_fuse_noalloc: device index %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fuse_scratch);
    if (e != cudaSuccess) return cuda_status(e, "eagle3_fuse_noalloc: cudaGetSymbolAddress");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return E3_OK;
}

}  // namespace

}  // namespace e3

using namespace e3;

extern "C" {

E3_API size_t eagle3_fuse_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

E3_API e3_status eagle3_fuse_noalloc(const void* h_low, const void* h_mid, const void* h_high, const void* W_f,
                                     const float* bias, void* g, int M, int d, int d_out, e3_dtype dt,
                                     int32_t* dev_err, e3_stream_t stream) {
  clear_error();
  E3_REQUIRE(h_low && h_mid && h_high && W_f && g, E3_ERR_INVALID_ARG, "eagle3_fuse_noalloc: null pointer");
  E3_REQUIRE(dt == E3_F32 || dt == E3_BF16, E3_ERR_INVALID_ARG, "eagle3_fuse_noalloc: bad dtype");
  E3_REQUIRE(M >= 1 && M <= 65536 && d >= 1 && d_out >= 1, E3_ERR_SHAPE,
             "eagle3_fuse_noalloc: bad sizes M=%d d=%d d_out=%d", M, d, d_out);
  E3_REQUIRE(static_cast<long>(d) * 3 < (1L << 30), E3_ERR_SHAPE, "eagle3_fuse_noalloc: d too large");
  if (eagle3_fuse_workspace_bytes(M, d, d_out, dt) == 0) {
    // this shape runs without scratch: the ordinary entry point allocates nothing either
    return eagle3_fuse(h_low, h_mid, h_high, W_f, bias, g, M, d, d_out, dt, nullptr, 0, dev_err, stream);
  }
  const size_t need = tc_fuse_workspace_bytes(M, d, d_out);
  E3_REQUIRE(need <= kNoAllocScratchBytes, E3_ERR_CAPACITY,
             "eagle3_fuse_noalloc: M=%d, d_out=%d need %zu bytes of scratch, more than the fixed %zu; use "
             "eagle3_fuse with a caller workspace",
             M, d_out, need, kNoAllocScratchBytes);
  E3_REQUIRE(aligned16(h_low) && aligned16(h_mid) && aligned16(h_high) && aligned16(W_f), E3_ERR_INVALID_ARG,
             "eagle3_fuse_noalloc: bf16 operands must be 16-byte aligned");
  void* scratch = nullptr;
  e3_status st = scratch_on_current_device(&scratch);
  if (st != E3_OK) return st;
  return launch_fuse_tc(h_low, h_mid, h_high, W_f, bias, g, M, d, d_out, scratch, kNoAllocScratchBytes, dev_err,
                        reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
