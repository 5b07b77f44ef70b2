// moe_noalloc.cu -- moe_layer_noalloc: the whole layer with no caller workspace.
//
// Some callers cannot hand this library a workspace: code that runs inside an
// engine whose device-memory arena was reserved up front (a cudaMalloc there
// either fails or fragments the arena other components rely on), plugins and
// pure-C hosts with no allocator of their own, and latency-critical paths that
// must never touch the allocator.  For them the scratch memory the layer needs
// lives in one fixed device array in this file instead.
//
// Limits and sharing rules:
//  * the array holds MOE_NOALLOC_SCRATCH_BYTES (16 MiB); every GPU that loads the
//    library keeps it until the process exits.  A call whose workspace would not
//    fit (moe_workspace_size(desc, T) > 16 MiB) is rejected with
//    MOE_ERR_WORKSPACE before anything is launched;
//  * every call on a device uses the same array and it keeps whatever the last
//    call left there.  What must start at zero -- the error word and the fused
//    decode kernel's counters -- is zero-filled at set-up; the counters are left
//    zeroed by every call that completes, and the error word keeps the bits any
//    call set until moe_check_device_error(NULL, 0, stream) reads and clears it
//    (after a timeout that also zeroes the counters).  Every other region is
//    written before it is read.  Calls that overlap on the GPU (two streams, or
//    two host threads) race on the array: serialise them;
//  * the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current), caches it and zero-fills
//    the array's fixed head on the call's stream; make that first call before
//    any stream capture starts.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "moe_internal.cuh"

namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
bool g_any_setup = false;  // some device has been set up (read under the mutex)

// Device address of g_noalloc_scratch on the current device (looked up once).
// The first lookup on a device also zero-fills the workspace's fixed head (the
// error word and the counters that every call leaves zeroed), on `stream`.
cudaError_t scratch_address(void **out, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p, 0, MOE_WS_FIXED_BYTES, stream);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    g_any_setup = true;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

namespace moe {
// The array's address on the current device for moe_check_device_error, or null
// when no moe_layer_noalloc call has set it up there.  Before the first set-up
// on any device this makes no CUDA call at all.
void *noalloc_scratch_current() {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_any_setup) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return g_scratch_addr[dev];
}
}  // namespace moe

extern "C" moe_status moe_layer_noalloc(const moe_desc *desc, const moe_weights *wts,
                                        const float *x, const float *logits, const float *bias,
                                        uint32_t T, float *y, void *stream) {
  const size_t need = moe_workspace_size(desc, T);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > kScratchBytes) {
    moe::set_last_error(
        "moe_layer_noalloc: the workspace for this desc and T exceeds the 16 MiB static scratch");
    return MOE_ERR_WORKSPACE;
  }
  void *scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    moe::set_last_error(cudaGetErrorName(e));
    return MOE_ERR_CUDA;
  }
  return moe::layer_on_workspace(desc, wts, x, logits, bias, T, y, scratch, kScratchBytes,
                                 stream);
}
