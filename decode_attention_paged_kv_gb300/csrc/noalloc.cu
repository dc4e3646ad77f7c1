// noalloc.cu -- exact decode attention for callers that cannot hand the
// library a workspace.
//
// Some callers have no way to allocate device memory for us: an inference
// host whose allocator owns the whole device-memory budget and gives plugins
// none, or a latency-critical loop that must never reach cudaMalloc (which can
// synchronise the device).  dkv_decode_attn_full_noalloc serves them with a
// scratch area that lives in the library itself: a file-scope __device__ array
// of DKV_NOALLOC_SCRATCH_BYTES, created when the library's device code is
// loaded on a GPU and held by every GPU that loads it until the process exits.
//
// The entry point calls no allocator.  On the first call for a device (with
// that device current) it looks up the array's device address once; that first
// call should come before any stream capture.  Every call shares the array:
// calls that can overlap on the GPU (different streams, or graphs replayed
// concurrently) race on it and must be serialised by the caller.  Each call
// zeroes the array's status word and work counters before use; device-side
// errors of this entry point (a bounded wait that expired) are not readable by
// the caller.

#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dkv.h"

namespace {

constexpr size_t kScratchBytes = DKV_NOALLOC_SCRATCH_BYTES;
constexpr size_t kZeroedPrefix = 256;  // status word and work counters
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol, not
// a device address: kernels get the address from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" dkv_status dkv_decode_attn_full_noalloc(const dkv_params* p, const void* q,
                                                   const dkv_kv* K, const dkv_kv* V, void* out,
                                                   int32_t out_dtype, void* stream) {
  const size_t need = dkv_workspace_bytes(p, 0);
  if (need == 0) {
    // Invalid parameters: let the workspace entry point report which one,
    // before it launches anything.
    return dkv_decode_attn_full(p, q, K, V, out, out_dtype, nullptr, 0, stream);
  }
  if (need > kScratchBytes) return DKV_ERR_WORKSPACE;  // beyond the fixed scratch
  void* ws = scratch_on_current_device();
  if (ws == nullptr) return DKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kZeroedPrefix, s) != cudaSuccess) return DKV_ERR_CUDA;
  return dkv_decode_attn_full(p, q, K, V, out, out_dtype, ws, kScratchBytes, stream);
}
