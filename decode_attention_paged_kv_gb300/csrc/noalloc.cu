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
// zeroes the array's status word and work counters before use.  The status
// word itself cannot be read by the caller, so a device-side error of the
// call (a bounded wait that expired) is made visible in its result instead:
// a last small kernel sets every element of `out` to NaN when the status word
// is not zero.
//
// The address is cached per device together with the context it was looked
// up in; a call made under another context (after a device reset, or with a
// context of the caller's own current) looks it up again.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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
struct ScratchSlot {
  CUcontext ctx;  // the context the address belongs to
  void* ptr;
};
ScratchSlot g_slot[kMaxDevices] = {};

// cuCtxGetCurrent through the runtime's driver entry point (no link to libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

// Device address of g_scratch on the current device, looked up once per
// (device, context).  The lookup also makes the runtime's context current if
// none was, so the context is read again after it.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return nullptr;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (ctx == nullptr || g_slot[dev].ptr == nullptr || g_slot[dev].ctx != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
    g_slot[dev].ctx = ctx;
    g_slot[dev].ptr = ptr;
  }
  return g_slot[dev].ptr;
}

// After the call: NaN into every element of out [B, Hq, d] when the status
// word (the scratch's first 4 bytes) records a device-side error.
__global__ void poison_on_error_kernel(const unsigned int* status, void* out, int out_dtype,
                                       int Hq, int d, long long sb, long long sh) {
  if (*status == 0u) return;
  const int b = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const long long row = b * sb + h * sh;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    if (out_dtype == DKV_FP32)
      static_cast<float*>(out)[row + i] = __int_as_float(0x7fc00000);
    else if (out_dtype == DKV_FP16)
      static_cast<__half*>(out)[row + i] = __ushort_as_half(0x7e00);
    else
      static_cast<__nv_bfloat16*>(out)[row + i] = __ushort_as_bfloat16(0x7fc0);
  }
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
  const dkv_status st = dkv_decode_attn_full(p, q, K, V, out, out_dtype, ws, kScratchBytes, stream);
  if (st != DKV_OK) return st;
  poison_on_error_kernel<<<p->batch * p->num_q_heads, 128, 0, s>>>(
      static_cast<const unsigned int*>(ws), out, out_dtype, p->num_q_heads, p->head_dim,
      p->o_stride_b, p->o_stride_h);
  return cudaGetLastError() == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}
