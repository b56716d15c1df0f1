// mf_attn_bwd_noalloc: the attention backward for callers that cannot
// allocate device memory.
//
// mf_attn_bwd needs a scratch workspace (the float32 row dots D, the float32
// dQ accumulator and fp16 rotated copies of Q and K) that the caller normally
// allocates.  Some callers cannot allocate at the point where they run the
// backward: for example an engine plugin whose execute step is forbidden to
// allocate, a runtime that hands all device memory to its own pool at
// start-up and has none left to give, or a latency-critical loop that must
// not call cudaMalloc because it can synchronize the device.  For them this
// file keeps a fixed scratch array in device memory, reserved when the
// library's GPU code is loaded and held by every GPU that loads it until the
// process exits.
#include <atomic>

#include "../../include/mf.h"
#include "common.cuh"

namespace {

// Scratch shared by every mf_attn_bwd_noalloc call on a device.
constexpr size_t kScratchBytes = static_cast<size_t>(MF_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_bwd_scratch on the current device.  The host-side name
// of the array is only a stand-in, so the address is looked up with the
// device current.  A call outside stream capture looks it up every time (a
// device reset reloads the module, and the array may then sit elsewhere) and
// caches it per device; a call made while `stream` is capturing takes the
// cached address, or looks it up if the device has none yet.
mf_status scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MF_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return MF_ERR_CUDA;
  void* p = cap == cudaStreamCaptureStatusNone ? nullptr : g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) return MF_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return MF_OK;
}

}  // namespace

extern "C" mf_status mf_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                         const float* lse, const void* dout, const mf_plan* plan,
                                         int32_t heads, int32_t head_dim, float softmax_scale, void* dq,
                                         void* dk, void* dv, void* stream) {
  if (plan == nullptr || heads < 1) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  if (plan->total_tokens < 0) return MF_ERR_INVALID_ARG;
  size_t need = 0;
  mf_status st = mf_attn_bwd_workspace_size(plan->total_tokens, heads, head_dim, &need);
  if (st != MF_OK) return st;
  if (need > kScratchBytes) return MF_ERR_UNSUPPORTED;  // pack too large for the fixed scratch
  void* scratch = nullptr;
  if ((st = scratch_address(static_cast<cudaStream_t>(stream), &scratch)) != MF_OK) return st;
  // The backward's first kernel overwrites D and the rotated copies and zeroes
  // the accumulator, so whatever an earlier call left in the array does not
  // leak into this one.
  return mf_attn_bwd(q, k, v, o, lse, dout, plan, heads, head_dim, softmax_scale, scratch, kScratchBytes, dq,
                     dk, dv, stream);
}
