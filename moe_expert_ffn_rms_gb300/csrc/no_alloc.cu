// moe_ffn_forward_static_ws: the whole forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to call cudaMalloc: a plug-in running inside a
// host program that owns the device-memory budget and refuses allocations
// from its plug-ins, code on a latency-critical path that must not pay for
// an allocation (cudaMalloc can synchronise the device), or plain C / FFI
// code that holds only the input and output buffers it was handed.  For
// them this entry point runs moe_ffn_forward with its scratch in a
// file-scope device array of fixed size instead of a caller workspace.
#include <stdio.h>

#include <mutex>

#include "api_internal.h"
#include "common.cuh"

namespace {

// 32 MiB: enough for every decode-sized shape of the reference workloads
// (the largest, T=64 H=7168 E=256 top_k=8 I=2048, needs about 26 MiB).
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;

// The scratch itself.  Every device on which the library's device code is
// loaded holds these 32 MiB until the process exits.  In host code the name
// is only a host-side stand-in; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device, looked up once
// per device with that device current.
moe_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    return moe::api_fail(MOE_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) return moe::api_fail(MOE_ERR_UNSUPPORTED_DEVICE, "device index out of range");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
      return moe::api_fail(MOE_ERR_CUDA, msg);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_ffn_forward_static_ws(
    const moe_shape* shape, const void* x, const void* norm_w, const float* router_w,
    const float* router_logits, const float* router_bias, const void* w13, const void* w2,
    const float* w13_scale, const float* w2_scale, void* out, int32_t* topk_ids_out,
    float* topk_w_out, moe_stream_t stream) {
  moe_status rc = moe::api_check_shape(shape);
  if (rc != MOE_OK) return rc;
  const size_t need = moe_ffn_workspace_size(shape);
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "this shape needs %zu bytes of scratch; the static scratch of "
             "moe_ffn_forward_static_ws holds %zu bytes (use moe_ffn_forward with a workspace)",
             need, kStaticScratchBytes);
    return moe::api_fail(MOE_ERR_WORKSPACE_TOO_SMALL, msg);
  }
  if ((rc = moe_check_device()) != MOE_OK) return rc;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != MOE_OK) return rc;
  // Nothing in the forward's scratch has to start at zero: every buffer in it
  // is written before it is read within one call.
  return moe_ffn_forward(shape, x, norm_w, router_w, router_logits, router_bias, w13, w2,
                         w13_scale, w2_scale, out, topk_ids_out, topk_w_out, scratch,
                         kStaticScratchBytes, stream);
}
