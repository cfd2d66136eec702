// Shared device helpers for the MoE expert FFN kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <float.h>
#include <math.h>
#include <stdint.h>

#include "../../include/moe_ffn.h"

typedef __nv_bfloat16 bf16;

#define MOE_DEV __device__ __forceinline__

// Largest supported expert count / top_k (shared-memory tables are sized by them).
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;

// ------------------------------------------------ programmatic dependent launch --
// Every kernel of the path is launched with programmatic stream serialisation:
// it lets the next kernel in the stream start (prologue only) once this one
// calls pdl_trigger(), and waits in pdl_wait() until the previous kernel has
// completed and its writes are visible.  Each kernel calls pdl_wait() before
// its first global-memory access.  Both are no-ops for a normal launch.
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- status --
// The device status word lives in api.cu; kernels receive its address.
MOE_DEV void flag_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ conversions --
MOE_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

MOE_DEV void unpack8_bf16(const uint4& u, float* f) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

MOE_DEV uint32_t pack2_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // RNE, a in the low half
  return *reinterpret_cast<uint32_t*>(&h);
}

MOE_DEV float bf16_round_f(float a) { return __bfloat162float(__float2bfloat16_rn(a)); }

// E4M3 code -> float (exact).
MOE_DEV float e4m3_to_f(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

// float -> E4M3 code, round to nearest even, saturating to +-448.
MOE_DEV uint8_t f_to_e4m3(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// silu(z) = z / (1 + exp(-z)), fp32.
MOE_DEV float silu_f(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------- top-k --
// Top-k of one token by one warp: lane l holds the logits of experts l, l+32,
// ... in v (-FLT_MAX past E).  The k winners are taken one at a time by a warp
// arg-max (larger logit first, lower index on ties); the weights are the
// softmax over the selected logits (= full softmax renormalised).  Lane 0
// writes ids[0..k) and w[0..k).  A NaN logit ranks as -inf (below every
// finite logit, ties to the lower index as usual), so each of the k slots
// always receives a distinct expert in [0, E) (k <= E); when every selected
// logit is -inf the softmax is undefined and the token's weights are 0.
// PER values per lane (PER >= ceil(E / 32); a kernel instance for the
// smallest PER that holds E keeps the scans short), at most kTopkPer.
constexpr int kTopkPer = kMaxExperts / 32;

template <int PER>
MOE_DEV void warp_topk(const float (&v)[PER], int E, int k, int lane, int32_t* ids,
                       float* w) {
  unsigned taken = 0;
  float sel_v[kMaxTopK];
  int sel_e[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j >= k) break;
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      const float vi = (v[i] != v[i]) ? -INFINITY : v[i];  // NaN ranks as -inf
      if (e < E && !(taken & (1u << i)) && (vi > bv || (vi == bv && e < be))) {
        bv = vi;
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    sel_v[j] = bv;
    sel_e[j] = be;
  }
  if (lane == 0) {
    const float m = sel_v[0];
    const bool finite_max = m > -INFINITY;
    float p[kMaxTopK];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= k) break;
      p[j] = finite_max ? expf(sel_v[j] - m) : 0.f;
      s += p[j];
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= k) break;
      ids[j] = sel_e[j];
      w[j] = finite_max ? p[j] / s : 0.f;
    }
  }
}

// Host: programmatic dependent launch is used unless the environment sets
// MOE_PDL=0 or the calling thread is inside a PdlOff scope with off = true.
bool pdl_enabled();

// Host-side count of the kernels the library has enqueued (every launch site
// calls count_launch() after a successful launch).
void count_launch();
long long launch_count();

class PdlOff {
 public:
  explicit PdlOff(bool off = true);
  ~PdlOff();
  PdlOff(const PdlOff&) = delete;
  PdlOff& operator=(const PdlOff&) = delete;

 private:
  bool prev_;
};

// Host: launch `kern` on `st`, with programmatic stream serialisation when
// pdl_enabled().

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

// ------------------------------------------------------------- reductions --
MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

MOE_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum / max for blockDim.x <= 1024 (a multiple of 32); every
// thread gets the result.  `red` is 32 floats of shared memory.
MOE_DEV float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : 0.0f;
  return warp_sum(r);
}

MOE_DEV float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : 0.0f;
  return warp_max(r);
}
