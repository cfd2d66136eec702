// Host-side launch functions of the MoE FFN kernels (internal to libmoeffn).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Router split-K: number of K chunks the router logits are split into.
int route_splits(int T, int H, int E);

// Threads per token row of the rms_norm launches (one CTA per token).
int rmsnorm_threads(int T, int nv);
cudaError_t launch_rmsnorm(const void* x, const void* w, int T, int H, float eps, void* y,
                           void* yq, float* yscale, cudaStream_t st);
cudaError_t launch_router_logits(const void* xhat, const float* wr, int T, int H, int E, int ks,
                                 float* part, cudaStream_t st);
// Logit of (t, e) = sum over z < ks of part[z*zstride + t*tstride + e]
// (+ bias[e]); zstride / tstride 0 mean T*E / E.
cudaError_t launch_topk(const float* part, int ks, const float* bias, int T, int E, int k,
                        int32_t* ids, float* w, float* logits_out, cudaStream_t st,
                        size_t zstride = 0, size_t tstride = 0);
// Router + top-k in one launch for small routers (one CTA per token); used
// when route_small(H, E).
bool route_small(int H, int E);
cudaError_t launch_route_small(const void* xhat, const float* wr, const float* bias, int T,
                               int H, int E, int k, int32_t* ids, float* w, float* logits_out,
                               cudaStream_t st);
// Tensor-core router: split W_r into three transposed bf16 pieces [3E, H]
// and write the one-segment offsets {0, T}.
cudaError_t launch_router_split(const float* wr, int H, int E, int T, void* wt, int32_t* seg,
                                cudaStream_t st);
// The permute kernels also zero nzero ints at zero_buf (counters of later
// kernels in the same forward); zero_buf may be NULL with nzero = 0.
cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets,
                           int32_t* row_src, int32_t* row_of_pair, int* status, cudaStream_t st,
                           int32_t* zero_buf = nullptr, int nzero = 0);
// Permute for any batch: the one-CTA kernel for small batches, else the
// parallel count / scan / scatter kernels, which need
// permute_workspace_bytes() of device scratch (cnt_ws).
size_t permute_workspace_bytes(int T, int E, int k);
cudaError_t launch_permute_any(const int32_t* ids, int T, int E, int k, int32_t* offsets,
                               int32_t* row_src, int32_t* row_of_pair, int32_t* cnt_ws,
                               int* status, cudaStream_t st, int32_t* zero_buf = nullptr,
                               int nzero = 0);
cudaError_t launch_gather_rows(const int32_t* offsets, int E, const int32_t* row_src, int k,
                               int R_max, const void* src, void* dst, int row_bytes,
                               const float* sscale, float* dscale, cudaStream_t st,
                               int scols = 1);  // fp32 scales per row gathered with it
cudaError_t launch_silu_and_mul(const void* h, int R, int I, void* a, cudaStream_t st);
cudaError_t launch_combine(const void* y, bool y_bf16, bool pair_order,
                           const int32_t* row_of_pair, int T, int k, int H, void* out,
                           cudaStream_t st);
cudaError_t launch_quant_rows(const void* x, int64_t rows, int cols, void* q, float* scale,
                              const int32_t* nrows_dev, cudaStream_t st);

// Grouped GEMM, SIMT tile engine (any supported shape).
// mode: 0 FC1 raw, 1 FC1 silu, 2 FC2 (fp32 out), 3 FC2 (bf16 out).  fp8: A/W
// are e4m3 codes with scales.
cudaError_t launch_gemm_simt(int mode, bool fp8, const void* a, const float* a_scale,
                             const void* w, const float* w_scale, const int32_t* offsets,
                             const int32_t* row_src, const float* topk_w, void* c, int E, int K,
                             int I, int N_out, int R_max, cudaStream_t st);

}  // namespace moe
