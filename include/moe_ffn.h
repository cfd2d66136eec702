/*
 * moe_ffn.h -- C ABI of libmoeffn.so, the MoE expert FFN forward for one
 * NVIDIA GB300 (sm_103a).
 *
 * The path (per token t):
 *   x_hat = rms_norm(x, norm_w)                      moe_rmsnorm
 *   logits = x_hat W_r (+ b); top-k of softmax,       moe_route_topk
 *            renormalised
 *   rows grouped by expert                            moe_permute
 *   a = silu(x_hat W_gate^T) * (x_hat W_up^T)         moe_grouped_gemm (FC1)
 *   y = w_tj * (a W2^T)                               moe_grouped_gemm (FC2)
 *   out_t = sum_j y_tj                                moe_combine
 * moe_ffn_forward runs all of it; the step entry points run one step each.
 *
 * Sources (web pages, by title and section):
 *   [V100]  Qiita, "running the latest vLLM on a Tesla V100": section
 *           "2nd wall" names rms_norm and silu_and_mul as the custom ops of
 *           the FFN; section "rewrite on torch::stable::Tensor" defines
 *           rms_norm as pow -> mean -> rsqrt -> mul.
 *   [RUBIN] "vLLM Support for NVIDIA Vera Rubin NVL72", section "Locality
 *           domain": at small token counts the MoE forward is FC1 then FC2
 *           over expert weights streamed from HBM, split by columns (split-N).
 *   [SM]    "vLLM's adaptation to different GPU SM architectures", sections
 *           3.1/3.2 (W8A8 scaled GEMM, FP8 E4M3, output-first signature
 *           cutlass_scaled_mm(c, ...)), 4.3 (experts take hidden_states,
 *           w1, w2; small batches want few launches), 4.4 and the MoE GEMM
 *           support table (FP8 block-wise and NVFP4 expert weights), and the
 *           Hopper data-flow figure (block-wise FP8 dequantised inside the
 *           GEMM loop).
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, unless a
 *     comment says "host".  The library never allocates or frees device
 *     memory; scratch comes from the caller's `workspace`.
 *   - Layouts are row-major with the last index contiguous.  bf16 is
 *     __nv_bfloat16 (2 bytes), e4m3 is OCP FP8 E4M3FN (1 byte).
 *   - Device pointers must be 16-byte aligned (weight scales included); row
 *     lengths must keep every row 16-byte aligned (H and I multiples of 64).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work on it and never synchronise the host.
 *   - Inputs are read only.  A return of MOE_OK means the work was enqueued;
 *     a kernel fault surfaces as MOE_ERR_CUDA at a later call or at the
 *     caller's synchronisation.  On any other status nothing was enqueued
 *     and moe_last_error() describes the problem (thread-local string).
 *   - Device-side waits are bounded; a wait that runs out records
 *     MOE_ERR_TIMEOUT in the library's device status word, which
 *     moe_device_status() reads.
 */
#ifndef MOE_FFN_H_
#define MOE_FFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, misalignment, bad value */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* shape outside the supported envelope */
  MOE_ERR_UNSUPPORTED_DEVICE = 3,  /* current device is not compute capability 10.3 */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes < the size query's answer */
  MOE_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 6              /* a bounded device-side wait ran out */
} moe_status;

/* Expert weight format.  MOE_W_NVFP4 weights go through moe_ffn_forward_nvfp4
 * (packed codes plus two scale arrays); the other entry points take BF16,
 * FP8_E4M3 (per-output-channel weight scales, per-token activation scales)
 * or FP8_BLOCK (block-wise FP8: one weight scale per 128 x 128 tile, one
 * activation scale per token and 128-element group; [SM] support table,
 * "FP8 block-wise" MoE GEMMs, and the Hopper data-flow figure, "block-wise
 * FP8 dequant inside GEMM loop").  FP8_BLOCK needs H % 256 == 0,
 * I % 128 == 0 and H, I <= 8192. */
typedef enum {
  MOE_W_BF16 = 0,
  MOE_W_FP8_E4M3 = 1,
  MOE_W_NVFP4 = 2,
  MOE_W_FP8_BLOCK = 3
} moe_wdtype;

/* Which step of the grouped GEMM moe_grouped_gemm runs. */
typedef enum {
  MOE_GEMM_FC1_RAW = 0,   /* c bf16 [R, 2I] = a W13^T                          */
  MOE_GEMM_FC1_SILU = 1,  /* c bf16 [R, I]  = silu(a W_gate^T) * (a W_up^T)   */
  MOE_GEMM_FC2 = 2,       /* c fp32 [R, H]  = topk_w[row] * (a W2^T)           */
  MOE_GEMM_FC2_BF16 = 3   /* c bf16 [R, H]: row r stored at row row_src[r]      */
} moe_gemm_mode;

/* Engine used for the grouped GEMMs.  AUTO picks by the host-known average
 * rows per expert (T*top_k/E): the weight-streaming decode engine for small
 * batches, the tile engine for large ones. */
typedef enum { MOE_ENGINE_AUTO = 0, MOE_ENGINE_DECODE = 1, MOE_ENGINE_PREFILL = 2 } moe_engine;

/* Problem size.  T tokens, H hidden, E experts, I intermediate, top_k <= 8. */
typedef struct {
  int32_t T, H, E, I, top_k;
  float eps;        /* rms_norm epsilon (1e-6 in the reference workloads) */
  int32_t wdtype;   /* moe_wdtype of w13 / w2 */
  int32_t engine;   /* moe_engine */
} moe_shape;

typedef void* moe_stream_t; /* cudaStream_t */

/* ---------------------------------------------------------------- misc -- */

/* MOE_ABI_VERSION of the built library. */
int32_t moe_abi_version(void);

/* Number of kernels the library has enqueued in this process so far, on every
 * device and stream (memsets excluded).  A host-side counter for launch
 * accounting (e.g. kernels per forward); no device synchronisation.  The
 * pages describe no such call; it has no counterpart there. */
int64_t moe_launch_count(void);

/* Thread-local description of the last non-MOE_OK status on this thread
 * (empty string if none).  Never NULL; valid until the next call. */
const char* moe_last_error(void);

/* Static name of a status code ("MOE_OK", ...). */
const char* moe_status_string(moe_status s);

/* Checks that the current CUDA device is compute capability 10.3 (GB300)
 * and caches its SM count.  Every compute entry point calls it. */
moe_status moe_check_device(void);

/* Reads (and if clear != 0, resets) the library's device status word:
 * MOE_OK, or MOE_ERR_TIMEOUT after a bounded wait ran out, or
 * MOE_ERR_INVALID_ARG after a kernel saw an out-of-range expert id.
 * `status_out` is a HOST pointer.  Synchronises the device. */
moe_status moe_device_status(int32_t* status_out, int32_t clear);

/* Self-test of the library's bounded device waits (failure detection; not a
 * step of the method).  Enqueues one kernel that waits on an mbarrier no
 * thread arrives on, gives up after limit_cycles SM cycles (0 < limit <=
 * 2^32), records MOE_ERR_TIMEOUT in the device status word and returns, so
 * the CUDA context stays usable.  Read the result with moe_device_status(). */
moe_status moe_selftest_wait_timeout(int64_t limit_cycles, moe_stream_t stream);

/* ------------------------------------------------------- whole forward -- */

/* Device workspace bytes moe_ffn_forward / moe_ffn_forward_routed need for
 * this shape (0 and an error message when the shape is invalid). */
size_t moe_ffn_workspace_size(const moe_shape* shape);

/* The whole MoE expert FFN forward:
 *   out = combine(FC2(silu_and_mul(FC1(permute(rms_norm(x))))))
 * with routing from the router ([SM] 4.3: experts(hidden_states, w1, w2);
 * [RUBIN] Locality domain: FC1 then FC2).
 *   shape       host pointer; T, H, E, I, top_k, eps, wdtype, engine.
 *   x           bf16 [T, H]          tokens.
 *   norm_w      bf16 [H]             rms_norm weight.
 *   router_w    fp32 [H, E]          router weight; or NULL when
 *   router_logits fp32 [T, E]        ... precomputed logits are given
 *                                    instead (exactly one of the two).
 *   router_bias fp32 [E] or NULL     added to the logits before softmax.
 *   w13         [E, 2I, H]           bf16, or e4m3 codes when wdtype is
 *                                    FP8 (rows 0..I-1 gate, I..2I-1 up).
 *   w2          [E, H, I]            bf16 or e4m3 codes.
 *   w13_scale   fp32 [E, 2I] / NULL  per-output-channel dequant scale (FP8);
 *                                    fp32 [E, 2I/128, H/128] tile scales
 *                                    (FP8_BLOCK).
 *   w2_scale    fp32 [E, H]  / NULL  ditto for w2 (FP8_BLOCK: [E, H/128, I/128]).
 *   out         bf16 [T, H]          result.
 *   topk_ids_out int32 [T, top_k] / NULL  the routing decision, descending
 *   topk_w_out  fp32 [T, top_k]  / NULL   weight, ties to the lower index.
 *   workspace   >= moe_ffn_workspace_size(shape) bytes, 256-byte aligned;
 *               must not be used by other work while this call runs.
 * FP8 (per channel): x_hat is quantised per token, the bf16 intermediate per
 * row; FC1/FC2 are E4M3 x E4M3 products accumulated in fp32 and scaled by
 * s_x[r] * s_w[e, n].  FP8_BLOCK: x_hat and the bf16 intermediate are
 * quantised per row and 128-element group; each 128-wide K group of a
 * product is accumulated on its own and scaled by s_a[r, g] * s_w[e, n/128, g]
 * before the groups are added in K order (decode engine: one persistent
 * launch for FC1 and FC2; prefill engine: FC1 tiles, the group quantisation
 * of the intermediate, FC2 tiles).
 * Errors: INVALID_ARG (null/misaligned/both or neither router input),
 * UNSUPPORTED_SHAPE (H or I not a multiple of 64, top_k > 8 or > E,
 * E > 256, the FP8_BLOCK limits above), WORKSPACE_TOO_SMALL,
 * UNSUPPORTED_DEVICE, CUDA. */
moe_status moe_ffn_forward(const moe_shape* shape, const void* x, const void* norm_w,
                           const float* router_w, const float* router_logits,
                           const float* router_bias, const void* w13, const void* w2,
                           const float* w13_scale, const float* w2_scale, void* out,
                           int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream);

/* As moe_ffn_forward, with the routing given by the caller (vLLM's
 * fused-experts form): topk_ids int32 [T, top_k] (distinct experts per
 * token, each in [0, E)) and topk_w fp32 [T, top_k].  An id outside [0, E)
 * is skipped and flagged in the device status word. */
moe_status moe_ffn_forward_routed(const moe_shape* shape, const void* x, const void* norm_w,
                                  const int32_t* topk_ids, const float* topk_w,
                                  const void* w13, const void* w2, const float* w13_scale,
                                  const float* w2_scale, void* out, void* workspace,
                                  size_t workspace_bytes, moe_stream_t stream);

/* moe_ffn_forward without a caller workspace, for callers that cannot
 * allocate device memory: a plug-in inside a host program that owns the
 * device-memory budget, a latency-critical path that must not pay for an
 * allocation, or plain C / FFI code that holds only the buffers it was
 * handed.  The pages describe no such entry point; it has no counterpart
 * there.
 *   Arguments and results are those of moe_ffn_forward, minus workspace.
 *   Scratch: a file-scope device array of 32 MiB inside the library, held on
 *   every device where the library's device code is loaded until the
 *   process exits.  Shapes whose moe_ffn_workspace_size() exceeds 32 MiB
 *   (large prefill batches) are rejected with MOE_ERR_WORKSPACE_TOO_SMALL
 *   and nothing is enqueued.  No call allocates or frees device memory.
 *   Set-up: the first call on a device (with that device current) looks up
 *   the array's device address; make that first call before any stream
 *   capture.
 *   The address belongs to the device's primary context (the one the CUDA
 *   runtime uses) and is kept for the life of the process: after
 *   cudaDeviceReset(), or from a different driver-API context on the same
 *   device, do not call this entry point.
 *   All calls on a device share the one array and it keeps the last call's
 *   contents (nothing in it needs to start at zero).  Calls whose work
 *   overlaps on the GPU (other streams, other host threads) race on it:
 *   serialise them, e.g. on one stream. */
moe_status moe_ffn_forward_static_ws(const moe_shape* shape, const void* x, const void* norm_w,
                                     const float* router_w, const float* router_logits,
                                     const float* router_bias, const void* w13, const void* w2,
                                     const float* w13_scale, const float* w2_scale, void* out,
                                     int32_t* topk_ids_out, float* topk_w_out,
                                     moe_stream_t stream);

/* The forward with NVFP4 expert weights and bf16 activations (W4A16).
 * [SM] section 4.4 and its support table list NVFP4 MoE expert weights for
 * Blackwell without defining the format; the library uses the public NVFP4
 * layout: per expert matrix W [N, K] (w13: N = 2I, K = H; w2: N = H, K = I),
 *   codes  uint8 [E, N, K/2]  E2M1 (1 sign, 2 exponent bits with bias 1,
 *                             1 mantissa bit), element 2i in the low nibble
 *   sb     uint8 [E, N, K/16] E4M3 scale of each block of 16 K elements
 *   sg     fp32  [E]          scale of each expert matrix
 *   w[n, k] = e2m1(code) * e4m3(sb[n, k/16]) * sg,
 * as written by moe_quantize_nvfp4.  Everything else (routing, outputs,
 * workspace from moe_ffn_workspace_size with shape->wdtype = MOE_W_NVFP4) is
 * as moe_ffn_forward.  Each code times its block scale is exact in fp16 and
 * bf16 activations are exact in fp16, so the GEMMs are those of the bf16
 * forward on the dequantised weights, accumulated in fp32; the intermediate
 * is rounded to bf16 as in the bf16 forward.
 * Errors: as moe_ffn_forward; UNSUPPORTED_SHAPE unless H and I are
 * multiples of 256. */
moe_status moe_ffn_forward_nvfp4(const moe_shape* shape, const void* x, const void* norm_w,
                                 const float* router_w, const float* router_logits,
                                 const float* router_bias, const uint8_t* w13, const uint8_t* w13_sb,
                                 const float* w13_sg, const uint8_t* w2, const uint8_t* w2_sb,
                                 const float* w2_sg, void* out, int32_t* topk_ids_out,
                                 float* topk_w_out, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream);

/* ------------------------------------------------------------ the steps -- */

/* rms_norm ([V100] "rewrite on torch::stable::Tensor"):
 *   y[t, i] = bf16( x[t, i] / sqrt(mean_i(x[t, :]^2) + eps) * w[i] )
 * fp32 arithmetic.  x bf16 [T, H], w bf16 [H], y bf16 [T, H].
 * If yq != NULL also writes the per-token E4M3 quantisation of y:
 *   yscale[t] = max|y[t, :]| / 448 (1 when the row is zero),
 *   yq[t, i] = e4m3_satfinite_rne(y[t, i] / yscale[t])   (e4m3 [T, H]).
 * yq and yscale are both NULL or both given.  H % 8 == 0. */
moe_status moe_rmsnorm(const void* x, const void* w, int32_t T, int32_t H, float eps, void* y,
                       void* yq, float* yscale, moe_stream_t stream);

/* Device workspace bytes moe_route_topk needs (router partial sums). */
size_t moe_route_workspace_size(int32_t T, int32_t H, int32_t E);

/* Router softmax and renormalised top-k.  [RUBIN] "Hardware grows..."
 * names the router softmax (exp-bound); the pages are silent on the router
 * layer, the selection rule and the renormalisation, so the plain reading is
 * used: a linear router over x_hat, softmax over all E, the k largest
 * probabilities (ties to the lower expert index), renormalised over the k.
 * Errors: MOE_ERR_INVALID_ARG for NULL or misaligned pointers, or when both
 * or neither of router_w and logits_in are given; UNSUPPORTED_SHAPE outside
 * the limits below.  A NaN logit ranks as -inf (below every finite logit,
 * ties to the lower index), so every slot holds a distinct expert in [0, E);
 * a token whose selected logits are all -inf gets weights 0.
 *   logits = xhat W_r + b   (fp32; skipped when logits_in != NULL, then
 *                            logits = logits_in + b)
 *   ids[t, :]  = the top_k experts by logit, descending, ties to the lower
 *                expert index (softmax is increasing in the logit, so this
 *                is the top-k of the probabilities);
 *   w[t, j]    = exp(l_j - l_max) / sum_j' exp(l_j' - l_max) over the
 *                selected experts (= softmax, then renormalised).
 *   xhat bf16 [T, H]; router_w fp32 [H, E]; router_bias fp32 [E] or NULL;
 *   logits_in fp32 [T, E] or NULL; ids int32 [T, k]; weights fp32 [T, k];
 *   logits_out fp32 [T, E] or NULL (receives logits incl. bias).
 *   E <= 256, k <= min(E, 8). */
moe_status moe_route_topk(const void* xhat, const float* router_w, const float* router_bias,
                          const float* logits_in, int32_t T, int32_t H, int32_t E, int32_t k,
                          int32_t* ids, float* weights, float* logits_out, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream);

/* Device workspace bytes moe_permute needs (0 for small batches, which use a
 * single-CTA sort; larger ones use a parallel count / scan / scatter). */
size_t moe_permute_workspace_size(int32_t T, int32_t E, int32_t k);

/* Token -> expert grouping (stable counting sort of the T*k (t, j) pairs by
 * expert; rows ordered by expert, then token).  [SM] 4.2/4.3 describe grouped
 * GEMM MoE backends that consume expert-grouped rows; the pages are silent on
 * the grouping itself, so the plain reading (a stable sort by expert) is used.
 * Errors: MOE_ERR_INVALID_ARG for NULL or misaligned pointers or a workspace
 * below moe_permute_workspace_size(); ids outside [0, E) are skipped on the
 * device and flagged (MOE_ERR_INVALID_ARG in the device status word).
 *   ids int32 [T, k]            routing (each row: distinct experts)
 *   offsets int32 [E + 1]       expert e owns rows offsets[e] .. offsets[e+1]-1
 *   row_src int32 [T*k]         row r holds pair t*k + j
 *   row_of_pair int32 [T*k]     inverse: pair t*k + j sits in row r
 *   xhat / xp                   optional gather xp[r, :] = xhat[row_src[r]/k, :]
 *                               (rows of row_bytes bytes, multiple of 16);
 *                               both NULL to skip.
 *   xscale / xp_scale           optional fp32 per-row scale gather (FP8), or NULL.
 *   workspace                   >= moe_permute_workspace_size(T, E, k) bytes
 *                               (may be NULL when that is 0).
 * E <= 256.  Ids outside [0, E) are skipped and flagged. */
moe_status moe_permute(const int32_t* ids, int32_t T, int32_t E, int32_t k, int32_t* offsets,
                       int32_t* row_src, int32_t* row_of_pair, const void* xhat, void* xp,
                       int32_t row_bytes, const float* xscale, float* xp_scale, void* workspace,
                       size_t workspace_bytes, moe_stream_t stream);

/* Grouped GEMM over the expert segments given by offsets ([RUBIN] FC1/FC2,
 * [SM] 3.1 scaled GEMM).  For each expert e and each row r in
 * offsets[e] .. offsets[e+1]-1:
 *   FC1_RAW:  c[r, n] = bf16( sum_h a[r, h] * w[e, n, h] )       n < 2I, K = H
 *   FC1_SILU: c[r, n] = bf16( silu(g) * u ),  g = sum_h a[r,h] w[e,n,h],
 *                                             u = sum_h a[r,h] w[e,I+n,h]  n < I
 *   FC2:      c[r, n] = topk_w[row_src[r]] * sum_i a[r, i] * w[e, n, i]   n < H
 *             (fp32 output; topk_w/row_src NULL -> weight 1)
 *   FC2_BF16: the same rounded to bf16 and written to row row_src[r] of c,
 *             i.e. back in (token, slot) order (row r when row_src is NULL)
 * a: bf16 [R, K] (or e4m3 with a_scale fp32 [R] when shape->wdtype is FP8,
 * then w is e4m3 with w_scale fp32 [E, N]); products accumulate in fp32 and
 * are scaled by a_scale[r] * w_scale[e, n].  R = offsets[E] <= T*top_k. */
moe_status moe_grouped_gemm(const moe_shape* shape, int32_t mode, const void* a,
                            const float* a_scale, const void* w, const float* w_scale,
                            const int32_t* offsets, const int32_t* row_src, const float* topk_w,
                            void* c, moe_stream_t stream);

/* Device workspace bytes moe_grouped_ffn needs (0 when the shape is invalid). */
size_t moe_grouped_ffn_workspace_size(const moe_shape* shape);

/* The expert FFN of the grouped rows in one call ([RUBIN] Locality domain:
 * FC1 then FC2):  act = FC1_SILU(xp), then y = FC2_BF16(act) -- exactly the
 * two moe_grouped_gemm steps the forward runs (same arguments and layouts:
 * xp [R, H] (+ xp_scale [R] for FP8), act bf16 [R, I], y bf16 [R, H] in
 * (token, slot) order, R = T * top_k).  On the decode engine with bf16
 * weights both GEMMs run in one persistent launch whose FC2 units wait per
 * expert for that expert's FC1 units.  FP8_BLOCK (one launch on the decode
 * engine, three on the prefill engine): xp
 * e4m3 [R, H] with xp_scale fp32 [R, H/128] (one scale per row and group,
 * as moe_quantize_fp8_blocks with block_rows = 1 writes them), act e4m3
 * [R, I] receives the quantised intermediate (its group scales stay in the
 * workspace).  workspace >= moe_grouped_ffn_workspace_size(shape) bytes,
 * 256-byte aligned. */
moe_status moe_grouped_ffn(const moe_shape* shape, const void* xp, const float* xp_scale,
                           const void* w13, const float* w13_scale, const void* w2,
                           const float* w2_scale, const int32_t* offsets, const int32_t* row_src,
                           const float* topk_w, void* act, void* y, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream);

/* The NVFP4 expert FFN of the grouped rows (the FFN step of
 * moe_ffn_forward_nvfp4): act = FC1_SILU(xp), y = FC2_BF16(act) with NVFP4
 * weights (codes, block and matrix scales as moe_ffn_forward_nvfp4 takes
 * them), in one persistent launch.  xp fp16 [R, H] (the gathered x_hat rows;
 * bf16 values are exact in fp16), act fp16 [R, I] (bf16-rounded values),
 * y bf16 [R, H] in (token, slot) order.  shape->wdtype = MOE_W_NVFP4;
 * workspace >= moe_grouped_ffn_workspace_size(shape) bytes, 256-byte aligned.
 * UNSUPPORTED_SHAPE unless H and I are multiples of 256. */
moe_status moe_grouped_ffn_nvfp4(const moe_shape* shape, const void* xp, const uint8_t* w13,
                                 const uint8_t* w13_sb, const float* w13_sg, const uint8_t* w2,
                                 const uint8_t* w2_sb, const float* w2_sg, const int32_t* offsets,
                                 const int32_t* row_src, const float* topk_w, void* act, void* y,
                                 void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* silu_and_mul ([V100] "2nd wall"): a[r, i] = bf16( silu(h[r, i]) * h[r, I+i] ),
 * silu(z) = z / (1 + exp(-z)); h bf16 [R, 2I], a bf16 [R, I]; I % 8 == 0. */
moe_status moe_silu_and_mul(const void* h, int32_t R, int32_t I, void* a, moe_stream_t stream);

/* Weighted combine: out[t, :] = bf16( sum_{j=0..k-1} y_{t,j} ) summed in fp32
 * in j order (the routing weight is already in y).  The pages are silent on
 * the combine; the plain reading is used (a weighted sum of the token's k
 * expert outputs, no residual and no shared expert, one bf16 rounding).
 * Errors: MOE_ERR_INVALID_ARG for NULL or misaligned pointers or H % 8 != 0.
 * y_{t,j} is row
 * row_of_pair[t*k+j] of y (y_pair_order = 0: rows in expert order, as
 * MOE_GEMM_FC2 writes them) or row t*k+j (y_pair_order = 1: rows in
 * (token, slot) order, as MOE_GEMM_FC2_BF16 writes them).  Pairs whose
 * row_of_pair is -1 are skipped.  y [T*k, H], fp32 (y_bf16 = 0) or bf16
 * (y_bf16 = 1); out bf16 [T, H]; H % 8 == 0. */
moe_status moe_combine(const void* y, int32_t y_bf16, int32_t y_pair_order,
                       const int32_t* row_of_pair, int32_t T, int32_t k, int32_t H, void* out,
                       moe_stream_t stream);

/* Row-wise dynamic E4M3 quantisation ([SM] 3.2, W8A8):
 *   scale[r] = max|x[r, :]| / 448 (1 for a zero row), fp32;
 *   q[r, c] = e4m3_satfinite_rne( x[r, c] / scale[r] ) (IEEE fp32 divide).
 * Used per output channel for weights (rows = E*N) and per token for
 * activations.  x bf16 [rows, cols], q e4m3 [rows, cols], cols % 16 == 0. */
moe_status moe_quantize_fp8_rows(const void* x, int64_t rows, int32_t cols, void* q,
                                 float* scale, moe_stream_t stream);

/* NVFP4 quantisation of M matrices w bf16 [M, N, K] along K (the layout
 * described at moe_ffn_forward_nvfp4), each step rounded to fp32:
 *   sg[m] = max|w[m]| / (448 * 6)   (1 for an all-zero matrix)
 *   sb    = e4m3_satfinite_rne( max|block of 16| / (6 * sg) )
 *   code  = e2m1_satfinite_rne( w / (e4m3(sb) * sg) )   (0 where sb is 0)
 * q uint8 [M, N, K/2], sb uint8 [M, N, K/16], sg fp32 [M]; K % 16 == 0;
 * w, q 16-byte aligned; sb, sg 4-byte aligned. */
moe_status moe_quantize_nvfp4(const void* w, int32_t M, int32_t N, int32_t K, uint8_t* q,
                              uint8_t* sb, float* sg, moe_stream_t stream);

/* Block-wise E4M3 quantisation (the FP8_BLOCK format) of x bf16 [N, K]:
 * tiles of block_rows x 128 elements (block_rows = 128 for weights: pass
 * N = E * rows per expert, whose row counts are multiples of 128; 1 for
 * activation rows), each with
 *   scale[N / block_rows, K / 128] = max|tile| / 448 (1 for a zero tile), fp32;
 *   q[n, k] = e4m3_satfinite_rne( x[n, k] / scale of its tile ) (IEEE fp32 divide).
 * q e4m3 [N, K]; K % 128 == 0, N % block_rows == 0; x, q 16-byte aligned,
 * scale 4-byte aligned. */
moe_status moe_quantize_fp8_blocks(const void* x, int32_t N, int32_t K, int32_t block_rows,
                                   uint8_t* q, float* scale, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H_ */
