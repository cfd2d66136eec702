// Tensor-core (tcgen05 / TMEM / TMA) grouped GEMM engines (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Per-device one-time set-up (driver entry points, kernel attributes).
void engine_init_device();

// Launches the tcgen05 grouped GEMM for one step, or returns
// cudaErrorNotSupported (nothing enqueued) when the shape is outside what
// the tensor-core engines cover; the caller then uses the SIMT engine.
//   mode   0 FC1 raw, 1 FC1 + silu_and_mul, 2 FC2 x routing weight (fp32 out),
//          3 the same with bf16 out
//   decode true: weights are the 128-row MMA operand and the expert's
//          tokens the narrow one (small batches); false: token tiles.
//   sched  token tiles only: NULL (static round-robin over the CTAs), or one
//          int that is zero when the kernel starts, from which the CTAs claim
//          work units in order (so CTAs working on units that share a weight
//          tile run close together in time and the tile is served by L2).
//   ksplit token tiles, mode 2 only: split K into ksplit ranges, each unit
//          once per range, split s writing fp32 columns s * N_out .. of rows
//          N_out * ksplit wide (the caller sums the splits); at most the K
//          stages (64 elements each).
cudaError_t launch_gemm_tc(int mode, bool fp8, bool decode, const void* a, const float* a_scale,
                           const void* w, const float* w_scale, const int32_t* offsets,
                           const int32_t* row_src, const float* topk_w, void* c, int E, int K,
                           int I, int N_out, int R_max, int T, int sms, int* status,
                           cudaStream_t st, int* sched = nullptr, int ksplit = 1);

// Decode FFN in one persistent launch: FC1 + silu_and_mul (xp -> act) and
// FC2 + routing weight (act -> y, bf16 rows in (token, slot) order), with a
// dynamic unit scheduler.  `sched` holds 1 + 2E ints that must be zero when
// the kernel starts.  With fp8, xp / w13 / w2 are E4M3 codes with scales and
// the FC1 rows are quantised per row into actq / act_scale inside the launch.
// cudaErrorNotSupported when not covered.
cudaError_t launch_decode_ffn_fused(bool fp8, const void* xp, const float* xp_scale,
                                    const void* w13, const float* w13_scale, const void* w2,
                                    const float* w2_scale, void* act, uint8_t* actq,
                                    float* act_scale, void* y, const int32_t* offsets,
                                    const int32_t* row_src, const float* topk_w, int* sched, int E,
                                    int H, int I, int R_max, int T, int sms, int* status,
                                    cudaStream_t st);

// The whole decode forward in one cooperative launch (one CTA per SM):
// rms_norm, routing, permute and row gather, the fused FC1 + FC2, the combine,
// separated by grid barriers.  bf16 tensors are passed as void pointers.
struct DecodeForward {
  const void* x;          // bf16 [T, H]
  const void* norm_w;     // bf16 [H]
  float eps;
  int T, H, k;
  const float* logits;    // router logits [T, E], or NULL
  const float* router_w;  // [H, E], or NULL (used when logits is NULL)
  const float* bias;      // [E] or NULL
  const int32_t* ids_in;  // caller routing [T, k] and weights, or NULL
  const float* tw_in;
  void* xhat;             // bf16 [T, H]
  uint8_t* xq;            // E4M3 path: quantised x_hat [T, H] and scales [T]
  float* xscale;
  int32_t* ids;           // routing outputs (used when ids_in is NULL)
  float* tw;
  int32_t* offsets;       // [E + 1]
  int32_t* row_src;       // [T k]
  int32_t* row_of_pair;   // [T k]
  void* xp;               // gathered rows [T k, H] (bf16, or E4M3 with xp_scale)
  float* xp_scale;
  void* y;                // FC2 rows bf16 [T k, H], (token, slot) order
  void* out;              // bf16 [T, H]
  int* bar;               // grid barrier words (2 ints), zeroed by the launcher
};

// Whether the one-launch forward is enabled (MOE_MEGA=1) and covers the
// batch and router (host check).
bool decode_forward_mega_covers(int T, int H, int E, int k, bool logits, bool routed);

cudaError_t launch_decode_forward_mega(bool fp8, const DecodeForward& f, const void* w13,
                                       const float* w13_scale, const void* w2,
                                       const float* w2_scale, void* act, uint8_t* actq,
                                       float* act_scale, int* sched, int E, int I, int sms,
                                       int* status, cudaStream_t st);

// NVFP4 weights (gemm_nvfp4.cu): quantiser, fp16 row gather, and the
// decode FFN (FC1 + silu_and_mul -> fp16 act, FC2 + routing weight -> bf16 y
// rows at row_src) in one persistent launch; `sched` as for
// launch_decode_ffn_fused.  cudaErrorNotSupported when not covered.
cudaError_t launch_quantize_nvfp4(const void* w, int M, int N, int K, uint8_t* q, uint8_t* sb,
                                  float* sg, cudaStream_t st);
cudaError_t launch_gather_rows_f16(const int32_t* offsets, int E, const int32_t* row_src, int k,
                                   int R_max, int H, const void* src, void* dst, cudaStream_t st);
bool nvfp4_decode_covers(int H, int I, int E);
cudaError_t launch_decode_ffn_nvfp4(const void* xp, const uint8_t* w13_q, const uint8_t* w13_sb,
                                    const float* w13_sg, const uint8_t* w2_q, const uint8_t* w2_sb,
                                    const float* w2_sg, void* act, void* y, const int32_t* offsets,
                                    const int32_t* row_src, const float* topk_w, int* sched, int E,
                                    int H, int I, int R_max, int T, int sms, int* status,
                                    cudaStream_t st);

// Block-wise FP8 weights (gemm_fp8b.cu): E4M3 codes with one fp32 scale per
// 128 x 128 weight tile and per 1 x 128 activation group.  Quantiser
// (block_rows 1 or 128), rms_norm with group quantisation of x_hat, and the
// decode FFN (FC1 + silu_and_mul -> E4M3 act with group scales, FC2 + routing
// weight -> bf16 y rows at row_src) in one persistent launch; `sched` as for
// launch_decode_ffn_fused.  cudaErrorNotSupported when not covered.
cudaError_t launch_quantize_fp8_blocks(const void* x, int N, int K, int block_rows, uint8_t* q,
                                       float* scale, cudaStream_t st);
cudaError_t launch_rmsnorm_q128(const void* x, const void* w, int T, int H, float eps, void* y,
                                uint8_t* yq, float* yscale, cudaStream_t st);
bool fp8b_decode_covers(int H, int I, int E);
cudaError_t launch_decode_ffn_fp8b(const uint8_t* xp, const float* xp_scale, const uint8_t* w13,
                                   const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                   uint8_t* actq, float* act_scale, void* y, const int32_t* offsets,
                                   const int32_t* row_src, const float* topk_w, int* sched, int E,
                                   int H, int I, int R_max, int T, int sms, int* status,
                                   cudaStream_t st);

// Block-wise FP8 for many rows per expert: FC1 tiles (128 tokens x 64 gate
// + 64 up rows) -> bf16 act, group quantisation of act, FC2 tiles (128
// tokens x 128 rows of W2) -> bf16 rows at row_src; three launches.
cudaError_t launch_prefill_ffn_fp8b(const uint8_t* xp, const float* xp_scale, const uint8_t* w13,
                                    const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, void* act, uint8_t* actq,
                                    float* act_scale, void* y, const int32_t* offsets,
                                    const int32_t* row_src, const float* topk_w, int E, int H,
                                    int I, int R_max, int sms, int* status, cudaStream_t st);

// Bounded-wait self-test: a kernel that waits on an mbarrier nothing arrives
// on for at most limit_cycles SM cycles and records MOE_ERR_TIMEOUT.
cudaError_t launch_wait_selftest(long long limit_cycles, int* status, cudaStream_t st);

}  // namespace moe
