// Grouped GEMM over expert segments on the CUDA cores (fp32 FMA).
//
// The general engine: any supported shape, every mode (FC1 raw, FC1 with the
// silu_and_mul epilogue, FC2 with the routing-weight epilogue), bf16 or E4M3
// operands.  A CTA computes a BM x BN output tile of one expert; the CTA grid
// is (N tiles) x (M tiles summed over experts), and each CTA maps its M-tile
// index to (expert, first row) from the expert offsets held in device memory,
// so the host never reads the routing.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BM = 32, BN = 64, BK = 32;

// Loads 8 consecutive K elements of a row into floats (bf16 or E4M3 codes).
template <bool FP8>
MOE_DEV void load8(const void* base, size_t elem_off, float* f) {
  if (!FP8) {
    uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(base) + elem_off);
    unpack8_bf16(u, f);
  } else {
    uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(base) + elem_off);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = e4m3_to_f((uint8_t)(u.x >> (8 * i)));
#pragma unroll
    for (int i = 0; i < 4; ++i) f[4 + i] = e4m3_to_f((uint8_t)(u.y >> (8 * i)));
  }
}
}  // namespace

// MODE 0: FC1 raw (W rows n of [2I]), out bf16 [R, 2I]
// MODE 1: FC1 silu (gate rows n, up rows I+n), out bf16 [R, I]
// MODE 2: FC2 (W rows n of [H]), out fp32 [R, H] x topk_w
// MODE 3: FC2, out bf16 x topk_w, row r stored at row_src[r] ((token, slot) order)
template <int MODE, bool FP8>
__global__ void __launch_bounds__(256) gemm_simt_kernel(
    const void* __restrict__ A, const float* __restrict__ a_scale, const void* __restrict__ W,
    const float* __restrict__ w_scale, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ row_src, const float* __restrict__ topk_w, void* __restrict__ C,
    int E, int K, int I, int N_out, int N_w) {
  constexpr int NW = (MODE == 1) ? 2 : 1;  // weight tiles per CTA (gate, up)
  __shared__ float As[BK][BM + 1];
  __shared__ float Ws[NW][BK][BN + 1];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_tp[kMaxExperts + 1];
  __shared__ int s_e, s_row0;

  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  for (int e = tid; e <= E; e += blockDim.x) s_off[e] = offsets[e];
  __syncthreads();
  if (tid < 32) {  // prefix of M tiles per expert
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + tid;
      const int v = (e < E) ? (s_off[e + 1] - s_off[e] + BM - 1) / BM : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += n;
      }
      if (e < E) s_tp[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid == 0) s_tp[E] = carry;
  }
  __syncthreads();
  const int m = blockIdx.y;
  if (m >= s_tp[E]) return;
  if (tid == 0) {
    int lo = 0, hi = E - 1;  // last e with s_tp[e] <= m
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tp[mid] <= m) lo = mid; else hi = mid - 1;
    }
    s_e = lo;
    s_row0 = s_off[lo] + (m - s_tp[lo]) * BM;
  }
  __syncthreads();
  const int e = s_e, row0 = s_row0, row_end = s_off[e + 1];
  const int n0 = blockIdx.x * BN;

  const int tx = tid & 31, ty = tid >> 5;  // cols tx, tx+32; rows ty*4 .. ty*4+3
  float acc[NW][4][2];
#pragma unroll
  for (int q = 0; q < NW; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[q][i][0] = acc[q][i][1] = 0.f;

  for (int kb = 0; kb < K; kb += BK) {
    {  // A tile: BM rows x BK; 4 threads per row, 8 k each
      const int rr = tid >> 2, kk = (tid & 3) * 8;
      const int r = row0 + rr;
      float f[8];
      if (rr < BM && r < row_end) {
        load8<FP8>(A, (size_t)r * K + kb + kk, f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
      if (rr < BM) {
#pragma unroll
        for (int i = 0; i < 8; ++i) As[kk + i][rr] = f[i];
      }
    }
#pragma unroll
    for (int q = 0; q < NW; ++q) {  // W tile(s): BN rows x BK; 4 threads per row
      const int nn = tid >> 2, kk = (tid & 3) * 8;
      const int n = n0 + nn + (q == 1 ? I : 0);
      float f[8];
      load8<FP8>(W, ((size_t)e * N_w + n) * K + kb + kk, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) Ws[q][kk + i][nn] = f[i];
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BK; ++kk) {
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int q = 0; q < NW; ++q) {
        const float b0 = Ws[q][kk][tx], b1 = Ws[q][kk][tx + 32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[q][i][0] = fmaf(a[i], b0, acc[q][i][0]);
          acc[q][i][1] = fmaf(a[i], b1, acc[q][i][1]);
        }
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= row_end) continue;
    const float sa = FP8 ? a_scale[r] : 1.f;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int n = n0 + tx + 32 * c;
      if (MODE == 0) {
        float v = acc[0][i][c];
        if (FP8) v = v * sa * w_scale[(size_t)e * N_w + n];
        reinterpret_cast<bf16*>(C)[(size_t)r * N_out + n] = __float2bfloat16_rn(v);
      } else if (MODE == 1) {
        float g = acc[0][i][c], u = acc[1][i][c];
        if (FP8) {
          g = g * sa * w_scale[(size_t)e * N_w + n];
          u = u * sa * w_scale[(size_t)e * N_w + I + n];
        }
        reinterpret_cast<bf16*>(C)[(size_t)r * N_out + n] = __float2bfloat16_rn(silu_f(g) * u);
      } else {
        float v = acc[0][i][c];
        if (FP8) v = v * sa * w_scale[(size_t)e * N_w + n];
        const float tw = topk_w ? topk_w[row_src[r]] : 1.f;
        if (MODE == 2) {
          reinterpret_cast<float*>(C)[(size_t)r * N_out + n] = tw * v;
        } else {  // bf16 rows go back to (token, slot) order
          const int orow = row_src ? row_src[r] : r;
          reinterpret_cast<bf16*>(C)[(size_t)orow * N_out + n] = __float2bfloat16_rn(tw * v);
        }
      }
    }
  }
}

cudaError_t launch_gemm_simt(int mode, bool fp8, const void* a, const float* a_scale,
                             const void* w, const float* w_scale, const int32_t* offsets,
                             const int32_t* row_src, const float* topk_w, void* c, int E, int K,
                             int I, int N_out, int R_max, cudaStream_t st) {
  if (R_max == 0) return cudaSuccess;
  // N_w: rows of one expert's weight matrix.
  const int N_w = (mode >= 2) ? N_out : 2 * I;
  dim3 grid(N_out / BN, (R_max + BM - 1) / BM + E);
#define MOE_SIMT_LAUNCH(MD, F8)                                                             \
  return launch_kernel(gemm_simt_kernel<MD, F8>, grid, dim3(256), 0, st, a, a_scale, w, w_scale, \
                       offsets, row_src, topk_w, c, E, K, I, N_out, N_w)
  if (mode == 0) { if (fp8) MOE_SIMT_LAUNCH(0, true); else MOE_SIMT_LAUNCH(0, false); }
  else if (mode == 1) { if (fp8) MOE_SIMT_LAUNCH(1, true); else MOE_SIMT_LAUNCH(1, false); }
  else if (mode == 2) { if (fp8) MOE_SIMT_LAUNCH(2, true); else MOE_SIMT_LAUNCH(2, false); }
  else { if (fp8) MOE_SIMT_LAUNCH(3, true); else MOE_SIMT_LAUNCH(3, false); }
#undef MOE_SIMT_LAUNCH
}

}  // namespace moe
