// The non-GEMM steps of the MoE expert FFN forward: rms_norm, router logits,
// softmax/top-k/renorm, permute (+ row gather), silu_and_mul, combine and
// row-wise E4M3 quantisation.  All are HBM- or latency-bound; they use
// 16-byte vector accesses and warp-shuffle reductions.
#include "common.cuh"
#include "kernels.h"

#include <float.h>
#include <stdlib.h>

#include <atomic>

namespace {
thread_local bool t_pdl_off = false;
std::atomic<long long> g_launch_count{0};
}  // namespace

void count_launch() { g_launch_count.fetch_add(1, std::memory_order_relaxed); }
long long launch_count() { return g_launch_count.load(std::memory_order_relaxed); }

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("MOE_PDL");
    return !(e && e[0] == '0');
  }();
  return on && !t_pdl_off;
}

PdlOff::PdlOff(bool off) : prev_(t_pdl_off) {
  if (off) t_pdl_off = true;
}

PdlOff::~PdlOff() { t_pdl_off = prev_; }

namespace moe {

// ===================================================================== rms_norm
// One CTA per token row.  y = bf16((x * r) * w), r = 1 / sqrt(mean(x^2) + eps)
// (the pow -> mean -> rsqrt -> mul composite, fp32).  With FP8 the bf16 row is
// also quantised per token: s = absmax / 448, q = e4m3(y / s).
template <bool FP8>
__global__ void __launch_bounds__(512) rmsnorm_kernel(const bf16* __restrict__ x,
                                                      const bf16* __restrict__ w, int H, float eps,
                                                      bf16* __restrict__ y, uint8_t* __restrict__ yq,
                                                      float* __restrict__ yscale) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int nv = H >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)t * H);
  float ss = 0.f;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float f[8];
    unpack8_bf16(xr[v], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
  ss = block_sum(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
  float amax = 0.f;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float f[8], g[8];
    unpack8_bf16(xr[v], f);
    unpack8_bf16(wr[v], g);
    uint4 o;
    o.x = pack2_bf16((f[0] * r) * g[0], (f[1] * r) * g[1]);
    o.y = pack2_bf16((f[2] * r) * g[2], (f[3] * r) * g[3]);
    o.z = pack2_bf16((f[4] * r) * g[4], (f[5] * r) * g[5]);
    o.w = pack2_bf16((f[6] * r) * g[6], (f[7] * r) * g[7]);
    yr[v] = o;
    if (FP8) {
      float h[8];
      unpack8_bf16(o, h);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(h[i]));
    }
  }
  if (FP8) {
    amax = block_max(amax, red);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint2* qr = reinterpret_cast<uint2*>(yq + (size_t)t * H);
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float h[8];
      unpack8_bf16(yr[v], h);  // this thread wrote yr[v] above
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) lo |= (uint32_t)f_to_e4m3(__fdiv_rn(h[i], s)) << (8 * i);
#pragma unroll
      for (int i = 0; i < 4; ++i) hi |= (uint32_t)f_to_e4m3(__fdiv_rn(h[4 + i], s)) << (8 * i);
      qr[v] = make_uint2(lo, hi);
    }
    if (threadIdx.x == 0) yscale[t] = s;
  }
}

// Threads per token row (one CTA each).  Large batches: about four 16-byte
// vectors per thread (128 threads at H = 4096), so an SM holds 16 tokens'
// CTAs instead of 4 and overlaps their load -> reduce -> store chains
// (prefill rms_norm 26 -> 19.5 us, with the E4M3 copy 41 -> 28 us).  Small
// batches have fewer CTAs than SMs, where one vector per thread is faster.
int rmsnorm_threads(int T, int nv) {
  int threads = T >= 512 ? ((nv + 3) / 4 + 31) / 32 * 32 : ((nv + 31) / 32) * 32;
  return threads < 32 ? 32 : (threads > 512 ? 512 : threads);
}

cudaError_t launch_rmsnorm(const void* x, const void* w, int T, int H, float eps, void* y,
                           void* yq, float* yscale, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int nv = H / 8;
  int threads = rmsnorm_threads(T, nv);
  if (yq)
    return launch_kernel(rmsnorm_kernel<true>, dim3(T), dim3(threads), 0, st, (const bf16*)x,
                         (const bf16*)w, H, eps, (bf16*)y, (uint8_t*)yq, yscale);
  return launch_kernel(rmsnorm_kernel<false>, dim3(T), dim3(threads), 0, st, (const bf16*)x,
                       (const bf16*)w, H, eps, (bf16*)y, (uint8_t*)nullptr, (float*)nullptr);
}

// ================================================================ router logits
// part[z, t, e] = sum over the z-th K chunk of xhat[t, h] * Wr[h, e]  (fp32,
// h ascending within the chunk).  The chunks are summed in order by the
// top-k kernel, so the logits are deterministic.  CTA tile: TT tokens x TE
// experts, K step 32; each thread owns an 8 x 8 register tile (four 16-byte
// shared-memory reads per 64 FMA).  The next K slice is prefetched into
// registers while the current one is multiplied out of shared memory.
constexpr int RT_K = 32;

struct RouterTile {
  int tt, te;
};

// 128x64 for many tokens, 64x128 for few tokens and many experts, else 64x64.
RouterTile router_tile(int T, int E) {
  if (T >= 128) return {128, 64};
  if (E >= 128) return {64, 128};
  return {64, 64};
}

template <int TT, int TE>
__global__ void __launch_bounds__((TT / 8) * (TE / 8)) router_logits_kernel(
    const bf16* __restrict__ xhat, const float* __restrict__ wr, int T, int H, int E, int kchunk,
    float* __restrict__ part) {
  constexpr int NT = (TT / 8) * (TE / 8);           // threads
  constexpr int XV = TT * RT_K * 2 / 16 / NT;       // x_hat uint4 loads per thread
  constexpr int WV = RT_K * TE * 4 / 16 / NT;       // W_r float4 loads per thread
  constexpr int XPT = RT_K / 8 / (NT / TT);         // uint4 of one token row per thread
  __shared__ __align__(16) float xs[RT_K][TT + 4];  // [k][token]
  __shared__ __align__(16) float ws[RT_K][TE];      // [k][expert]
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * TT, e0 = blockIdx.y * TE;
  const int kb0 = blockIdx.z * kchunk;
  const int kb1 = min(H, kb0 + kchunk);
  const int tx = tid % (TE / 8), ty = tid / (TE / 8);  // experts tx*8.., tokens ty*8..
  const bool e_vec = (E % 4 == 0);
  // x_hat loads: thread -> token xt, uint4 chunks xc .. xc + XV - 1 of its 32-k row
  const int xt = tid / (NT / TT), xc = (tid % (NT / TT)) * XPT;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  uint4 xr[XV];
  float4 wv[WV];
  auto gload = [&](int kb) {
    const int t = t0 + xt;
#pragma unroll
    for (int i = 0; i < XV; ++i)
      xr[i] = (t < T) ? *reinterpret_cast<const uint4*>(xhat + (size_t)t * H + kb + (xc + i) * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < WV; ++i) {
      const int idx = tid + i * NT;
      const int kk = idx / (TE / 4), e = e0 + (idx % (TE / 4)) * 4;
      const float* src = wr + (size_t)(kb + kk) * E + e;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e_vec && e + 3 < E) {
        v = *reinterpret_cast<const float4*>(src);
      } else {
        if (e < E) v.x = src[0];
        if (e + 1 < E) v.y = src[1];
        if (e + 2 < E) v.z = src[2];
        if (e + 3 < E) v.w = src[3];
      }
      wv[i] = v;
    }
  };
  if (kb0 < kb1) gload(kb0);
  for (int kb = kb0; kb < kb1; kb += RT_K) {
#pragma unroll
    for (int i = 0; i < XV; ++i) {
      float f[8];
      unpack8_bf16(xr[i], f);
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[(xc + i) * 8 + q][xt] = f[q];
    }
#pragma unroll
    for (int i = 0; i < WV; ++i) {
      const int idx = tid + i * NT;
      *reinterpret_cast<float4*>(&ws[idx / (TE / 4)][(idx % (TE / 4)) * 4]) = wv[i];
    }
    __syncthreads();
    if (kb + RT_K < kb1) gload(kb + RT_K);
#pragma unroll 4
    for (int kk = 0; kk < RT_K; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&xs[kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&xs[kk][ty * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&ws[kk][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&ws[kk][tx * 8 + 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= T) continue;
    float* dst = part + ((size_t)blockIdx.z * T + t) * E;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + tx * 8 + j;
      if (e < E) dst[e] = acc[i][j];
    }
  }
}

int route_splits(int T, int H, int E) {
  const RouterTile rt = router_tile(T, E);
  const int tiles = ((T + rt.tt - 1) / rt.tt) * ((E + rt.te - 1) / rt.te);
  const int steps = H / RT_K;
  int ks = (4 * 152 + tiles - 1) / tiles;  // about four CTAs per SM
  const int min_steps = 4;                 // at least 128 K per chunk
  if (ks > steps / min_steps) ks = steps / min_steps;
  if (ks < 1) ks = 1;
  const int per = (steps + ks - 1) / ks;  // K steps per chunk
  return (steps + per - 1) / per;         // chunks actually needed
}

cudaError_t launch_router_logits(const void* xhat, const float* wr, int T, int H, int E, int ks,
                                 float* part, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  // K chunk: a multiple of RT_K covering H in ks pieces.
  const int steps = H / RT_K;
  const int per = (steps + ks - 1) / ks;
  const int kchunk = per * RT_K;
  const int ks_eff = (H + kchunk - 1) / kchunk;
  if (ks_eff != ks) return cudaErrorInvalidValue;  // route_splits() keeps these equal
  const RouterTile rt = router_tile(T, E);
  dim3 grid((T + rt.tt - 1) / rt.tt, (E + rt.te - 1) / rt.te, ks);
  if (rt.tt == 128)
    return launch_kernel(router_logits_kernel<128, 64>, grid, dim3(128), 0, st, (const bf16*)xhat,
                         wr, T, H, E, kchunk, part);
  if (rt.te == 128)
    return launch_kernel(router_logits_kernel<64, 128>, grid, dim3(128), 0, st, (const bf16*)xhat,
                         wr, T, H, E, kchunk, part);
  return launch_kernel(router_logits_kernel<64, 64>, grid, dim3(64), 0, st, (const bf16*)xhat, wr,
                       T, H, E, kchunk, part);
}

// ==================================================== softmax / top-k / renorm
// One warp per token.  Logit of expert e = sum_z part[z, t, e] (+ bias[e]).
template <int PER>
__global__ void __launch_bounds__(128) topk_kernel(const float* __restrict__ part, int ks,
                                                   size_t zstride, size_t tstride,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ wout,
                                                   float* __restrict__ logits_out) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  float v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) v[i] = 0.f;
  // Partial sums: four chunks are loaded before they are added (4 x PER
  // loads in flight per lane, PER = ceil(E / 32) values of each logit row
  // per lane); each logit is still summed in z order.
  const float* pt = part + (size_t)t * tstride;
  int z = 0;
  for (; z + 4 <= ks; z += 4) {
    float l[4][PER];
#pragma unroll
    for (int zz = 0; zz < 4; ++zz)
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        l[zz][i] = e < E ? pt[(size_t)(z + zz) * zstride + e] : 0.f;
      }
#pragma unroll
    for (int zz = 0; zz < 4; ++zz)
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (lane + 32 * i < E) v[i] += l[zz][i];
  }
  for (; z < ks; ++z) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (e < E) v[i] += pt[(size_t)z * zstride + e];
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      if (bias) v[i] += bias[e];
      if (logits_out) logits_out[(size_t)t * E + e] = v[i];
    } else {
      v[i] = -FLT_MAX;
    }
  }
  warp_topk(v, E, k, lane, ids + (size_t)t * k, wout + (size_t)t * k);
}

// Router + top-k for small routers (H * E <= kRouteSmallMaxHE, H <= 8192): one
// CTA per token.  The token's x_hat row is staged in shared memory as fp32;
// thread (g, e), g < G = 256 / E, sums x_hat[h] * W_r[h, e] over the rows
// h = g, g + G, ... (a row of W_r is read by consecutive threads), the G
// partial sums of expert e are added in g order, and warp 0 selects the top k.
constexpr int kRouteSmallMaxHE = 65536;
constexpr int kRouteSmallMaxH = 8192;

template <int PER>
__global__ void __launch_bounds__(256) route_small_kernel(const bf16* __restrict__ xhat,
                                                          const float* __restrict__ wr,
                                                          const float* __restrict__ bias, int T,
                                                          int H, int E, int k,
                                                          int32_t* __restrict__ ids,
                                                          float* __restrict__ wout,
                                                          float* __restrict__ logits_out) {
  __shared__ float xs[kRouteSmallMaxH];
  __shared__ float ps[256];
  __shared__ float lg[kMaxExperts];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(xhat + (size_t)t * H);
  for (int v = tid; v < H / 8; v += blockDim.x) {
    float f[8];
    unpack8_bf16(xr[v], f);
#pragma unroll
    for (int q = 0; q < 8; ++q) xs[v * 8 + q] = f[q];
  }
  __syncthreads();
  const int G = blockDim.x / E;  // row groups (>= 1: E <= 256)
  const int g = tid / E, e = tid % E;
  float acc = 0.f;
  if (g < G) {
    for (int h = g; h < H; h += G) acc = fmaf(xs[h], wr[(size_t)h * E + e], acc);
  }
  ps[tid] = acc;
  __syncthreads();
  for (int ee = tid; ee < E; ee += blockDim.x) {
    float s = 0.f;
    for (int gg = 0; gg < G; ++gg) s += ps[gg * E + ee];
    if (bias) s += bias[ee];
    lg[ee] = s;
    if (logits_out) logits_out[(size_t)t * E + ee] = s;
  }
  __syncthreads();
  if (tid < 32) {
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int ex = tid + 32 * i;
      v[i] = ex < E ? lg[ex] : -FLT_MAX;
    }
    warp_topk(v, E, k, tid, ids + (size_t)t * k, wout + (size_t)t * k);
  }
}

bool route_small(int H, int E) {
  return H <= kRouteSmallMaxH && (int64_t)H * E <= kRouteSmallMaxHE;
}

cudaError_t launch_route_small(const void* xhat, const float* wr, const float* bias, int T,
                               int H, int E, int k, int32_t* ids, float* w, float* logits_out,
                               cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (!route_small(H, E)) return cudaErrorInvalidValue;
  // the selection scans ceil(E / 32) values per lane (1, 2, 4 or 8)
  auto go = [&](auto kern) {
    return launch_kernel(kern, dim3(T), dim3(256), 0, st, (const bf16*)xhat, wr, bias, T, H, E, k,
                         ids, w, logits_out);
  };
  if (E <= 32) return go(route_small_kernel<1>);
  if (E <= 64) return go(route_small_kernel<2>);
  if (E <= 128) return go(route_small_kernel<4>);
  return go(route_small_kernel<kTopkPer>);
}

cudaError_t launch_topk(const float* part, int ks, const float* bias, int T, int E, int k,
                        int32_t* ids, float* w, float* logits_out, cudaStream_t st,
                        size_t zstride, size_t tstride) {
  if (T == 0) return cudaSuccess;
  if (zstride == 0) zstride = (size_t)T * E;  // default: part[z][t][e]
  if (tstride == 0) tstride = (size_t)E;
  // the selection scans ceil(E / 32) values per lane (1, 2, 4 or 8)
  auto go = [&](auto kern) {
    return launch_kernel(kern, dim3((T + 3) / 4), dim3(128), 0, st, part, ks, zstride, tstride,
                         bias, T, E, k, ids, w, logits_out);
  };
  if (E <= 32) return go(topk_kernel<1>);
  if (E <= 64) return go(topk_kernel<2>);
  if (E <= 128) return go(topk_kernel<4>);
  return go(topk_kernel<kTopkPer>);
}

// Router weights for the tensor-core router: W_r fp32 [H, E] -> three bf16
// pieces, transposed to K-major rows wt[p*E + e][h] (p = 0 hi, 1 mid, 2 lo):
// hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid); the differences
// are exact in fp32, so hi + mid + lo equals w to 2^-24 relative and each
// product with a bf16 x_hat is exact.  Also writes the one-segment offsets
// {0, T} the grouped GEMM reads.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ wr, int H,
                                                           int E, int T, bf16* __restrict__ wt,
                                                           int32_t* __restrict__ seg) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[32][33];
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int i = ty; i < 32; i += 8) {
    const int h = h0 + i, e = e0 + tx;
    tile[i][tx] = (h < H && e < E) ? wr[(size_t)h * E + e] : 0.f;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + i, h = h0 + tx;
    if (e < E && h < H) {
      const float w = tile[tx][i];
      const bf16 hi = __float2bfloat16_rn(w);
      const float r1 = w - __bfloat162float(hi);
      const bf16 mid = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid);
      const bf16 lo = __float2bfloat16_rn(r2);
      wt[(size_t)e * H + h] = hi;
      wt[((size_t)E + e) * H + h] = mid;
      wt[((size_t)2 * E + e) * H + h] = lo;
    }
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    seg[0] = 0;
    seg[1] = T;
  }
}

cudaError_t launch_router_split(const float* wr, int H, int E, int T, void* wt, int32_t* seg,
                                cudaStream_t st) {
  dim3 grid((H + 31) / 32, (E + 31) / 32);
  return launch_kernel(router_split_kernel, grid, dim3(256), 0, st, wr, H, E, T, (bf16*)wt, seg);
}

// ====================================================================== permute
// Stable counting sort of the T*k pairs by expert in one CTA of 32 warps.
// Warp w owns a contiguous chunk of tokens.  Pass 1 counts per (warp, expert);
// pass 2 turns the counts into each warp's first row per expert (expert-major
// exclusive prefix, then warp order); pass 3 walks each chunk in pair order in
// batches of 32 and ranks equal experts inside a batch with __match_any_sync.
constexpr int PERM_WARPS = 32;

__global__ void __launch_bounds__(PERM_WARPS * 32) permute_kernel(
    const int32_t* __restrict__ ids, int T, int E, int k, int32_t* __restrict__ offsets,
    int32_t* __restrict__ row_src, int32_t* __restrict__ row_of_pair, int* status,
    int32_t* __restrict__ zero_buf, int nzero) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sm[];
  for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero_buf[i] = 0;  // later kernels' counters
  int* cnt = sm;                         // [PERM_WARPS][E]
  int* tot = sm + PERM_WARPS * E;        // [E + 1]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < PERM_WARPS * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int chunk = (T + PERM_WARPS - 1) / PERM_WARPS;
  const int tb = min(T, w * chunk), te = min(T, (w + 1) * chunk);
  const int p0 = tb * k, p1 = te * k;
  for (int p = p0 + lane; p < p1; p += 32) {
    const int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[w * E + e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int ww = 0; ww < PERM_WARPS; ++ww) s += cnt[ww * E + e];
    tot[e] = s;
  }
  __syncthreads();
  if (w == 0) {  // exclusive scan of tot[0..E) by warp 0
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int v = (e < E) ? tot[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) tot[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tot[E] = carry;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    offsets[e] = tot[e];
    if (e < E) {
      int run = tot[e];
      for (int ww = 0; ww < PERM_WARPS; ++ww) {
        const int c = cnt[ww * E + e];
        cnt[ww * E + e] = run;
        run += c;
      }
    }
  }
  __syncthreads();
  bool bad = false;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    const bool valid = p < p1;
    int e = valid ? ids[p] : -1;
    const bool ok = valid && e >= 0 && e < E;
    if (valid && !ok) bad = true;
    const int key = ok ? e : -1 - lane;  // invalid lanes form singleton groups
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    if (ok) {
      const int rank = __popc(grp & ((1u << lane) - 1u));
      const int r = cnt[w * E + e] + rank;
      row_src[r] = p;
      row_of_pair[p] = r;
    } else if (valid) {
      row_of_pair[p] = -1;
    }
    __syncwarp();
    if (ok && (grp & ((1u << lane) - 1u)) == 0) cnt[w * E + e] += __popc(grp);
    __syncwarp();
  }
  if (bad) flag_status(status, MOE_ERR_INVALID_ARG);
}

cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* offsets,
                           int32_t* row_src, int32_t* row_of_pair, int* status, cudaStream_t st,
                           int32_t* zero_buf, int nzero) {
  size_t smem = (size_t)(PERM_WARPS * E + E + 1) * sizeof(int);
  return launch_kernel(permute_kernel, dim3(1), dim3(PERM_WARPS * 32), smem, st, ids, T, E, k,
                       offsets, row_src, row_of_pair, status, zero_buf, nzero);
}

// Parallel form of the same stable counting sort, for large batches: chunks
// of PC_TOK tokens.  (1) per-chunk expert counts; (2) one CTA turns them into
// each chunk's first row per expert (expert-major prefix, then chunk order)
// and the expert offsets; (3) one warp per chunk ranks its pairs in pair
// order exactly as permute_kernel's pass 3.
constexpr int PC_TOK = 32;

int permute_chunks(int T) { return (T + PC_TOK - 1) / PC_TOK; }

bool permute_parallel(int T, int k) { return (int64_t)T * k > 4096; }

__global__ void __launch_bounds__(256) permute_count_kernel(const int32_t* __restrict__ ids, int T,
                                                            int E, int k, int32_t* __restrict__ cnt,
                                                            int* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ int c[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) c[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * PC_TOK * k, p1 = min(T, (blockIdx.x + 1) * PC_TOK) * k;
  bool bad = false;
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&c[e], 1);
    else bad = true;
  }
  if (bad) flag_status(status, MOE_ERR_INVALID_ARG);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[(size_t)blockIdx.x * E + e] = c[e];
}

__global__ void __launch_bounds__(256) permute_scan_kernel(int nch, int E,
                                                           int32_t* __restrict__ cnt,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ zero_buf,
                                                           int nzero) {
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero_buf[i] = 0;  // later kernels' counters
  __shared__ int tot[kMaxExperts + 1];
  const int e = threadIdx.x;
  if (e < E) {
    int s = 0;
    for (int ch = 0; ch < nch; ++ch) s += cnt[(size_t)ch * E + e];
    tot[e] = s;
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // exclusive scan over experts by warp 0
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int ee = base + lane;
      const int v = (ee < E) ? tot[ee] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (ee < E) tot[ee] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tot[E] = carry;
  }
  __syncthreads();
  if (e < E) offsets[e] = tot[e];
  if (threadIdx.x == 0) offsets[E] = tot[E];
  if (e < E) {
    int run = tot[e];
    for (int ch = 0; ch < nch; ++ch) {
      const int c = cnt[(size_t)ch * E + e];
      cnt[(size_t)ch * E + e] = run;
      run += c;
    }
  }
}

__global__ void __launch_bounds__(32) permute_scatter_kernel(const int32_t* __restrict__ ids,
                                                             int T, int E, int k,
                                                             const int32_t* __restrict__ base,
                                                             int32_t* __restrict__ row_src,
                                                             int32_t* __restrict__ row_of_pair) {
  pdl_trigger();
  pdl_wait();
  __shared__ int nxt[kMaxExperts];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) nxt[e] = base[(size_t)blockIdx.x * E + e];
  __syncwarp();
  const int p0 = blockIdx.x * PC_TOK * k, p1 = min(T, (blockIdx.x + 1) * PC_TOK) * k;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    const bool valid = p < p1;
    const int e = valid ? ids[p] : -1;
    const bool ok = valid && e >= 0 && e < E;
    const int key = ok ? e : -1 - lane;
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    if (ok) {
      const int r = nxt[e] + __popc(grp & ((1u << lane) - 1u));
      row_src[r] = p;
      row_of_pair[p] = r;
    } else if (valid) {
      row_of_pair[p] = -1;
    }
    __syncwarp();
    if (ok && (grp & ((1u << lane) - 1u)) == 0) nxt[e] += __popc(grp);
    __syncwarp();
  }
}

size_t permute_workspace_bytes(int T, int E, int k) {
  return permute_parallel(T, k) ? (size_t)permute_chunks(T) * E * sizeof(int32_t) : 0;
}

cudaError_t launch_permute_any(const int32_t* ids, int T, int E, int k, int32_t* offsets,
                               int32_t* row_src, int32_t* row_of_pair, int32_t* cnt_ws,
                               int* status, cudaStream_t st, int32_t* zero_buf, int nzero) {
  if (!permute_parallel(T, k))
    return launch_permute(ids, T, E, k, offsets, row_src, row_of_pair, status, st, zero_buf,
                          nzero);
  const int nch = permute_chunks(T);
  cudaError_t e = launch_kernel(permute_count_kernel, dim3(nch), dim3(256), 0, st, ids, T, E, k,
                                cnt_ws, status);
  if (e != cudaSuccess) return e;
  e = launch_kernel(permute_scan_kernel, dim3(1), dim3(256), 0, st, nch, E, cnt_ws, offsets,
                    zero_buf, nzero);
  if (e != cudaSuccess) return e;
  return launch_kernel(permute_scatter_kernel, dim3(nch), dim3(32), 0, st, ids, T, E, k,
                       (const int32_t*)cnt_ws, row_src, row_of_pair);
}

// Row gather dst[r, :] = src[row_src[r] / k, :] for r < offsets[E]
// (row_bytes a multiple of 16); optional per-row scale gather.
__global__ void __launch_bounds__(256) gather_rows_kernel(const int32_t* __restrict__ offsets,
                                                          int E, const int32_t* __restrict__ row_src,
                                                          int k, int R_max,
                                                          const uint4* __restrict__ src,
                                                          uint4* __restrict__ dst, int row_vec,
                                                          const float* __restrict__ sscale,
                                                          float* __restrict__ dscale, int scols,
                                                          int parts) {
  pdl_trigger();
  pdl_wait();
  const int R = min(offsets[E], R_max);
  const int warps = blockDim.x >> 5, lane = threadIdx.x & 31;
  const int per = (row_vec + parts - 1) / parts;  // 16-byte vectors of one part of a row
  const int64_t n = (int64_t)R * parts;
  for (int64_t wi = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); wi < n;
       wi += (int64_t)gridDim.x * warps) {
    const int r = (int)(wi / parts), part = (int)(wi % parts);
    const int t = row_src[r] / k;
    const uint4* s = src + (size_t)t * row_vec;
    uint4* d = dst + (size_t)r * row_vec;
    const int v1 = min(row_vec, (part + 1) * per);
    int v = part * per + lane;
    for (; v + 96 < v1; v += 128) {  // four 16-byte loads in flight per lane
      const uint4 a = s[v], b = s[v + 32], c = s[v + 64], e4 = s[v + 96];
      d[v] = a;
      d[v + 32] = b;
      d[v + 64] = c;
      d[v + 96] = e4;
    }
    for (; v < v1; v += 32) d[v] = s[v];
    if (dscale && part == 0)
      for (int c = lane; c < scols; c += 32) dscale[(size_t)r * scols + c] = sscale[(size_t)t * scols + c];
  }
}

// Small batches (decode: R <= 2048 rows) split each row over four warps, so a
// row's loads go out in one round instead of four (the kernel sits between
// the permute and the FFN on the decode chain); large batches keep one warp
// per row.
cudaError_t launch_gather_rows(const int32_t* offsets, int E, const int32_t* row_src, int k,
                               int R_max, const void* src, void* dst, int row_bytes,
                               const float* sscale, float* dscale, cudaStream_t st, int scols) {
  if (R_max == 0) return cudaSuccess;
  const int parts = R_max <= 2048 ? 4 : 1;
  int64_t blocks = ((int64_t)R_max * parts + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  return launch_kernel(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, offsets, E,
                       row_src, k, R_max, (const uint4*)src, (uint4*)dst, row_bytes / 16, sscale,
                       dscale, scols, parts);
}

// ================================================================ silu_and_mul
__global__ void __launch_bounds__(256) silu_and_mul_kernel(const bf16* __restrict__ h, int R,
                                                           int I, bf16* __restrict__ a) {
  pdl_trigger();
  pdl_wait();
  const int vpr = I >> 3;  // 8-element vectors per output row
  const size_t n = (size_t)R * vpr;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / vpr, c = i % vpr;
    const uint4 g = reinterpret_cast<const uint4*>(h + r * 2 * I)[c];
    const uint4 u = reinterpret_cast<const uint4*>(h + r * 2 * I + I)[c];
    float gf[8], uf[8];
    unpack8_bf16(g, gf);
    unpack8_bf16(u, uf);
    uint4 o;
    o.x = pack2_bf16(silu_f(gf[0]) * uf[0], silu_f(gf[1]) * uf[1]);
    o.y = pack2_bf16(silu_f(gf[2]) * uf[2], silu_f(gf[3]) * uf[3]);
    o.z = pack2_bf16(silu_f(gf[4]) * uf[4], silu_f(gf[5]) * uf[5]);
    o.w = pack2_bf16(silu_f(gf[6]) * uf[6], silu_f(gf[7]) * uf[7]);
    reinterpret_cast<uint4*>(a + r * I)[c] = o;
  }
}

cudaError_t launch_silu_and_mul(const void* h, int R, int I, void* a, cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  size_t n = (size_t)R * (I / 8);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  return launch_kernel(silu_and_mul_kernel, dim3(blocks), dim3(256), 0, st, (const bf16*)h, R, I,
                       (bf16*)a);
}

// ===================================================================== combine
// out[t, :] = bf16( sum_j y_j ), fp32, j ascending, where y_j is row
// t*k + j of y (PAIR = true: rows in (token, slot) order, row_of_pair only
// marks skipped pairs with -1) or row row_of_pair[t*k + j] (PAIR = false:
// rows in expert order).  y is fp32 or bf16.  Each thread handles 8 columns.
template <bool YBF16, bool PAIR>
__global__ void __launch_bounds__(256) combine_kernel(const void* __restrict__ y,
                                                      const int32_t* __restrict__ row_of_pair,
                                                      int T, int k, int H, bf16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int h8 = blockIdx.x * blockDim.x + threadIdx.x;  // 8-column group
  if (h8 * 8 >= H) return;
  int rows[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) rows[j] = (j < k) ? row_of_pair[(size_t)t * k + j] : -1;
  float v[kMaxTopK][8];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {  // all loads first (up to 8 rows in flight)
    // in pair order the row address does not wait for the index load
    const int64_t row = PAIR ? (int64_t)t * k + j : (int64_t)rows[j];
    if (j < k && (PAIR || rows[j] >= 0)) {
      if (YBF16) {
        unpack8_bf16(reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(y) +
                                                    row * H)[h8], v[j]);
      } else {
        const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(y) +
                                                            row * H) + 2 * h8;
        const float4 a = src[0], b = src[1];
        v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
        v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[j][i] = 0.f;
    }
  }
  float s[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) s[i] = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {  // summed in j order, skipped pairs excluded
    if (j < k && rows[j] >= 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i] += v[j][i];
    }
  }
  uint4 o;
  o.x = pack2_bf16(s[0], s[1]);
  o.y = pack2_bf16(s[2], s[3]);
  o.z = pack2_bf16(s[4], s[5]);
  o.w = pack2_bf16(s[6], s[7]);
  reinterpret_cast<uint4*>(out + (size_t)t * H)[h8] = o;
}

// Persistent form for (token, slot)-ordered bf16 rows: each thread takes two
// (token, 8-column group) items per pass with all of their row loads in
// flight before any sum, and the grid strides over the items.
__global__ void __launch_bounds__(256) combine_pair_bf16_kernel(const bf16* __restrict__ y,
                                                                const int32_t* __restrict__ rop,
                                                                int T, int k, int H,
                                                                bf16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int g8 = H >> 3;
  const int64_t total = (int64_t)T * g8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 2 * stride) {
    uint4 raw[2][kMaxTopK];
    int valid[2][kMaxTopK];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t it = i0 + u * stride;
      const bool in = it < total;
      const int64_t t = in ? it / g8 : 0;
      const int64_t g = in ? it % g8 : 0;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        const bool use = in && j < k;
        valid[u][j] = use ? rop[t * k + j] : -1;
        raw[u][j] = use ? reinterpret_cast<const uint4*>(y + (t * k + j) * H)[g]
                        : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t it = i0 + u * stride;
      if (it >= total) break;
      float s[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i] = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {  // summed in j order, skipped pairs excluded
        if (j < k && valid[u][j] >= 0) {
          float f[8];
          unpack8_bf16(raw[u][j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) s[i] += f[i];
        }
      }
      uint4 o;
      o.x = pack2_bf16(s[0], s[1]);
      o.y = pack2_bf16(s[2], s[3]);
      o.z = pack2_bf16(s[4], s[5]);
      o.w = pack2_bf16(s[6], s[7]);
      reinterpret_cast<uint4*>(out)[it] = o;
    }
  }
}

cudaError_t launch_combine(const void* y, bool y_bf16, bool pair_order,
                           const int32_t* row_of_pair, int T, int k, int H, void* out,
                           cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (y_bf16 && pair_order) {
    const int64_t items = (int64_t)T * (H / 8);
    int64_t blocks = (items + 511) / 512;
    if (blocks > 152 * 4) blocks = 152 * 4;
    return launch_kernel(combine_pair_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                         (const bf16*)y, row_of_pair, T, k, H, (bf16*)out);
  }
  const int h8 = H / 8;
  dim3 grid((h8 + 255) / 256, T);
#define MOE_COMBINE(B, P) \
  return launch_kernel(combine_kernel<B, P>, grid, dim3(256), 0, st, y, row_of_pair, T, k, H, (bf16*)out)
  if (y_bf16) { if (pair_order) MOE_COMBINE(true, true); else MOE_COMBINE(true, false); }
  else { if (pair_order) MOE_COMBINE(false, true); else MOE_COMBINE(false, false); }
#undef MOE_COMBINE
}

// ========================================================== row E4M3 quantiser
// One warp per row: s = absmax / 448 (1 for a zero row); q = e4m3(x / s).
// Rows of up to 2048 columns stay in registers between the absmax and the
// quantisation (one read of x); longer rows are read twice.  Rows at or
// beyond *nrows_dev (when given) are skipped.
constexpr int kQuantRegVec = 8;  // 16-byte vectors per lane held in registers

MOE_DEV uint2 quant8_e4m3(const float (&f)[8], float s) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) lo |= (uint32_t)f_to_e4m3(__fdiv_rn(f[i], s)) << (8 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i) hi |= (uint32_t)f_to_e4m3(__fdiv_rn(f[4 + i], s)) << (8 * i);
  return make_uint2(lo, hi);
}

__global__ void __launch_bounds__(256) quant_rows_kernel(const bf16* __restrict__ x, int64_t rows,
                                                         int cols, uint8_t* __restrict__ q,
                                                         float* __restrict__ scale,
                                                         const int32_t* __restrict__ nrows_dev) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t nr = nrows_dev ? min(rows, (int64_t)*nrows_dev) : rows;
  const int nv = cols >> 3;
  const int64_t wpb = blockDim.x >> 5;
  for (int64_t r = blockIdx.x * wpb + (threadIdx.x >> 5); r < nr; r += (int64_t)gridDim.x * wpb) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * cols);
    uint2* qr = reinterpret_cast<uint2*>(q + r * cols);
    float amax = 0.f;
    if (nv <= 32 * kQuantRegVec) {
      uint4 buf[kQuantRegVec];
#pragma unroll
      for (int i = 0; i < kQuantRegVec; ++i) {
        const int v = lane + 32 * i;
        if (v < nv) {
          buf[i] = xr[v];
          float f[8];
          unpack8_bf16(buf[i], f);
#pragma unroll
          for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(f[t]));
        }
      }
      amax = warp_max(amax);
      const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
#pragma unroll
      for (int i = 0; i < kQuantRegVec; ++i) {
        const int v = lane + 32 * i;
        if (v < nv) {
          float f[8];
          unpack8_bf16(buf[i], f);
          qr[v] = quant8_e4m3(f, s);
        }
      }
      if (lane == 0) scale[r] = s;
    } else {
      for (int v = lane; v < nv; v += 32) {
        float f[8];
        unpack8_bf16(xr[v], f);
#pragma unroll
        for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(f[t]));
      }
      amax = warp_max(amax);
      const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      for (int v = lane; v < nv; v += 32) {
        float f[8];
        unpack8_bf16(xr[v], f);
        qr[v] = quant8_e4m3(f, s);
      }
      if (lane == 0) scale[r] = s;
    }
  }
}

cudaError_t launch_quant_rows(const void* x, int64_t rows, int cols, void* q, float* scale,
                              const int32_t* nrows_dev, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;  // eight rows (warps) per CTA
  if (blocks > 152 * 16) blocks = 152 * 16;
  return launch_kernel(quant_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, (const bf16*)x,
                       rows, cols, (uint8_t*)q, scale, nrows_dev);
}

}  // namespace moe
