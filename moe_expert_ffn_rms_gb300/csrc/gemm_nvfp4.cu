// NVFP4 expert weights for decode (W4A16).
//
// Format (the public NVFP4 layout): E2M1 codes, two per byte (element 2i in
// the low nibble), blocks of 16 consecutive K elements with one E4M3 scale
// each, one fp32 scale per expert matrix:  w = e2m1(q) * e4m3(s_b) * s_g.
// A code times its block scale has at most 5 significant bits and lies in
// [2^-10, 2688], so it is exact in fp16; activations are bf16 values, exact
// in fp16 within its range.  The FFN therefore runs tcgen05 kind::f16 MMAs on
// fp16 operands: dequantising warps turn each TMA-staged FP4 tile (128-byte
// swizzled rows, so that a warp's row reads spread over the banks) into fp16
// rows (cvt.rn.f16x2.e2m1x2, then one f16x2 multiply by the block scale) and
// store them into tensor memory, from where the MMA reads its A operand; the
// fp16 tile, 3.5 times the bytes of its codes, never passes through shared
// memory.  The fp32 matrix scale is applied in the epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "engine.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

// ------------------------------------------------------------ quantiser --
// One expert matrix [N, K] per blockIdx.y: the absmax, as the fp32 bit
// pattern (non-negative floats order like their bits), by atomicMax.
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const bf16* __restrict__ w, int64_t nk,
                                                         unsigned* __restrict__ amax_bits) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const bf16* m = w + (size_t)blockIdx.y * nk;
  float a = 0.f;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < nk;
       i += (int64_t)gridDim.x * blockDim.x * 8) {
    float f[8];
    unpack8_bf16(*reinterpret_cast<const uint4*>(m + i), f);
#pragma unroll
    for (int q = 0; q < 8; ++q) a = fmaxf(a, fabsf(f[q]));
  }
  a = block_max(a, red);
  if (threadIdx.x == 0) atomicMax(amax_bits + blockIdx.y, __float_as_uint(a));
}

// s_g = amax / (448 * 6), 1 for a zero matrix (in place over the bits).
__global__ void nvfp4_global_scale_kernel(unsigned* amax_bits, int M) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const float a = __uint_as_float(amax_bits[m]);
  const float sg = a > 0.f ? __fdiv_rn(a, 2688.0f) : 1.0f;
  reinterpret_cast<float*>(amax_bits)[m] = sg;
}

// E2M1 code of x: nearest-even, saturating to +-6 (from the format's value
// grid 0, 0.5, 1, 1.5, 2, 3, 4, 6; each boundary is a midpoint and goes to
// the neighbour with mantissa bit 0).
MOE_DEV uint32_t f_to_e2m1(float x) {
  const float a = fabsf(x);
  uint32_t c;
  if (a <= 0.25f) c = 0;
  else if (a < 0.75f) c = 1;
  else if (a <= 1.25f) c = 2;
  else if (a < 1.75f) c = 3;
  else if (a <= 2.5f) c = 4;
  else if (a < 3.5f) c = 5;
  else if (a <= 5.0f) c = 6;
  else c = 7;
  return c | (signbit(x) ? 8u : 0u);
}

// One thread per (matrix, row, block of 16): s_b = e4m3(amax_b / (6 s_g)),
// q = e2m1(w / (s_b s_g)), each step rounded to fp32.
__global__ void __launch_bounds__(256) nvfp4_quant_kernel(const bf16* __restrict__ w, int64_t nblk_per_mat,
                                                          const float* __restrict__ sg_m,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ sb) {
  pdl_trigger();
  pdl_wait();
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = nblk_per_mat * gridDim.y;
  const int64_t gb = (int64_t)blockIdx.y * nblk_per_mat + b;
  if (b >= nblk_per_mat || gb >= total) return;
  const float sg = sg_m[blockIdx.y];
  float f[16];
  unpack8_bf16(*reinterpret_cast<const uint4*>(w + gb * 16), f);
  unpack8_bf16(*reinterpret_cast<const uint4*>(w + gb * 16 + 8), f + 8);
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(f[i]));
  const float six_sg = __fmul_rn(6.0f, sg);
  const uint8_t code = f_to_e4m3(__fdiv_rn(a, six_sg));
  sb[gb] = code;
  const float scale = __fmul_rn(e4m3_to_f(code), sg);
  uint32_t lo = 0, hi = 0;
  if (scale > 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) lo |= f_to_e2m1(__fdiv_rn(f[i], scale)) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) hi |= f_to_e2m1(__fdiv_rn(f[8 + i], scale)) << (4 * i);
  }
  reinterpret_cast<uint2*>(q)[gb] = make_uint2(lo, hi);
}

// ------------------------------------------------------- fp16 row gather --
// xp[r] = fp16(x_hat[row_src[r] / k]) for r < offsets[E] (exact: bf16 values
// inside fp16's range), one warp per row.
__global__ void __launch_bounds__(256) gather_rows_f16_kernel(const int32_t* __restrict__ offsets,
                                                              int E, const int32_t* __restrict__ row_src,
                                                              int k, int R_max, int H,
                                                              const bf16* __restrict__ src,
                                                              __half* __restrict__ dst) {
  pdl_trigger();
  pdl_wait();
  const int R = min(offsets[E], R_max);
  const int warps = blockDim.x >> 5, lane = threadIdx.x & 31;
  const int nv = H >> 3;
  for (int r = blockIdx.x * warps + (threadIdx.x >> 5); r < R; r += gridDim.x * warps) {
    const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)(row_src[r] / k) * H);
    uint4* d = reinterpret_cast<uint4*>(dst + (size_t)r * H);
    for (int v = lane; v < nv; v += 32) {
      float f[8];
      unpack8_bf16(s[v], f);
      __half2 h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      d[v] = *reinterpret_cast<uint4*>(h);
    }
  }
}

// ------------------------------------------------------- fused FFN kernel --
constexpr int kNvThreads = 480;   // warp 0 TMA, 1 MMA, 2-5 epilogue, 6-13 dequantise, 14 MMA
// MMA issuers: warp 1, then warp 14.  With the issue warp-uniform, a third
// issuer (one more accumulator bank for the epilogue to add) was slower.
constexpr int kMaxIssuersNv = 2;
constexpr int kDqWarps = 8;       // two per TMEM lane quarter: each takes two of a stage's four atoms
constexpr int kKStage = 256;      // K elements per stage: 128 B of codes, 16 B of scales per row
constexpr int kRowsNv = 128;      // weight rows per unit (MMA M)
constexpr int kFp4Bytes = kRowsNv * (kKStage / 2);   // 16 KB
constexpr int kSbBytes = kRowsNv * (kKStage / 16);   // 2 KB
constexpr int kMaxStagesNv = 8;
constexpr int kBoxRowsNv = 16;    // token rows per TMA box
constexpr int kRingNv = 4;        // claimed-unit slots
constexpr int kMaxChunkNv = 64;   // token rows per unit (MMA N)
// TMEM columns: two fp32 accumulators of kMaxChunkNv columns (each split
// into one bank of chunk columns per MMA issuer), then kASlots
// slots of one stage's fp16 A (128 lanes x 256 K elements = 128 columns: four
// 64-element atoms of 32 columns).  The dequantising warps and the MMA hand
// over whole stages, so each side waits on one barrier per stage.
constexpr int kAccColsNv = kMaxChunkNv;
constexpr int kACol0 = 2 * kAccColsNv;
constexpr int kAColsPerAtom = 32;
constexpr int kAColsPerStage = 4 * kAColsPerAtom;
constexpr int kASlots = 3;
constexpr int kTmemColsNv = 512;  // >= kACol0 + kASlots * kAColsPerStage, a power of two
constexpr int kSmemLimitNv = 227 * 1024;
static_assert(kACol0 + kASlots * kAColsPerStage <= kTmemColsNv, "TMEM budget");
// an issuer's own previous stage must be at least kASlots back for its A-slot
// waits to stay in order (see the MMA issuers)
static_assert(kMaxIssuersNv <= kASlots, "A slots per issuer");

struct NvJob {
  const float* sg;          // [E] fp32 matrix scales
  const int32_t* row_src;
  const float* topk_w;      // FC2: routing weight of pair row_src[r]
  void* out;                // FC1: fp16 [R, I]; FC2: bf16 [R, H], row r at row_src[r]
  int N_w;                  // weight rows per expert
  int n_out;                // output columns
  int nt;                   // N slices per (expert, token chunk)
  int kst;                  // K stages
};

// Every stage is three TMA loads (the per-load issue cost, not the bytes,
// bounded the first versions): one 3D box of all four 64-element atoms of
// the token rows, one 3D box of the unit's two 64-row weight slices of codes
// (FC1: gate rows and the matching up rows, I rows apart; FC2: 64 + 64
// consecutive rows), one of their block scales.
MOE_DEV void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int x, int y, int z,
                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// 16 accumulator columns at taddr summed over the nclass stage classes:
// class c (c = 0, 1, .. in that order) is in bank (first + c) mod ni, which
// lies b * chunk columns further for bank b.
MOE_DEV void load_acc16(uint32_t taddr, int chunk, int ni, int first, int nclass, float* v) {
  tmem_ld16(taddr + first * chunk, v);
  tmem_ld_wait();
  for (int c = 1; c < nclass; ++c) {
    int b = first + c;
    if (b >= ni) b -= ni;
    float w[16];
    tmem_ld16(taddr + b * chunk, w);
    tmem_ld_wait();
#pragma unroll
    for (int t = 0; t < 16; ++t) v[t] += w[t];
  }
}

struct NvParams {
  const int32_t* offsets;
  int E, I, R_max;
  int chunk;                // token rows per unit (a multiple of 16, <= 64)
  int stages, stage_bytes, b_bytes;  // ring: [B: 4 atoms x chunk rows x 128 B][codes][scales]
  int* sched;               // [0] unit counter, [1 + e] finished FC1 epilogue warps of e
  int* status;
  NvJob job[2];
};

// Four E2M1 code pairs (one 32-bit word, element 2i in the low nibble of
// byte i) -> four f16x2 times the block scale s2 (exact products).
MOE_DEV void e2m1x8_scaled(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n .reg .b32 t0, t1, t2, t3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 t0, b0;\n cvt.rn.f16x2.e2m1x2 t1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 t2, b2;\n cvt.rn.f16x2.e2m1x2 t3, b3;\n"
      " mul.rn.f16x2 %0, t0, %5;\n mul.rn.f16x2 %1, t1, %5;\n"
      " mul.rn.f16x2 %2, t2, %5;\n mul.rn.f16x2 %3, t3, %5;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w), "r"(s2));
}

// The four E4M3 block scales of a 32-bit word, each as an fp16 pair (both
// halves the scale): two paired conversions and four byte permutes.
MOE_DEV void e4m3x4_to_h2(uint32_t w, uint32_t (&bs)[4]) {
  asm("{\n .reg .b16 lo, hi;\n .reg .b32 h01, h23;\n mov.b32 {lo, hi}, %4;\n"
      " cvt.rn.f16x2.e4m3x2 h01, lo;\n cvt.rn.f16x2.e4m3x2 h23, hi;\n"
      " prmt.b32 %0, h01, 0, 0x1010;\n prmt.b32 %1, h01, 0, 0x3232;\n"
      " prmt.b32 %2, h23, 0, 0x1010;\n prmt.b32 %3, h23, 0, 0x3232;\n}"
      : "=r"(bs[0]), "=r"(bs[1]), "=r"(bs[2]), "=r"(bs[3])
      : "r"(w));
}

__global__ void __launch_bounds__(kNvThreads, 1) moe_tc_nvfp4_kernel(
    const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_s0,
    const __grid_constant__ CUtensorMap tm_q1, const __grid_constant__ CUtensorMap tm_s1,
    const __grid_constant__ CUtensorMap tm_b0, const __grid_constant__ CUtensorMap tm_b1,
    const NvParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_up[2][kMaxExperts + 1];
  __shared__ __align__(8) uint64_t sfull[kMaxStagesNv];
  __shared__ __align__(8) uint64_t sempty[kMaxStagesNv];
  __shared__ __align__(8) uint64_t afull[kASlots];
  __shared__ __align__(8) uint64_t aempty[kASlots];
  __shared__ __align__(8) uint64_t tfull[2];
  __shared__ __align__(8) uint64_t tempty[2];
  __shared__ __align__(8) uint64_t ufull[kRingNv];
  __shared__ __align__(8) uint64_t uempty[kRingNv];
  __shared__ __align__(8) uint64_t drain_bar[kMaxIssuersNv];
  __shared__ __align__(8) uint64_t xch_bar;
  __shared__ int s_uring[kRingNv];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_xch[64 * 17];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~(uintptr_t)1023);
  // ni MMA issuers, issuer b summing the K stages n = b (mod ni) into its
  // own bank of chunk columns: as many as fit an accumulator, at most
  // kMaxIssuersNv and at most the ring's stages
  int ni = kAccColsNv / p.chunk;
  ni = ni < kMaxIssuersNv ? ni : kMaxIssuersNv;
  ni = ni < p.stages ? ni : p.stages;
  const int mma_par = warp == 1 ? 0 : (warp >= 14 ? warp - 13 : -1);  // issuer index

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 1 + kDqWarps * 32);  // the MMA commit (B read) + every dequantiser
    }
    for (int q = 0; q < kASlots; ++q) {
      mbar_init(&afull[q], kDqWarps * 32);
      mbar_init(&aempty[q], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], ni);  // a commit of each active issuer
      mbar_init(&tempty[a], 128);
    }
    for (int i = 0; i < kRingNv; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], kMaxIssuersNv + 4 + kDqWarps);  // MMA threads, epilogue, dequantisers
    }
    for (int b = 0; b < kMaxIssuersNv; ++b) mbar_init(&drain_bar[b], 1);
    mbar_init(&xch_bar, 128);
    s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q0);
    prefetch_tmap(&tm_s0);
    prefetch_tmap(&tm_q1);
    prefetch_tmap(&tm_s1);
    prefetch_tmap(&tm_b0);
    prefetch_tmap(&tm_b1);
  } else if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemColsNv);
    tmem_relinquish();
  }
  pdl_trigger();
  pdl_wait();
  for (int e = threadIdx.x; e <= p.E; e += blockDim.x) s_off[e] = p.offsets[e];
  __syncthreads();
  if (threadIdx.x == 0) {  // offsets must be monotone within [0, R_max]
    int prev = 0;
    bool bad = false;
    for (int e = 0; e <= p.E; ++e) {
      int v = s_off[e];
      if (v < prev || v > p.R_max || (e == 0 && v != 0)) {
        bad = true;
        v = v < prev ? prev : (v > p.R_max ? p.R_max : v);
        if (e == 0) v = 0;
      }
      s_off[e] = v;
      prev = v;
    }
    if (bad && blockIdx.x == 0) flag_status(p.status, MOE_ERR_INVALID_ARG);
  }
  __syncthreads();
  if (warp < 2) {  // warp jb builds job jb's unit prefix
    const int nt = p.job[warp].nt;
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      const int cnt = (e < p.E) ? s_off[e + 1] - s_off[e] : 0;
      const int v = ((cnt + p.chunk - 1) / p.chunk) * nt;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < p.E) s_up[warp][e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_up[warp][p.E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int U0 = s_up[0][p.E];
  const int U = U0 + s_up[1][p.E];

  auto decode_unit = [&](int u) -> Unit {
    if (u >= U0) {
      Unit un = unit_of(u - U0, s_off, s_up[1], p.E, p.job[1].nt, p.chunk);
      un.job = 1;
      return un;
    }
    return unit_of(u, s_off, s_up[0], p.E, p.job[0].nt, p.chunk);
  };
  auto next_unit = [&](int i) -> int {
    const int slot = i % kRingNv;
    if (!mbar_wait(&ufull[slot], (uint32_t)((i / kRingNv) & 1), &s_abort)) return -2;
    return s_uring[slot];
  };

  if (warp == 0) {
    // ===================================================== TMA producer
    // The whole warp runs the loop and waits; lane 0 claims the units, waits
    // for FC1's rows and issues the loads.
    const uint64_t pol_w = l2_policy_evict_first();  // weights: streamed once
    const uint64_t pol_x = l2_policy_evict_last();
    int s = 0;
    uint32_t ph = 0;
    uint32_t armed = 0, armed_ph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int slot = i % kRingNv;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&uempty[slot], (uint32_t)(((i / kRingNv) & 1) ^ 1), &s_abort))) {
        ok = false;
        break;
      }
      int u = 0;
      if (lane == 0) {
        u = atomicAdd(p.sched, 1);
        if (u >= U) u = -1;
        s_uring[slot] = u;
        mbar_arrive(&ufull[slot]);
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u < 0) break;
      const Unit un = decode_unit(u);
      const NvJob& j = p.job[un.job];
      if (un.job == 1) {
        // FC2 of expert e reads its FC1 rows: wait until every FC1 epilogue
        // warp of e has published them (FC1 units are all claimed first)
        int fok = 1;
        if (lane == 0) {
          const int cnt = s_off[un.e + 1] - s_off[un.e];
          const int need = ((cnt + p.chunk - 1) / p.chunk) * p.job[0].nt * 4;
          const int* flag = p.sched + 1 + un.e;
          const long long t0 = clock64();
          while (ld_acquire(flag) < need) {
            if (s_abort || clock64() - t0 > kSpinLimitCycles) {
              s_abort = 1;
              fok = 0;
              break;
            }
          }
          if (fok) fence_proxy_async_global();
        }
        if (!__shfl_sync(0xffffffffu, fok, 0)) {
          ok = false;
          break;
        }
      }
      // all chunk token rows are loaded (rows of other experts or past the
      // end are ignored by the epilogue; the box is zero-filled past R_max)
      const uint32_t tx = (uint32_t)(kFp4Bytes + kSbBytes + p.b_bytes);
      const CUtensorMap* tq = un.job ? &tm_q1 : &tm_q0;
      const CUtensorMap* ts = un.job ? &tm_s1 : &tm_s0;
      const CUtensorMap* tb = un.job ? &tm_b1 : &tm_b0;
      // FC1: 64 gate rows and the matching 64 up rows (the map's third
      // dimension steps I rows); FC2: 128 consecutive rows (steps of 64)
      const int r0 = un.e * j.N_w + (un.job == 0 ? un.nt * 64 : un.nt * 128);
      for (int ks = 0; ks < j.kst; ++ks) {
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(&sempty[s], ph ^ 1, &s_abort))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&sfull[s], tx);
          uint8_t* st = ring + (size_t)s * p.stage_bytes;
          uint8_t* codes = st + p.b_bytes;
          uint8_t* scales = codes + kFp4Bytes;
          tma_load_3d(codes, tq, &sfull[s], ks * (kKStage / 2), r0, 0, pol_w);
          tma_load_3d(scales, ts, &sfull[s], ks * (kKStage / 16), r0, 0, pol_w);
          tma_load_3d(st, tb, &sfull[s], 0, un.row0, ks * 4, pol_x);
        }
        __syncwarp();
        armed |= 1u << s;
        armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
        if (++s == p.stages) { s = 0; ph ^= 1; }
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, producer_tail(sempty, p.stages, s, ph, &s_abort));
    if (!ok && lane == 0) {
      flag_status(p.status, MOE_ERR_TIMEOUT);
      drain_armed(sfull, p.stages, armed, armed_ph);
    }
  } else if (mma_par >= 0) {
    // ===================================================== MMA issuers
    // Issuer b takes the CTA's K stages n = b (mod ni), counted over all
    // units, into its own bank.  A stage ring slot and an A slot pass between
    // the issuers, but every wait stays in order: an issuer reaches stage n
    // only after its own stage n - ni, so the loads and conversions up to
    // n - ni (in order) are done, and ni <= min(stages, kASlots) means no
    // barrier it waits on can be a whole phase behind; none can be a phase
    // ahead, since that needs this issuer's own stage n released.  Issuers
    // past ni only follow the units.  The whole warp runs the loop and
    // waits; one elected lane issues.
    {
      const int par = mma_par;
      int s = 0, q = 0, acc = 0;
      uint32_t ph = 0, qph = 0, aph = 0, n = 0;
      bool ok = true;
      bool issued = false;
      for (int i = 0; ok; ++i) {
        const int u = __shfl_sync(0xffffffffu, next_unit(i), 0);  // every lane has read it
        if (u == -2) { ok = false; break; }
        if (lane == 0) mbar_arrive(&uempty[i % kRingNv]);
        if (u < 0) break;
        const Unit un = decode_unit(u);
        const int kst = p.job[un.job].kst;
        if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], aph ^ 1, &s_abort))) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * kAccColsNv + par * p.chunk;
        const uint32_t idesc = make_idesc(((un.rows + 15) / 16) * 16, 0u);  // fp16 A and B
        bool first = true;  // this issuer's first stage of the unit starts its sum
        for (int ks = 0; ks < kst && ok; ++ks, ++n) {
          if ((int)(n % (uint32_t)ni) == par) {
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(&sfull[s], ph, &s_abort) &&
                                             mbar_wait_sleep(&afull[q], qph, &s_abort))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t b0 = smem_u32(ring + (size_t)s * p.stage_bytes);
            const uint32_t a0 = tmem + kACol0 + q * kAColsPerStage;
            if (elect_one()) {
              for (int a = 0; a < 4; ++a) {
                const uint32_t bb = b0 + a * p.chunk * 128;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // four 16-element K steps (8 columns) per atom
                  const uint32_t accum = (!first || a || kk) ? 1u : 0u;
                  mma_f16_ts(d, a0 + a * kAColsPerAtom + kk * 8, sw128_desc(bb + kk * 32), idesc,
                             accum);
                }
              }
              mma_commit(&aempty[q]);
              mma_commit(&sempty[s]);
            }
            __syncwarp();
            first = false;
            issued = true;
          }
          if (++q == kASlots) { q = 0; qph ^= 1; }
          if (++s == p.stages) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        if (par < ni) {
          if (elect_one()) mma_commit(&tfull[acc]);
          __syncwarp();
        }
        if (++acc == 2) { acc = 0; aph ^= 1; }
      }
      if (ok) ok = __all_sync(0xffffffffu, accumulator_tail(tempty, acc, aph, &s_abort));
      if (!ok && lane == 0) flag_status(p.status, MOE_ERR_TIMEOUT);
      if (issued) {
        if (elect_one()) mma_commit(&drain_bar[par]);
        __syncwarp();
        if (lane == 0) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&drain_bar[par], 0) && clock64() - t0 < kSpinLimitCycles) {
          }
        }
        __syncwarp();
      }
    }
  } else if (warp < 6) {
    // ======================================================== epilogue
    // TMEM lane = weight row of the unit's slice, columns = its token rows.
    const int qw = warp & 3;
    const int lrow = qw * 32 + lane;
    int acc = 0;
    uint32_t aph = 0, xph = 0, n0 = 0;
    for (int i = 0;; ++i) {
      const int u = next_unit(i);
      __syncwarp();
      if (lane == 0 && u != -2) mbar_arrive(&uempty[i % kRingNv]);
      if (u == -2) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      if (u < 0) break;
      const Unit un = decode_unit(u);
      const NvJob& j = p.job[un.job];
      // the unit's stages ks = c (mod ni) are in bank (n0 + c) mod ni; the
      // epilogue adds the classes c = 0, 1, .. in that order, so the sum does
      // not depend on where the unit fell in the CTA's stage count (which
      // the dynamic unit claims change from run to run)
      const int kst = j.kst;
      const int bank_first = (int)(n0 % (uint32_t)ni);
      const int nclass = kst < ni ? kst : ni;
      n0 += (uint32_t)kst;
      if (!mbar_wait(&tfull[acc], aph, &s_abort)) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + acc * kAccColsNv + ((uint32_t)(qw * 32) << 16);
      const float sg = j.sg[un.e];
      const int ncols = ((un.rows + 15) / 16) * 16;
      bool ok = true;
      if (un.job == 0) {
        // lanes 0..63 gate rows, 64..127 the matching up rows of slice nt
        const bool is_gate = lrow < 64;
        const int n = un.nt * 64 + (lrow & 63);
        for (int c = 0; c < ncols && ok; c += 16) {
          float v[16];
          load_acc16(tbase + c, p.chunk, ni, bank_first, nclass, v);
          if (!is_gate) {
#pragma unroll
            for (int t = 0; t < 16; ++t) s_xch[(lrow - 64) * 17 + t] = v[t] * sg;
          }
          mbar_arrive(&xch_bar);
          if (!mbar_wait(&xch_bar, xph, &s_abort)) { ok = false; break; }
          xph ^= 1;
          if (is_gate && n < p.I) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              if (c + t < un.rows) {
                const int r = un.row0 + c + t;
                const float g = v[t] * sg;
                const float a = bf16_round_f(silu_f(g) * s_xch[lrow * 17 + t]);
                reinterpret_cast<__half*>(j.out)[(size_t)r * j.n_out + n] = __float2half_rn(a);
              }
            }
          }
          mbar_arrive(&xch_bar);
          if (!mbar_wait(&xch_bar, xph, &s_abort)) { ok = false; break; }
          xph ^= 1;
        }
      } else {
        const int n = un.nt * 128 + lrow;
        for (int c = 0; c < ncols; c += 16) {
          float v[16];
          load_acc16(tbase + c, p.chunk, ni, bank_first, nclass, v);
          if (n < j.n_out) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              if (c + t < un.rows) {
                const int r = un.row0 + c + t;
                const int orow = j.row_src[r];
                const float x = v[t] * sg * j.topk_w[orow];
                reinterpret_cast<bf16*>(j.out)[(size_t)orow * j.n_out + n] = __float2bfloat16_rn(x);
              }
            }
          }
        }
      }
      if (!ok) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) { acc = 0; aph ^= 1; }
      if (un.job == 0) {
        // publish this warp's FC1 rows to the TMA readers of FC2
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.sched + 1 + un.e, 1);
      }
    }
  } else {
    // ================================================ dequantising warps
    // Warp w (6..13) owns weight rows r = 32 (w % 4) + lane of the unit's
    // 128-row slice (its TMEM lane quarter) and atoms 2h, 2h + 1 (h = (w - 6)
    // / 4) of every stage: per 64-element atom a thread reads 32 B of codes
    // (rows are 128-byte swizzled: 16-byte chunk c of row r sits at chunk
    // c ^ (r % 8)) and one block scale per 16 elements, and stores its 64 fp16
    // values into 32 TMEM columns of atom a of stage slot n % kASlots, n = the
    // stage count.  The loop is bound by instruction issue, so the slot and
    // its phase are running counters and each thread loads only the 8 bytes
    // of block scales of its two atoms.
    const int qtr = warp & 3;
    const int half = (warp - 6) >> 2;
    const int r = qtr * 32 + lane;
    const uint32_t tlane = (uint32_t)(qtr * 32) << 16;
    const uint32_t c_off0 = (uint32_t)r * (kKStage / 2) + (((4 * half) ^ (r & 7)) << 4);
    const uint32_t c_off1 = (uint32_t)r * (kKStage / 2) + (((4 * half + 1) ^ (r & 7)) << 4);
    const uint32_t c_off2 = (uint32_t)r * (kKStage / 2) + (((4 * half + 2) ^ (r & 7)) << 4);
    const uint32_t c_off3 = (uint32_t)r * (kKStage / 2) + (((4 * half + 3) ^ (r & 7)) << 4);
    const uint32_t s_off8 = (uint32_t)kFp4Bytes + (uint32_t)r * (kKStage / 16) + 8u * half;
    int s = 0, slot = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int u = next_unit(i);
      __syncwarp();
      if (lane == 0 && u != -2) mbar_arrive(&uempty[i % kRingNv]);
      if (u == -2) { ok = false; break; }
      if (u < 0) break;
      const Unit un = decode_unit(u);
      const int kst = p.job[un.job].kst;
      for (int ks = 0; ks < kst; ++ks) {
        // every lane waits for the staged codes and a free A slot, and every
        // lane arrives below: the stage loop has no divergent branch
        if (!__all_sync(0xffffffffu, mbar_wait_spin(&sfull[s], ph, &s_abort) &&
                                         mbar_wait_spin(&aempty[slot], aph ^ 1, &s_abort))) {
          ok = false;
          break;
        }
        const uint8_t* st = ring + (size_t)s * p.stage_bytes + p.b_bytes;
        const uint2 scales = *reinterpret_cast<const uint2*>(st + s_off8);
        uint32_t v[64];  // the warp's two atoms: 64 adjacent TMEM columns
#pragma unroll
        for (int aa = 0; aa < 2; ++aa) {
          const uint32_t swa = aa ? scales.y : scales.x;
          const uint4 c0 = *reinterpret_cast<const uint4*>(st + (aa ? c_off2 : c_off0));
          const uint4 c1 = *reinterpret_cast<const uint4*>(st + (aa ? c_off3 : c_off1));
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint32_t bs[4];
          e4m3x4_to_h2(swa, bs);
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // word c = elements 8c .. 8c + 7, block c / 2
            uint32_t o[4];
            e2m1x8_scaled(w[c], bs[c >> 1], o);
#pragma unroll
            for (int t = 0; t < 4; ++t) v[32 * aa + 4 * c + t] = o[t];
          }
        }
        tmem_st64(tmem + tlane + kACol0 + slot * kAColsPerStage + 2 * half * kAColsPerAtom, v);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&afull[slot]);
        mbar_arrive(&sempty[s]);
        if (++s == p.stages) { s = 0; ph ^= 1; }
        if (++slot == kASlots) { slot = 0; aph ^= 1; }
      }
    }
    // tail: the MMAs have released every A slot before the CTA exits
    for (int i = 0; ok && i < kASlots; ++i) {
      ok = mbar_wait(&aempty[slot], aph ^ 1, &s_abort);
      if (++slot == kASlots) { slot = 0; aph ^= 1; }
    }
    if (!ok) flag_status(p.status, MOE_ERR_TIMEOUT);
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemColsNv);
}

}  // namespace

// ------------------------------------------------------------------ host --
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode3 = nullptr;
std::once_flag g_encode3_once;

void load_encode3() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode3 = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// 3D tensor map: extents e0 (contiguous), e1, e2; byte strides s1, s2 of
// dimensions 1 and 2; box b0 x b1 x b2, zero fill out of range.
bool encode_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t e0,
                   uint64_t e1, uint64_t e2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1,
                   uint32_t b2, CUtensorMapSwizzle sw) {
  std::call_once(g_encode3_once, load_encode3);
  if (!g_encode3) return false;
  cuuint64_t dims[3] = {e0, e1, e2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode3(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const void* w, int M, int N, int K, uint8_t* q, uint8_t* sb,
                                  float* sg, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (K % 16 != 0) return cudaErrorInvalidValue;
  const int64_t nk = (int64_t)N * K;
  cudaError_t e = cudaMemsetAsync(sg, 0, (size_t)M * sizeof(float), st);
  if (e != cudaSuccess) return e;
  int bx = (int)((nk / 8 + 255) / 256);
  if (bx > 256) bx = 256;
  e = launch_kernel(nvfp4_amax_kernel, dim3(bx, M), dim3(256), 0, st, (const bf16*)w, nk,
                    reinterpret_cast<unsigned*>(sg));
  if (e != cudaSuccess) return e;
  e = launch_kernel(nvfp4_global_scale_kernel, dim3((M + 255) / 256), dim3(256), 0, st,
                    reinterpret_cast<unsigned*>(sg), M);
  if (e != cudaSuccess) return e;
  const int64_t nblk = nk / 16;
  return launch_kernel(nvfp4_quant_kernel, dim3((unsigned)((nblk + 255) / 256), M), dim3(256), 0,
                       st, (const bf16*)w, nblk, (const float*)sg, q, sb);
}

cudaError_t launch_gather_rows_f16(const int32_t* offsets, int E, const int32_t* row_src, int k,
                                   int R_max, int H, const void* src, void* dst, cudaStream_t st) {
  if (R_max == 0) return cudaSuccess;
  int blocks = (R_max + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  return launch_kernel(gather_rows_f16_kernel, dim3(blocks), dim3(256), 0, st, offsets, E, row_src,
                       k, R_max, H, (const bf16*)src, (__half*)dst);
}

bool nvfp4_decode_covers(int H, int I, int E) {
  return H % kKStage == 0 && I % kKStage == 0 && E <= kMaxExperts;
}

cudaError_t launch_decode_ffn_nvfp4(const void* xp, const uint8_t* w13_q, const uint8_t* w13_sb,
                                    const float* w13_sg, const uint8_t* w2_q, const uint8_t* w2_sb,
                                    const float* w2_sg, void* act, void* y, const int32_t* offsets,
                                    const int32_t* row_src, const float* topk_w, int* sched, int E,
                                    int H, int I, int R_max, int T, int sms, int* status,
                                    cudaStream_t st) {
  if (R_max == 0) return cudaSuccess;
  if (!nvfp4_decode_covers(H, I, E) || !sched) return cudaErrorNotSupported;
  NvParams p{};
  p.offsets = offsets;
  p.E = E;
  p.I = I;
  p.R_max = R_max;
  // token rows per unit: up to 64, so that at least three stages fit
  int chunk = T < kMaxChunkNv ? T : kMaxChunkNv;
  chunk = ((chunk < 1 ? 1 : chunk) + kBoxRowsNv - 1) / kBoxRowsNv * kBoxRowsNv;
  p.chunk = chunk;
  p.sched = sched;
  p.status = status;
  p.b_bytes = 4 * chunk * 128;
  p.stage_bytes = p.b_bytes + kFp4Bytes + kSbBytes;
  const int static_smem = 10 * 1024;
  int stages = (kSmemLimitNv - static_smem - 1024) / p.stage_bytes;
  if (stages > kMaxStagesNv) stages = kMaxStagesNv;
  if (stages < 2) return cudaErrorNotSupported;
  p.stages = stages;
  const size_t smem = 1024 + (size_t)stages * p.stage_bytes;
  // job 0: FC1 + silu_and_mul, fp16 rows [R, I]; job 1: FC2 + routing weight, bf16 rows at row_src
  p.job[0] = NvJob{w13_sg, row_src, nullptr, act, 2 * I, I, I / 64, H / kKStage};
  p.job[1] = NvJob{w2_sg, row_src, topk_w, y, H, H, (H + 127) / 128, I / kKStage};
  // maps[0..3]: FC1 codes, FC1 scales, FC2 codes, FC2 scales as [half][64
  // rows][K bytes] boxes; maps[4..5]: token rows as [atom][chunk rows][64
  // fp16 elements] boxes
  CUtensorMap m[6];
  const uint64_t rows13 = (uint64_t)E * 2 * I, rows2 = (uint64_t)E * H;
  if (!encode_map_3d(&m[0], w13_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, H / 2, rows13, 2, H / 2,
                     (uint64_t)I * (H / 2), kKStage / 2, 64, 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_3d(&m[1], w13_sb, CU_TENSOR_MAP_DATA_TYPE_UINT8, H / 16, rows13, 2, H / 16,
                     (uint64_t)I * (H / 16), kKStage / 16, 64, 2, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_map_3d(&m[2], w2_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, I / 2, rows2, 2, I / 2,
                     (uint64_t)64 * (I / 2), kKStage / 2, 64, 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_3d(&m[3], w2_sb, CU_TENSOR_MAP_DATA_TYPE_UINT8, I / 16, rows2, 2, I / 16,
                     (uint64_t)64 * (I / 16), kKStage / 16, 64, 2, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_map_3d(&m[4], xp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 64, (uint64_t)R_max, H / 64,
                     (uint64_t)H * 2, 128, 64, chunk, 4, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_3d(&m[5], act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 64, (uint64_t)R_max, I / 64,
                     (uint64_t)I * 2, 128, 64, chunk, 4, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(moe_tc_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_tc_nvfp4_kernel, dim3(sms), dim3(kNvThreads), smem, st, m[0], m[1], m[2],
                       m[3], m[4], m[5], p);
}

}  // namespace moe
