// Block-wise FP8 expert weights with per-group activation scales (W8A8).
//
// Format: E4M3 codes; each 128 x 128 tile of an expert matrix W [N, K] has
// one fp32 scale s_w (absmax / 448), and each group of 128 consecutive K
// elements of an activation row has one fp32 scale s_a.  The product is
//   y[r, n] = sum over K groups g of  s_a[r, g] * s_w[n / 128, g] * (q_a[r, g] . q_w[n, g]),
// i.e. the scales change every 128 K elements, so they cannot be applied
// once after the whole dot product as with per-channel scales.
//
// Design.  The tensor cores compute each 128-wide K group on its own: the MMA
// thread writes the group's E4M3 x E4M3 product (fp32, four K = 32 steps of
// tcgen05 kind::f8f6f4) into a fresh TMEM slot of a ring of up to 16, and four
// epilogue warps fold each slot into fp32 registers with the group's two
// scales (one per weight tile, one per token column), then hand the slot
// back.  The MMA never waits for the fold unless every slot is full, and the
// TMA ring behind it keeps streaming weights.
//
// A unit is 256 weight rows x up to 64 token rows of one expert: FC1 takes
// the 128 gate rows and the matching 128 up rows of one 128-column slice of
// the intermediate (one TMEM lane, and so one epilogue thread, holds g and u
// of the same column), FC2 two consecutive 128-row slices of W2.  FC1's epilogue forms a = bf16(silu(g) u)
// for 128 consecutive intermediate columns, which is exactly one K group of
// FC2, so it quantises them in place: group absmax over the 128 lanes, one
// scale per token row, E4M3 codes.  FC2's epilogue multiplies by the routing
// weight and writes bf16 rows in (token, slot) order.  FC1 and FC2 share one
// persistent launch with a dynamic unit scheduler; an FC2 unit waits until
// every FC1 unit of its expert has published its rows.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "engine.h"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kGroup = 128;  // K elements per scale group; rows per weight tile

// ------------------------------------------------------------ quantiser --
// absmax over 16 lanes (one 128-element group as 16 vectors of 8); every
// lane of the warp takes part, each half-warp reduces its own group.
MOE_DEV float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

MOE_DEV uint2 quant8(const float (&f)[8], float s) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) lo |= (uint32_t)f_to_e4m3(__fdiv_rn(f[i], s)) << (8 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i) hi |= (uint32_t)f_to_e4m3(__fdiv_rn(f[4 + i], s)) << (8 * i);
  return make_uint2(lo, hi);
}

// block_rows = 1: sixteen (row, group) tiles per CTA, sixteen threads a tile.
__global__ void __launch_bounds__(256) quant_groups_kernel(const bf16* __restrict__ x, int64_t tiles,
                                                           int K, uint8_t* __restrict__ q,
                                                           float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
  const int KG = K / kGroup;
  const int64_t tile = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);
  const int sub = threadIdx.x & 15;
  const bool valid = tile < tiles;
  const int64_t r = valid ? tile / KG : 0;
  const int g = valid ? (int)(tile % KG) : 0;
  const size_t off = (size_t)r * K + (size_t)g * kGroup + sub * 8;
  float f[8];
  float amax = 0.f;
  if (valid) {
    unpack8_bf16(*reinterpret_cast<const uint4*>(x + off), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = half_warp_max(amax);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (valid) {
    *reinterpret_cast<uint2*>(q + off) = quant8(f, s);
    if (sub == 0) scale[tile] = s;
  }
}

// block_rows = 128: one 128 x 128 tile per CTA (64 elements a thread).
__global__ void __launch_bounds__(256) quant_tiles_kernel(const bf16* __restrict__ x, int K,
                                                          uint8_t* __restrict__ q,
                                                          float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int g = blockIdx.x, rb = blockIdx.y, KG = K / kGroup;
  const bf16* base = x + (size_t)rb * kGroup * K + (size_t)g * kGroup;
  float amax = 0.f;
  for (int v = threadIdx.x; v < kGroup * 16; v += blockDim.x) {
    float f[8];
    unpack8_bf16(*reinterpret_cast<const uint4*>(base + (size_t)(v >> 4) * K + (v & 15) * 8), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = block_max(amax, red);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint8_t* qb = q + (size_t)rb * kGroup * K + (size_t)g * kGroup;
  for (int v = threadIdx.x; v < kGroup * 16; v += blockDim.x) {
    float f[8];
    unpack8_bf16(*reinterpret_cast<const uint4*>(base + (size_t)(v >> 4) * K + (v & 15) * 8), f);
    *reinterpret_cast<uint2*>(qb + (size_t)(v >> 4) * K + (v & 15) * 8) = quant8(f, s);
  }
  if (threadIdx.x == 0) scale[(size_t)rb * KG + g] = s;
}

// rms_norm of one token per CTA (the arithmetic of the bf16 path's rms_norm),
// then E4M3 codes of x_hat with one scale per 128-element group.
__global__ void __launch_bounds__(512) rmsnorm_q128_kernel(const bf16* __restrict__ x,
                                                           const bf16* __restrict__ w, int H,
                                                           float eps, bf16* __restrict__ y,
                                                           uint8_t* __restrict__ yq,
                                                           float* __restrict__ ys) {
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
  // blockDim.x is a multiple of 16 and nv of 16, so each run of 16 threads
  // holds one group in every pass
  for (int v0 = 0; v0 < nv; v0 += blockDim.x) {
    const int v = v0 + threadIdx.x;
    const bool valid = v < nv;
    float h[8];
    float amax = 0.f;
    if (valid) {
      float f[8], g[8];
      unpack8_bf16(xr[v], f);
      unpack8_bf16(wr[v], g);
      uint4 o;
      o.x = pack2_bf16((f[0] * r) * g[0], (f[1] * r) * g[1]);
      o.y = pack2_bf16((f[2] * r) * g[2], (f[3] * r) * g[3]);
      o.z = pack2_bf16((f[4] * r) * g[4], (f[5] * r) * g[5]);
      o.w = pack2_bf16((f[6] * r) * g[6], (f[7] * r) * g[7]);
      yr[v] = o;
      unpack8_bf16(o, h);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(h[i]));
    }
    amax = half_warp_max(amax);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (valid) {
      *reinterpret_cast<uint2*>(yq + (size_t)t * H + (size_t)v * 8) = quant8(h, s);
      if ((v & 15) == 0) ys[(size_t)t * (H / kGroup) + (v >> 4)] = s;
    }
  }
}

// ------------------------------------------------------- fused FFN kernel --
constexpr int kThreadsB = 224;      // warp 0 TMA, 1 MMA (+ TMEM owner), 2-5 epilogue, 6 publisher
constexpr int kEpiWarpsB = 4;       // one per TMEM lane quarter, both 128-row halves
constexpr int kHalfBytes = 128 * 128;  // one 128-row x 128-byte E4M3 weight tile
constexpr int kMaxStagesB = 8;
constexpr int kBoxRowsB = 16;       // token rows per TMA box
constexpr int kRingB = 4;           // claimed-unit slots
constexpr int kMaxChunkB = 64;      // token rows per unit (MMA N)
// K-group accumulator slots: 2 x chunk TMEM columns each (two 128-row
// halves), as many as fit in 512 columns, at most 16: 16 slots at chunk 16,
// 4 at chunk 64.  The slots are the slack that lets the MMA (and behind it
// the TMA ring) run on while the epilogue finishes a unit.
constexpr int kMaxSlotsB = 16;
constexpr int kTmemColsB = 512;
constexpr int kMaxKG = 64;          // K groups per unit (K <= 8192)
constexpr int kSmemLimitB = 227 * 1024;

struct BJob {
  const float* w_scale;     // [E, N_w / 128, kg] weight tile scales
  const float* a_scale;     // [R, kg] activation group scales of the job's input rows
  const int32_t* row_src;
  const float* topk_w;      // FC2: routing weight of pair row_src[r]
  void* out;                // FC1: E4M3 codes [R, I]; FC2: bf16 [R, H], row r at row_src[r]
  float* out_scale;         // FC1: [R, I / 128] group scales of `out`
  int N_w;                  // weight rows per expert
  int n_out;                // output columns
  int nt;                   // units per (expert, token chunk)
  int kg;                   // K groups
};

// Token-row (B) tensor maps per job with box heights 2, 4, 8 and 16 rows.
struct BMaps {
  CUtensorMap m[2][4];
};

struct BParams {
  const int32_t* offsets;
  int E, I, R_max;
  int chunk;                // token rows per unit (a multiple of 16, <= 64)
  int stages, stage_bytes;  // ring: [W rows 0-127][W rows 128-255][B: chunk rows x 128 B]
  int slots, slot_cols;     // accumulator ring in TMEM
  // after the ring: the unit's activation scales [kg][chunk]
  int* sched;               // [0] unit counter, [1 + e] finished FC1 units of e
  int* status;
  BJob job[2];
};

__global__ void __launch_bounds__(kThreadsB, 1) moe_tc_fp8b_kernel(
    const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
    const __grid_constant__ BMaps bx, const BParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_up[2][kMaxExperts + 1];
  __shared__ __align__(8) uint64_t sfull[kMaxStagesB];
  __shared__ __align__(8) uint64_t sempty[kMaxStagesB];
  __shared__ __align__(8) uint64_t kfull[kMaxSlotsB];
  __shared__ __align__(8) uint64_t kempty[kMaxSlotsB];
  __shared__ __align__(8) uint64_t ufull[kRingB];
  __shared__ __align__(8) uint64_t uempty[kRingB];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t epi_bar;   // the 128 epilogue threads
  __shared__ __align__(8) uint64_t pub_bar;   // FC1 unit written (128 epilogue threads)
  __shared__ __align__(8) uint64_t pub_free;  // the publisher is done with the previous one
  __shared__ int s_uring[kRingB];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_ws[2][kMaxKG];                          // unit's weight scales [half][g]
  __shared__ int s_rs[kMaxChunkB];                           // FC2: row_src of the unit's rows
  __shared__ float s_tw[kMaxChunkB];                         // FC2: their routing weights
  __shared__ float s_red[2][4][16];                          // FC1: per-warp token maxima

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~(uintptr_t)1023);
  float* s_as = reinterpret_cast<float*>(ring + (size_t)p.stages * p.stage_bytes);

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 1);  // the MMA commit
    }
    for (int q = 0; q < p.slots; ++q) {
      mbar_init(&kfull[q], 1);             // the MMA commit
      mbar_init(&kempty[q], kEpiWarpsB * 32);  // every thread of the epilogue warps
    }
    for (int i = 0; i < kRingB; ++i) {
      mbar_init(&ufull[i], 1);
      mbar_init(&uempty[i], 2 + kEpiWarpsB);  // MMA thread, epilogue warps, publisher
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&epi_bar, 32 * kEpiWarpsB);
    mbar_init(&pub_bar, 32 * kEpiWarpsB);
    mbar_init(&pub_free, 1);
    s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w0);
    prefetch_tmap(&tm_w1);
    for (int jb = 0; jb < 2; ++jb)
      for (int bi = 0; bi < 4; ++bi) prefetch_tmap(&bx.m[jb][bi]);
  } else if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemColsB);
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
    const int slot = i % kRingB;
    if (!mbar_wait(&ufull[slot], (uint32_t)((i / kRingB) & 1), &s_abort)) return -2;
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
      const int slot = i % kRingB;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&uempty[slot], (uint32_t)(((i / kRingB) & 1) ^ 1), &s_abort))) {
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
      const BJob& j = p.job[un.job];
      if (un.job == 1) {
        // FC2 of expert e reads its FC1 rows: wait until every FC1 unit of
        // e has been published (FC1 units are all claimed first)
        int fok = 1;
        if (lane == 0) {
          const int cnt = s_off[un.e + 1] - s_off[un.e];
          const int need = ((cnt + p.chunk - 1) / p.chunk) * p.job[0].nt;
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
      // B boxes: the smallest height of 2, 4, 8, 16 rows covering the unit
      const int bi = un.rows > 8 ? 3 : (un.rows > 4 ? 2 : (un.rows > 2 ? 1 : 0));
      const int brows = 2 << bi;
      const int nb = bi == 3 ? (un.rows + kBoxRowsB - 1) / kBoxRowsB : 1;
      const uint32_t tx = (uint32_t)(2 * kHalfBytes + nb * brows * 128);
      const CUtensorMap* tw = un.job ? &tm_w1 : &tm_w0;
      const CUtensorMap* tx_map = &bx.m[un.job][bi];
      const int wrow = un.e * j.N_w;
      // FC1: 128 gate rows and the matching 128 up rows; FC2: 256 rows
      const int r0 = un.job == 0 ? wrow + un.nt * 128 : wrow + un.nt * 256;
      const int r1 = un.job == 0 ? wrow + p.I + un.nt * 128 : r0 + 128;
      for (int g = 0; g < j.kg; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait_spin(&sempty[s], ph ^ 1, &s_abort))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&sfull[s], tx);
          uint8_t* st = ring + (size_t)s * p.stage_bytes;
          tma_load_2d(st, tw, &sfull[s], g * kGroup, r0, pol_w);
          tma_load_2d(st + kHalfBytes, tw, &sfull[s], g * kGroup, r1, pol_w);
          for (int bb = 0; bb < nb; ++bb)
            tma_load_2d(st + 2 * kHalfBytes + bb * kBoxRowsB * 128, tx_map, &sfull[s], g * kGroup,
                        un.row0 + bb * kBoxRowsB, pol_x);
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
  } else if (warp == 1) {
    // ====================================================== MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues, so the
    // descriptors and TMEM addresses stay warp-uniform (each group is eight
    // small MMAs at decode's N, where a loop run by one divergent lane paid
    // about 100 cycles per tcgen05 instruction).
    int s = 0, q = 0;
    uint32_t ph = 0, qph = 0;
    bool ok = true, issued = false;
    for (int i = 0; ok; ++i) {
      const int u = __shfl_sync(0xffffffffu, next_unit(i), 0);  // every lane has read it
      if (u == -2) { ok = false; break; }
      if (lane == 0) mbar_arrive(&uempty[i % kRingB]);
      if (u < 0) break;
      const Unit un = decode_unit(u);
      const int kg = p.job[un.job].kg;
      const uint32_t idesc = make_idesc(((un.rows + 15) / 16) * 16, 0u);  // E4M3 A and B
      for (int g = 0; g < kg; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait_spin(&sfull[s], ph, &s_abort) &&
                                         mbar_wait_spin(&kempty[q], qph ^ 1, &s_abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(ring + (size_t)s * p.stage_bytes);
        const uint32_t b0 = a0 + 2 * kHalfBytes;
        if (elect_one()) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t d = tmem + q * p.slot_cols + h * p.chunk;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // four 32-byte K steps: each group starts a fresh sum
              mma_e4m3(d, sw128_desc(a0 + h * kHalfBytes + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                       kk ? 1u : 0u);
          }
          mma_commit(&sempty[s]);
          mma_commit(&kfull[q]);
        }
        __syncwarp();
        issued = true;
        if (++s == p.stages) { s = 0; ph ^= 1; }
        if (++q == p.slots) { q = 0; qph ^= 1; }
      }
    }
    // tail: the epilogues have handed back every slot
    for (int i = 0; ok && i < p.slots; ++i) {
      ok = __all_sync(0xffffffffu, mbar_wait(&kempty[q], qph ^ 1, &s_abort));
      if (++q == p.slots) { q = 0; qph ^= 1; }
    }
    if (!ok && lane == 0) flag_status(p.status, MOE_ERR_TIMEOUT);
    if (issued) {  // all issued MMAs complete before TMEM is released
      if (elect_one()) mma_commit(&drain_bar);
      __syncwarp();
      if (lane == 0) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&drain_bar, 0) && clock64() - t0 < kSpinLimitCycles) {
        }
      }
      __syncwarp();
    }
  } else if (warp < 2 + kEpiWarpsB) {
    // ======================================================== epilogue
    // Warp w (2..5) owns rows l = 32 (w % 4) + lane (its TMEM lane quarter)
    // of both 128-row halves of the unit: FC1 gate and up row of one
    // intermediate column, or two W2 rows 128 apart.
    const int qtr = warp & 3;
    const int l = qtr * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..127
    const uint32_t tlane = (uint32_t)(qtr * 32) << 16;
    int q = 0;
    uint32_t qph = 0, eph = 0;
    uint32_t nf = 0;  // FC1 units handed to the publisher
    bool ok = true;
    auto epi_sync = [&]() -> bool {
      mbar_arrive(&epi_bar);
      const bool r = mbar_wait(&epi_bar, eph, &s_abort);
      eph ^= 1;
      return r;
    };
    for (int i = 0; ok; ++i) {
      const int u = next_unit(i);
      __syncwarp();
      if (lane == 0 && u != -2) mbar_arrive(&uempty[i % kRingB]);
      if (u == -2) { ok = false; break; }
      if (u < 0) break;
      const Unit un = decode_unit(u);
      const BJob& j = p.job[un.job];
      const int ncols = ((un.rows + 15) / 16) * 16;
      // stage the unit's scales (and FC2's row_src / routing weights) once
      // every epilogue thread is done with the previous unit's
      if (!epi_sync()) { ok = false; break; }
      if (un.job == 1) {
        // FC2's activation scales are FC1 output: every thread acquires the
        // expert's FC1 count itself before reading them (the unit is handed
        // out before the producer's own wait on that count)
        const int cnt = s_off[un.e + 1] - s_off[un.e];
        const int need = ((cnt + p.chunk - 1) / p.chunk) * p.job[0].nt;
        const int* flag = p.sched + 1 + un.e;
        const long long t0 = clock64();
        while (ld_acquire(flag) < need) {
          if (s_abort || clock64() - t0 > kSpinLimitCycles) {
            s_abort = 1;
            ok = false;
            break;
          }
        }
        if (!ok) break;
      }
      for (int idx = et; idx < j.kg * ncols; idx += 32 * kEpiWarpsB) {
        const int g = idx / ncols, c = idx - g * ncols;
        s_as[g * p.chunk + c] = c < un.rows ? j.a_scale[(size_t)(un.row0 + c) * j.kg + g] : 0.f;
      }
      for (int idx = et; idx < 2 * j.kg; idx += 32 * kEpiWarpsB) {
        const int hh = idx / j.kg, g = idx - hh * j.kg;
        const int rb = un.job == 0 ? (hh ? p.I / kGroup + un.nt : un.nt) : 2 * un.nt + hh;
        s_ws[hh][g] = j.w_scale[((size_t)un.e * (j.N_w / kGroup) + rb) * j.kg + g];
      }
      if (un.job == 1 && et < un.rows) {
        const int orow = j.row_src[un.row0 + et];
        s_rs[et] = orow;
        s_tw[et] = j.topk_w[orow];
      }
      if (!epi_sync()) { ok = false; break; }

      float acc0[kMaxChunkB], acc1[kMaxChunkB];  // rows l and 128 + l of the unit
#pragma unroll
      for (int c = 0; c < kMaxChunkB; ++c) {
        acc0[c] = 0.f;
        acc1[c] = 0.f;
      }
      for (int g = 0; g < j.kg; ++g) {
        // a suspending wait: the epilogue has slack (the slot ring), while a
        // polling loop here would take issue slots from the TMA and MMA
        // threads that share the SM's sub-partitions.  Every lane waits and
        // every lane arrives below: the group loop has no divergent branch.
        if (!__all_sync(0xffffffffu, mbar_wait(&kfull[q], qph, &s_abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = tmem + tlane + q * p.slot_cols;
        const float sw0 = s_ws[0][g], sw1 = s_ws[1][g];
        const float4* sa = reinterpret_cast<const float4*>(s_as + g * p.chunk);
        // passes of up to 16 columns of both halves
#pragma unroll
        for (int c16 = 0; c16 < kMaxChunkB; c16 += 16) {
          if (c16 < ncols) {
            float v0[16], v1[16];
            tmem_ld16(ta + c16, v0);
            tmem_ld16(ta + p.chunk + c16, v1);
            tmem_ld_wait();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const float4 a = sa[c16 / 4 + c4];
              const float as[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int c = c16 + 4 * c4 + t;
                acc0[c] = fmaf(v0[4 * c4 + t], sw0 * as[t], acc0[c]);
                acc1[c] = fmaf(v1[4 * c4 + t], sw1 * as[t], acc1[c]);
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&kempty[q]);
        if (++q == p.slots) { q = 0; qph ^= 1; }
      }
      if (!ok) break;

      if (un.job == 1) {
        // FC2: bf16(routing weight x y) at row row_src[r] of the output
        const int n = un.nt * 256 + l;
        bf16* out = reinterpret_cast<bf16*>(j.out);
#pragma unroll
        for (int c = 0; c < kMaxChunkB; ++c)
          if (c < un.rows) {
            bf16* o = out + (size_t)s_rs[c] * j.n_out + n;
            o[0] = __float2bfloat16_rn(acc0[c] * s_tw[c]);
            o[128] = __float2bfloat16_rn(acc1[c] * s_tw[c]);
          }
      } else {
        // FC1: a = bf16(silu(g) u) of intermediate column n for each token,
        // 16 tokens a pass; each token's absmax over the unit's 128 columns
        // (one K group of FC2) from a warp reduction and four per-warp
        // maxima (double-buffered, so one barrier a pass); then the E4M3
        // codes and the group scale.  Each code is decided from a / s with
        // the correctly rounded divide: a and s carry few significant bits,
        // so a / s often lands exactly on a midpoint between two E4M3
        // values, where a * (1 / s) can round to the other side.
        const int n = un.nt * 128 + l;
        uint8_t* outq = reinterpret_cast<uint8_t*>(j.out);
        const int kg_out = j.n_out / kGroup;
#pragma unroll
        for (int c0 = 0; c0 < kMaxChunkB; c0 += 16) {
          if (c0 < ncols) {
            float (*red)[16] = s_red[(c0 / 16) & 1];
            float a[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const float gt = acc0[c0 + t];
              a[t] = bf16_round_f(__fdividef(gt, 1.0f + __expf(-gt)) * acc1[c0 + t]);
              // |a| >= 0 orders like its bit pattern
              const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(a[t])));
              if (lane == 0) red[qtr][t] = __uint_as_float(m);
            }
            if (!epi_sync()) { ok = false; break; }
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const int c = c0 + t;
              const float amax = fmaxf(fmaxf(red[0][t], red[1][t]), fmaxf(red[2][t], red[3][t]));
              const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
              if (c < un.rows) {
                const size_t r = (size_t)(un.row0 + c);
                outq[r * j.n_out + n] = f_to_e4m3(__fdiv_rn(a[t], s));
                if (l == 0) j.out_scale[r * kg_out + un.nt] = s;
              }
            }
          }
        }
        if (!ok) break;
        // make this thread's rows visible to the async proxy (FC2's TMA
        // loads) and hand the unit to the publisher, once it has taken the
        // previous one (so that pub_bar never runs two phases ahead)
        fence_proxy_async_global();
        if (nf > 0 && !mbar_wait(&pub_free, (nf - 1) & 1, &s_abort)) { ok = false; break; }
        mbar_arrive(&pub_bar);
        ++nf;
      }
    }
    if (!ok) flag_status(p.status, MOE_ERR_TIMEOUT);
  } else if (warp == 6) {
    // ====================================================== publisher
    // Per FC1 unit: once its 128 epilogue threads have arrived, a gpu-scope
    // fence (cumulative over the writes ordered before the arrivals) and the
    // count FC2's readers acquire.  Off the epilogue's path, which goes on
    // with the next unit.
    uint32_t pph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int u = next_unit(i);
      __syncwarp();
      if (lane == 0 && u != -2) mbar_arrive(&uempty[i % kRingB]);
      if (u == -2) { ok = false; break; }
      if (u < 0) break;
      const Unit un = decode_unit(u);
      if (un.job != 0) continue;
      if (lane == 0) {
        ok = mbar_wait(&pub_bar, pph, &s_abort);
        if (ok) {
          __threadfence();
          atomicAdd(p.sched + 1 + un.e, 1);
          mbar_arrive(&pub_free);
        }
      }
      pph ^= 1;
      ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    }
    if (!ok && lane == 0) flag_status(p.status, MOE_ERR_TIMEOUT);
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemColsB);
}


// ------------------------------------------- prefill tile kernel (FC1 / FC2) --
// For batches with many rows per expert the weight-streaming layout above
// re-reads each expert's weights once per 64-token chunk.  This kernel tiles
// the tokens instead: a unit is 128 token rows (MMA M, TMEM lanes) x 128
// weight rows (MMA N) of one expert over all of K, one 128-wide K group per
// 32 KB stage.  FC1 (MODE 1) takes 64 gate rows and the matching 64 up rows
// and writes bf16 a = silu(g) u; FC2 (MODE 3) takes 128 rows of W2 and writes
// bf16 (routing weight x y) at row row_src[r].  The forward quantises a per
// 128-column group between the two launches.
//
// Each K group's product goes to its own 128-column TMEM slot (ring of four).
// Eight epilogue warps, two per TMEM lane quarter, each own 64 accumulator
// columns of their 32 token rows in registers: a thread's group scale is one
// activation scale (its token row) times one weight-tile scale per 32
// columns, so the fold is a scalar multiply-add per element.  The warps never
// synchronise with one another.
// The fold runs on register pairs (__ffma2_rn: each half an IEEE fused
// multiply-add, round to nearest, the same bits as two fmaf).

constexpr int kThreadsT = 352;       // warp 0 TMA, 1 MMA (+ TMEM owner), 2-9 epilogue, 10 MMA
constexpr int kMma2WarpT = 10;
constexpr int kTileBytesT = 128 * 128;
constexpr int kStageBytesT = 2 * kTileBytesT;  // token tile + weight tile of one K group
constexpr int kSlotsT = 4;
constexpr int kMaxStagesT = 6;
static_assert(kSlotsT % 2 == 0, "each TMEM slot belongs to one of the two MMA issuers");

struct TParams {
  const int32_t* offsets;
  int E, I, R_max;
  int N_w;                  // weight rows per expert
  int nt;                   // N tiles per (expert, token tile)
  int kg;                   // K groups
  int stages;
  const float* a_scale;     // [R, kg] activation group scales
  const float* w_scale;     // [E, N_w / 128, kg] weight tile scales
  const int32_t* row_src;   // FC2: destination row of row r
  const float* topk_w;      // FC2: routing weight of pair row_src[r]
  void* out;                // bf16 rows
  int ldo;
  int* status;
};

// What an epilogue thread needs of one unit: its token row and the scale
// rows of its two 32-column runs.
struct TileCtx {
  int r, nt;
  bool rvalid;
  const float* sa_row;      // activation scales of row r, one per K group
  const float* sw_lo;       // weight-tile scales of the two column runs
  const float* sw_hi;
};

template <int MODE>
MOE_DEV TileCtx tile_ctx(int u, const int* s_off, const int* s_up, const TParams& p, int lrow) {
  const Unit un = unit_of(u, s_off, s_up, p.E, p.nt, 128);
  const int nblk = p.N_w / kGroup;
  // FC1: gate rows nt*64.. and the matching up rows I further; FC2: one tile
  const int rb_lo = MODE == 1 ? (un.nt * 64) / kGroup : un.nt;
  const int rb_hi = MODE == 1 ? (p.I + un.nt * 64) / kGroup : un.nt;
  TileCtx c;
  c.nt = un.nt;
  c.rvalid = lrow < un.rows;
  c.r = un.row0 + lrow;
  c.sa_row = p.a_scale + (size_t)(c.rvalid ? c.r : 0) * p.kg;
  c.sw_lo = p.w_scale + ((size_t)un.e * nblk + rb_lo) * p.kg;
  c.sw_hi = p.w_scale + ((size_t)un.e * nblk + rb_hi) * p.kg;
  return c;
}

template <int MODE>
__global__ void __launch_bounds__(kThreadsT, 1) moe_tc_fp8b_tile_kernel(
    const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
    const TParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_up[kMaxExperts + 1];
  __shared__ __align__(8) uint64_t sfull[kMaxStagesT];
  __shared__ __align__(8) uint64_t sempty[kMaxStagesT];
  __shared__ __align__(8) uint64_t kfull[kSlotsT];
  __shared__ __align__(8) uint64_t kempty[kSlotsT];
  __shared__ __align__(8) uint64_t drain_bar[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~(uintptr_t)1023);
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 1);
    }
    for (int q = 0; q < kSlotsT; ++q) {
      mbar_init(&kfull[q], 1);
      mbar_init(&kempty[q], 8 * 32);  // every thread of the eight epilogue warps
    }
    mbar_init(&drain_bar[0], 1);
    mbar_init(&drain_bar[1], 1);
    s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_w);
  } else if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemColsB);
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
  if (warp == 0) {  // unit prefix: ceil(rows / 128) token tiles x nt per expert
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      const int cnt = (e < p.E) ? s_off[e + 1] - s_off[e] : 0;
      const int v = ((cnt + 127) / 128) * p.nt;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < p.E) s_up[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_up[p.E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int U = s_up[p.E];

  if (warp == 0) {
    // ===================================================== TMA producer
    // The whole warp runs the loop and waits; one elected lane arms the
    // stage and issues its loads.
    const uint64_t pol_w = l2_policy_evict_last();  // re-read by the expert's other token tiles
    const uint64_t pol_a = l2_policy_evict_first();
    int s = 0;
    uint32_t ph = 0, armed = 0, armed_ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < U; u += gridDim.x) {
      const Unit un = unit_of(u, s_off, s_up, p.E, p.nt, 128);
      const int wrow = un.e * p.N_w;
      // FC1: gate rows nt*64.. and the matching up rows; FC2: 128 rows
      const int r0 = MODE == 1 ? wrow + un.nt * 64 : wrow + un.nt * 128;
      const int r1 = MODE == 1 ? wrow + p.I + un.nt * 64 : r0 + 64;
      for (int g = 0; g < p.kg; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sempty[s], ph ^ 1, &s_abort))) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&sfull[s], (uint32_t)kStageBytesT);
          uint8_t* st = ring + (size_t)s * kStageBytesT;
          tma_load_2d(st, &tm_a, &sfull[s], g * kGroup, un.row0, pol_a);
          tma_load_2d(st + kTileBytesT, &tm_w, &sfull[s], g * kGroup, r0, pol_w);
          tma_load_2d(st + kTileBytesT + kTileBytesT / 2, &tm_w, &sfull[s], g * kGroup, r1, pol_w);
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
  } else if (warp == 1 || warp == kMma2WarpT) {
    // ===================================================== MMA issuers
    // Two warps issue the MMAs: warp 1 the even K groups (counted over all
    // units), warp 10 the odd ones, so one thread's per-instruction issue
    // cost no longer paces the tensor pipe.  Each group has its own stage and
    // TMEM slot, and both rings have even lengths, so every stage and every
    // slot belongs to one issuer and is used in order.  The whole warp runs
    // the loop and waits, and one elected lane issues, so the descriptors and
    // TMEM addresses stay warp-uniform (a loop run by one divergent lane paid
    // about 100 cycles per tcgen05 instruction).
    const int par = warp == 1 ? 0 : 1;
    int s = 0, q = 0, gi = 0;
    uint32_t ph = 0, qph = 0;
    bool ok = true, issued = false;
    const uint32_t idesc = make_idesc(128, 0u);  // M = N = 128, E4M3 A and B
    for (int u = blockIdx.x; ok && u < U; u += gridDim.x) {
      for (int g = 0; g < p.kg; ++g, ++gi) {
        if ((gi & 1) == par) {
          const bool w = mbar_wait(&sfull[s], ph, &s_abort) && mbar_wait(&kempty[q], qph ^ 1, &s_abort);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + (size_t)s * kStageBytesT);
          const uint32_t d = tmem + q * 128;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // each group starts a fresh sum
              mma_e4m3(d, sw128_desc(a0 + kk * 32), sw128_desc(a0 + kTileBytesT + kk * 32), idesc,
                       kk ? 1u : 0u);
            mma_commit(&sempty[s]);
            mma_commit(&kfull[q]);
          }
          __syncwarp();
          issued = true;
        }
        if (++s == p.stages) { s = 0; ph ^= 1; }
        if (++q == kSlotsT) { q = 0; qph ^= 1; }
      }
    }
    // tail: this issuer's slots handed back (the next four ring positions
    // are the last use of each slot)
    for (int i = 0; ok && i < kSlotsT; ++i, ++gi) {
      if ((gi & 1) == par) ok = __all_sync(0xffffffffu, mbar_wait(&kempty[q], qph ^ 1, &s_abort));
      if (++q == kSlotsT) { q = 0; qph ^= 1; }
    }
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
  } else {
    // ======================================================== epilogue
    // Warp w (2..9): token rows 32 (w % 4) .. +31 of the tile (its TMEM lane
    // quarter) and half h = (w - 2) / 4 of the columns: FC1 gate columns
    // 32h .. 32h + 31 with the matching up columns 64 + 32h ..; FC2 columns
    // 64h .. 64h + 63.  acc[0..31] and acc[32..63] are those two 32-column runs.
    // The MMA threads run at most four K groups ahead, so the global loads a
    // unit needs are issued early: the next group's scales during this one
    // (at a unit's last group, the next unit's first), FC2's destination row
    // one unit ahead and its routing weight halfway through the unit.
    const int h = (warp - 2) >> 2;
    const int qtr = warp & 3;
    const int lrow = qtr * 32 + lane;
    const uint32_t tlane = (uint32_t)(qtr * 32) << 16;
    const int c_lo = MODE == 1 ? 32 * h : 64 * h;
    const int c_hi = MODE == 1 ? 64 + 32 * h : 64 * h + 32;
    int q = 0;
    uint32_t qph = 0;
    bool ok = true;
    int u = blockIdx.x;
    TileCtx cur{}, nxt{};
    float sa = 0.f, wl = 0.f, wh = 0.f;
    int orow = 0, orow_n = 0;
    if (u < U) {
      cur = tile_ctx<MODE>(u, s_off, s_up, p, lrow);
      sa = cur.rvalid ? cur.sa_row[0] : 0.f;
      wl = cur.sw_lo[0];
      wh = cur.sw_hi[0];
      if (MODE == 3 && cur.rvalid) orow = p.row_src[cur.r];
    }
    for (; ok && u < U; u += gridDim.x) {
      const bool has_next = u + (int)gridDim.x < U;
      if (has_next) {
        nxt = tile_ctx<MODE>(u + gridDim.x, s_off, s_up, p, lrow);
        if (MODE == 3 && nxt.rvalid) orow_n = p.row_src[nxt.r];
      }
      float tw = 0.f;
      float2 acc[32];  // columns 2c, 2c + 1 of the lo run (c < 16), then of the hi run
#pragma unroll
      for (int c = 0; c < 32; ++c) acc[c] = make_float2(0.f, 0.f);
      for (int g = 0; g < p.kg; ++g) {
        // the scales of the group after this one load while this group's
        // product is awaited
        float sa_n = 0.f, wl_n = 0.f, wh_n = 0.f;
        if (g + 1 < p.kg) {
          sa_n = cur.rvalid ? cur.sa_row[g + 1] : 0.f;
          wl_n = cur.sw_lo[g + 1];
          wh_n = cur.sw_hi[g + 1];
        } else if (has_next) {
          sa_n = nxt.rvalid ? nxt.sa_row[0] : 0.f;
          wl_n = nxt.sw_lo[0];
          wh_n = nxt.sw_hi[0];
        }
        if (MODE == 3 && g == (p.kg >> 1) && cur.rvalid) tw = p.topk_w[orow];
        // every lane waits and every lane hands the slot back: no divergent
        // branch in the loop
        if (!__all_sync(0xffffffffu, mbar_wait(&kfull[q], qph, &s_abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float v[64];
        const uint32_t ta = tmem + tlane + q * 128;
        if (MODE == 3) {  // FC2: the two runs are adjacent
          tmem_ld64(ta + c_lo, v);
        } else {
          tmem_ld32(ta + c_lo, v);
          tmem_ld32(ta + c_hi, v + 32);
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&kempty[q]);
        if (++q == kSlotsT) { q = 0; qph ^= 1; }
        const float2 fl = make_float2(sa * wl, sa * wl), fh = make_float2(sa * wh, sa * wh);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          acc[c] = __ffma2_rn(make_float2(v[2 * c], v[2 * c + 1]), fl, acc[c]);
          acc[16 + c] = __ffma2_rn(make_float2(v[32 + 2 * c], v[33 + 2 * c]), fh, acc[16 + c]);
        }
        sa = sa_n;
        wl = wl_n;
        wh = wh_n;
      }
      if (!ok) break;
      if (cur.rvalid) {
        bf16* out = reinterpret_cast<bf16*>(p.out);
        if (MODE == 1) {
          // a = bf16(silu(g) u): 32 columns from nt*64 + 32h, 64 bytes; silu
          // with the fast exponential and divide, as in the decode epilogue
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float g0 = acc[c].x, g1 = acc[c].y;
            pk[c] = pack2_bf16(__fdividef(g0, 1.0f + __expf(-g0)) * acc[16 + c].x,
                               __fdividef(g1, 1.0f + __expf(-g1)) * acc[16 + c].y);
          }
          uint4* dst = reinterpret_cast<uint4*>(out + (size_t)cur.r * p.ldo + cur.nt * 64 + 32 * h);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        } else {
          // routing weight x y, bf16, at row row_src[r]: 64 columns from nt*128 + 64h
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = pack2_bf16(acc[c].x * tw, acc[c].y * tw);
          uint4* dst = reinterpret_cast<uint4*>(out + (size_t)orow * p.ldo + cur.nt * 128 + 64 * h);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      cur = nxt;
      orow = orow_n;
    }
    if (!ok) flag_status(p.status, MOE_ERR_TIMEOUT);
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemColsB);
}

template <int MODE>
cudaError_t launch_tile(const void* a, const float* a_scale, const uint8_t* w, const float* w_scale,
                        int K, int N_w, int nt, const int32_t* offsets, const int32_t* row_src,
                        const float* topk_w, void* out, int ldo, int E, int I, int R_max, int sms,
                        int* status, cudaStream_t st) {
  TParams p{};
  p.offsets = offsets;
  p.E = E;
  p.I = I;
  p.R_max = R_max;
  p.N_w = N_w;
  p.nt = nt;
  p.kg = K / kGroup;
  p.a_scale = a_scale;
  p.w_scale = w_scale;
  p.row_src = row_src;
  p.topk_w = topk_w;
  p.out = out;
  p.ldo = ldo;
  p.status = status;
  auto k = moe_tc_fp8b_tile_kernel<MODE>;
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, k);
  if (e != cudaSuccess) return e;
  int stages = (int)((kSmemLimitB - (int)fa.sharedSizeBytes - 1024) / kStageBytesT);
  if (stages > kMaxStagesT) stages = kMaxStagesT;
  stages &= ~1;  // even: each stage belongs to one of the two MMA issuers
  if (stages < 2) return cudaErrorNotSupported;
  p.stages = stages;
  const size_t smem = 1024 + (size_t)stages * kStageBytesT;
  CUtensorMap ma, mw;
  if (!tc::encode_map(&ma, a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, R_max, K, kGroup, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::encode_map(&mw, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (int64_t)E * N_w, K, kGroup, 64,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorNotSupported;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(k, dim3(sms), dim3(kThreadsT), smem, st, ma, mw, p);
}

}  // namespace

// ------------------------------------------------------------------ host --
cudaError_t launch_quantize_fp8_blocks(const void* x, int N, int K, int block_rows, uint8_t* q,
                                       float* scale, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  if (K % kGroup != 0 || (block_rows != 1 && block_rows != kGroup) || N % block_rows != 0)
    return cudaErrorInvalidValue;
  if (block_rows == 1) {
    const int64_t tiles = (int64_t)N * (K / kGroup);
    return launch_kernel(quant_groups_kernel, dim3((unsigned)((tiles + 15) / 16)), dim3(256), 0, st,
                         (const bf16*)x, tiles, K, q, scale);
  }
  return launch_kernel(quant_tiles_kernel, dim3(K / kGroup, N / kGroup), dim3(256), 0, st,
                       (const bf16*)x, K, q, scale);
}

cudaError_t launch_rmsnorm_q128(const void* x, const void* w, int T, int H, float eps, void* y,
                                uint8_t* yq, float* yscale, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (H % kGroup != 0) return cudaErrorInvalidValue;
  // the rms_norm launch shape (a multiple of 32, so of 16 too)
  const int threads = rmsnorm_threads(T, H / 8);
  return launch_kernel(rmsnorm_q128_kernel, dim3(T), dim3(threads), 0, st,
                       (const bf16*)x, (const bf16*)w, H, eps, (bf16*)y, yq, yscale);
}

bool fp8b_decode_covers(int H, int I, int E) {
  return H % 256 == 0 && I % kGroup == 0 && H / kGroup <= kMaxKG && I / kGroup <= kMaxKG &&
         E <= kMaxExperts;
}

cudaError_t launch_decode_ffn_fp8b(const uint8_t* xp, const float* xp_scale, const uint8_t* w13,
                                   const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                   uint8_t* actq, float* act_scale, void* y, const int32_t* offsets,
                                   const int32_t* row_src, const float* topk_w, int* sched, int E,
                                   int H, int I, int R_max, int T, int sms, int* status,
                                   cudaStream_t st) {
  if (R_max == 0) return cudaSuccess;
  if (!fp8b_decode_covers(H, I, E) || !sched) return cudaErrorNotSupported;
  BParams p{};
  p.offsets = offsets;
  p.E = E;
  p.I = I;
  p.R_max = R_max;
  int chunk = T < kMaxChunkB ? T : kMaxChunkB;
  chunk = ((chunk < 1 ? 1 : chunk) + kBoxRowsB - 1) / kBoxRowsB * kBoxRowsB;
  p.chunk = chunk;
  p.sched = sched;
  p.status = status;
  p.stage_bytes = 2 * kHalfBytes + chunk * 128;
  p.slot_cols = 2 * chunk;
  p.slots = kTmemColsB / p.slot_cols < kMaxSlotsB ? kTmemColsB / p.slot_cols : kMaxSlotsB;
  const int kg_max = (H > I ? H : I) / kGroup;
  const int scratch = kg_max * chunk * 4;
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, moe_tc_fp8b_kernel);
  if (e != cudaSuccess) return e;
  int stages = (int)((kSmemLimitB - (int)fa.sharedSizeBytes - 1024 - scratch) / p.stage_bytes);
  if (stages > kMaxStagesB) stages = kMaxStagesB;
  if (stages < 2) return cudaErrorNotSupported;
  p.stages = stages;
  const size_t smem = 1024 + (size_t)stages * p.stage_bytes + scratch;
  // job 0: FC1 + silu_and_mul -> E4M3 act [R, I] + group scales [R, I/128];
  // job 1: FC2 + routing weight -> bf16 rows at row_src
  p.job[0] = BJob{w13_scale, xp_scale, row_src, nullptr, actq, act_scale, 2 * I, I, I / kGroup,
                  H / kGroup};
  p.job[1] = BJob{w2_scale, act_scale, row_src, topk_w, y, nullptr, H, H, H / 256, I / kGroup};
  CUtensorMap m[2];
  BMaps bx;
  for (int bi = 0; bi < 4; ++bi)
    if (!tc::encode_map(&bx.m[0][bi], xp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, R_max, H, kGroup, 2 << bi,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tc::encode_map(&bx.m[1][bi], actq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, R_max, I, kGroup,
                        2 << bi, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorNotSupported;
  if (!tc::encode_map(&m[0], w13, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (int64_t)E * 2 * I, H, kGroup,
                      kGroup, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::encode_map(&m[1], w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (int64_t)E * H, I, kGroup, kGroup,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorNotSupported;
  e = cudaFuncSetAttribute(moe_tc_fp8b_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_tc_fp8b_kernel, dim3(sms), dim3(kThreadsB), smem, st, m[0], m[1], bx, p);
}

cudaError_t launch_prefill_ffn_fp8b(const uint8_t* xp, const float* xp_scale, const uint8_t* w13,
                                    const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, void* act, uint8_t* actq,
                                    float* act_scale, void* y, const int32_t* offsets,
                                    const int32_t* row_src, const float* topk_w, int E, int H,
                                    int I, int R_max, int sms, int* status, cudaStream_t st) {
  if (R_max == 0) return cudaSuccess;
  if (!fp8b_decode_covers(H, I, E)) return cudaErrorNotSupported;
  // FC1 + silu_and_mul -> bf16 act [R, I]
  cudaError_t e = launch_tile<1>(xp, xp_scale, w13, w13_scale, H, 2 * I, I / 64, offsets, nullptr,
                                 nullptr, act, I, E, I, R_max, sms, status, st);
  if (e != cudaSuccess) return e;
  // act -> E4M3 codes with one scale per row and 128 columns
  e = launch_quantize_fp8_blocks(act, R_max, I, 1, actq, act_scale, st);
  if (e != cudaSuccess) return e;
  // FC2 + routing weight -> bf16 rows at row_src
  return launch_tile<3>(actq, act_scale, w2, w2_scale, I, H, H / 128, offsets, row_src, topk_w, y,
                        H, E, I, R_max, sms, status, st);
}

}  // namespace moe
