// Tensor-core grouped GEMM engines for the MoE FFN (tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised kernel template covers FC1 (raw, or with
// the silu_and_mul epilogue) and FC2 (with the routing-weight epilogue,
// fp32 or bf16 output), on
// bf16 (kind::f16) or E4M3 (kind::f8f6f4) operands, in two orientations:
//
//  decode  (SWAP = true)   the MMA's 128-row operand is a slice of one
//          expert's weight matrix and the expert's token rows (16..128,
//          padded to a multiple of 16) are the narrow N operand.  Every CTA
//          owns contiguous N-slices of the expert weights and streams them
//          from HBM through a deep shared-memory ring, which is what bounds
//          small-batch MoE (the weight-streaming, split-N view of the
//          "Locality domain" section of the Vera Rubin article).
//  prefill (SWAP = false)  classic tiles: 128 token rows x 256 weight rows.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns the TMEM
// allocation and issues tcgen05.mma, warps 2..5 are the epilogue (each reads
// its 32-lane quarter of TMEM).  Work units are (expert, 128-row chunk of its
// tokens, N tile), enumerated on the device from the expert offsets; CTA c
// takes units c, c + grid, ...  Shared memory holds `stages` ring slots of
// one 128-byte-wide K slice each (64 bf16 or 128 e4m3), written by TMA with
// the 128-byte swizzle and read by the MMA through matching descriptors.
// TMEM holds two 256-column fp32 accumulators so the epilogue of one unit
// overlaps the main loop of the next.  For FC1 + silu the gate accumulator
// sits in columns 0..127 of a buffer and the up accumulator in 128..255.
//
// Every wait is bounded (see tc_ptx.cuh); a wait that runs out raises the
// CTA's abort flag, records MOE_ERR_TIMEOUT and the roles wind down, with
// outstanding TMA copies and MMAs drained before TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "engine.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kThreads = 192;
constexpr int kRowBytes = 128;       // one swizzle row: K slice of a stage
constexpr int kTileRows = 128;       // MMA M
constexpr int kTileBytes = kTileRows * kRowBytes;  // 16 KB
constexpr int kAccCols = 256;        // TMEM columns per accumulator buffer
constexpr int kMaxStages = 8;
constexpr int kDecodeMaxN = 128;     // token rows per decode unit
constexpr int kDecodeBoxRows = 16;   // token rows per TMA box (decode)
constexpr int kSmemLimit = 227 * 1024;

struct Params {
  const int32_t* offsets;
  const int32_t* row_src;
  const float* topk_w;
  const float* a_scale;  // per token row (E4M3)
  const float* w_scale;  // per weight row (E4M3)
  void* out;
  int ldo;     // output row stride (elements)
  int E, I, N_w, n_out;
  int R_max;   // rows of the activation operand / output
  int nt;      // N tiles per (expert, token chunk)
  int chunk;   // token rows per unit (decode: the B tile height; prefill: 128)
  int kst;     // K stages (128-byte K slices)
  int stages;
  int stage_bytes;
  int a_bytes;  // bytes of the A region of a stage (decode FC1: gate+up tiles)
  int* status;
};

struct Unit {
  int e, nt, row0, rows;
};

// Unit enumeration shared by all roles: expert e has ceil(cnt/chunk) token
// chunks, each with nt N tiles; s_up[e] is the exclusive prefix of units.
MOE_DEV Unit unit_of(int u, const int* s_off, const int* s_up, int E, int nt, int chunk) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_up[mid] <= u) lo = mid; else hi = mid - 1;
  }
  const int local = u - s_up[lo];
  const int mt = local / nt;
  Unit un;
  un.e = lo;
  un.nt = local - mt * nt;
  un.row0 = s_off[lo] + mt * chunk;
  un.rows = min(chunk, s_off[lo + 1] - un.row0);
  return un;
}

template <bool SWAP, int MODE, bool FP8>
__global__ void __launch_bounds__(kThreads, 1) moe_tc_gemm_kernel(
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
    const Params p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_up[kMaxExperts + 1];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t xch_bar;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_xch[SWAP && MODE == 1 ? 64 * 17 : 1];  // decode FC1: up values

  constexpr bool IS_FC2 = (MODE == 2 || MODE == 3);  // routing-weight epilogue
  constexpr bool OUT_F32 = (MODE == 2);              // fp32 output (else bf16)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~(uintptr_t)1023);

  // ---- set-up: barriers and TMEM first (no global memory), then wait for
  // the previous kernel and build the unit table from the expert offsets
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 128);
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&xch_bar, 128);
    s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_x);
  } else if (warp == 1) {
    tmem_alloc(&s_tmem, 2 * kAccCols);
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
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      const int cnt = (e < p.E) ? s_off[e + 1] - s_off[e] : 0;
      const int v = ((cnt + p.chunk - 1) / p.chunk) * p.nt;
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
    if (lane == 0) {
      const uint64_t pol_w = SWAP ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_x = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        const Unit un = unit_of(u, s_off, s_up, p.E, p.nt, p.chunk);
        const int nb = SWAP ? (un.rows + kDecodeBoxRows - 1) / kDecodeBoxRows : 0;
        const uint32_t tx = SWAP ? (uint32_t)(p.a_bytes + nb * kDecodeBoxRows * kRowBytes)
                                 : (uint32_t)(kTileBytes + 2 * kTileBytes);
        for (int ks = 0; ks < p.kst; ++ks) {
          if (!mbar_wait(&empty_bar[s], ph ^ 1, &s_abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&full_bar[s], tx);
          uint8_t* a = ring + (size_t)s * p.stage_bytes;
          uint8_t* b = a + p.a_bytes;
          const int kx = ks * (FP8 ? 128 : 64);  // element coordinate along K
          const int wrow = un.e * p.N_w;
          if (SWAP) {
            if (MODE == 1) {  // 64 gate rows then 64 up rows of N-slice nt
              tma_load_2d(a, &tm_w, &full_bar[s], kx, wrow + un.nt * 64, pol_w);
              tma_load_2d(a + 64 * kRowBytes, &tm_w, &full_bar[s], kx, wrow + p.I + un.nt * 64, pol_w);
            } else {
              tma_load_2d(a, &tm_w, &full_bar[s], kx, wrow + un.nt * 128, pol_w);
              tma_load_2d(a + 64 * kRowBytes, &tm_w, &full_bar[s], kx, wrow + un.nt * 128 + 64, pol_w);
            }
            for (int bb = 0; bb < nb; ++bb)
              tma_load_2d(b + bb * kDecodeBoxRows * kRowBytes, &tm_x, &full_bar[s], kx,
                          un.row0 + bb * kDecodeBoxRows, pol_x);
          } else {
            tma_load_2d(a, &tm_x, &full_bar[s], kx, un.row0, pol_x);
            if (MODE == 1) {  // 128 gate rows then 128 up rows of N-slice nt
              tma_load_2d(b, &tm_w, &full_bar[s], kx, wrow + un.nt * 128, pol_w);
              tma_load_2d(b + kTileBytes, &tm_w, &full_bar[s], kx, wrow + p.I + un.nt * 128, pol_w);
            } else {
              tma_load_2d(b, &tm_w, &full_bar[s], kx, wrow + un.nt * 256, pol_w);
              tma_load_2d(b + kTileBytes, &tm_w, &full_bar[s], kx, wrow + un.nt * 256 + 128, pol_w);
            }
          }
          if (++s == p.stages) { s = 0; ph ^= 1; }
        }
      }
      if (!ok) {
        // Drain: every slot armed last and not consumed completes its copies.
        flag_status(p.status, MOE_ERR_TIMEOUT);
        for (int i = 0; i < p.stages; ++i) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&full_bar[i], 0) && !mbar_try_wait(&full_bar[i], 1) &&
                 clock64() - t0 < kSpinLimitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ====================================================== MMA issuer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      bool issued = false;
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        const Unit un = unit_of(u, s_off, s_up, p.E, p.nt, p.chunk);
        if (!mbar_wait(&tempty_bar[acc], aph ^ 1, &s_abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * kAccCols;
        const int n = SWAP ? ((un.rows + 15) / 16) * 16 : 256;
        const uint32_t idesc = make_idesc(n, FP8 ? 0u : 1u);
        for (int ks = 0; ks < p.kst; ++ks) {
          if (!mbar_wait(&full_bar[s], ph, &s_abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a = smem_u32(ring + (size_t)s * p.stage_bytes);
          const uint32_t b = a + p.a_bytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // four 32-byte K steps per 128-byte slice
            const uint64_t ad = sw128_desc(a + kk * 32);
            const uint64_t bd = sw128_desc(b + kk * 32);
            const uint32_t accum = (ks | kk) ? 1u : 0u;
            if (FP8) mma_e4m3(d, ad, bd, idesc, accum);
            else mma_bf16(d, ad, bd, idesc, accum);
          }
          issued = true;
          mma_commit(&empty_bar[s]);
          if (++s == p.stages) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[acc]);
        if (++acc == 2) { acc = 0; aph ^= 1; }
      }
      if (!ok) flag_status(p.status, MOE_ERR_TIMEOUT);
      if (issued) {  // all issued MMAs complete before TMEM can be released
        mma_commit(&drain_bar);
        const long long t0 = clock64();
        while (!mbar_try_wait(&drain_bar, 0) && clock64() - t0 < kSpinLimitCycles) {
        }
      }
    }
  } else {
    // ======================================================== epilogue
    const int q = warp & 3;            // TMEM lane quarter of this warp
    const int lrow = q * 32 + lane;    // accumulator row (TMEM lane)
    int acc = 0;
    uint32_t aph = 0;
    uint32_t xph = 0;  // phase of xch_bar (decode FC1 exchange)
    bool ok = true;
    for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
      const Unit un = unit_of(u, s_off, s_up, p.E, p.nt, p.chunk);
      if (!mbar_wait(&tfull_bar[acc], aph, &s_abort)) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + acc * kAccCols + ((uint32_t)(q * 32) << 16);
      const int wrow0 = un.e * p.N_w;
      if (SWAP) {
        // lane = weight row of the slice, columns = the unit's token rows
        const int ncols = ((un.rows + 15) / 16) * 16;
        if (MODE == 1) {
          const bool is_gate = lrow < 64;
          const int n = un.nt * 64 + (lrow & 63);  // output column (intermediate index)
          const float ws = FP8 ? p.w_scale[wrow0 + (is_gate ? n : p.I + n)] : 1.f;
          for (int c = 0; c < ncols; c += 16) {
            float v[16];
            tmem_ld16(tbase + c, v);
            tmem_ld_wait();
            if (!is_gate) {
#pragma unroll
              for (int t = 0; t < 16; ++t) s_xch[(lrow - 64) * 17 + t] = v[t] * ws;
            }
            // bounded sync of the 128 epilogue threads (up values written)
            mbar_arrive(&xch_bar);
            if (!mbar_wait(&xch_bar, xph, &s_abort)) { ok = false; break; }
            xph ^= 1;
            if (is_gate && n < p.I) {
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                const int r = un.row0 + c + t;
                if (c + t < un.rows) {
                  const float sa = FP8 ? p.a_scale[r] : 1.f;
                  const float g = v[t] * ws * sa;
                  const float up = s_xch[lrow * 17 + t] * sa;
                  reinterpret_cast<bf16*>(p.out)[(size_t)r * p.ldo + n] =
                      __float2bfloat16_rn(silu_f(g) * up);
                }
              }
            }
            // bounded sync (up values consumed before the next chunk)
            mbar_arrive(&xch_bar);
            if (!mbar_wait(&xch_bar, xph, &s_abort)) { ok = false; break; }
            xph ^= 1;
          }
          if (!ok) {
            flag_status(p.status, MOE_ERR_TIMEOUT);
            break;
          }
        } else {
          const int n = un.nt * 128 + lrow;
          const bool nvalid = n < p.n_out;
          const float ws = (FP8 && nvalid) ? p.w_scale[wrow0 + n] : 1.f;
          for (int c = 0; c < ncols; c += 16) {
            float v[16];
            tmem_ld16(tbase + c, v);
            tmem_ld_wait();
            if (nvalid) {
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                const int r = un.row0 + c + t;
                if (c + t < un.rows) {
                  float x = v[t] * ws * (FP8 ? p.a_scale[r] : 1.f);
                  if (IS_FC2 && p.topk_w) x *= p.topk_w[p.row_src[r]];
                  if (OUT_F32) {
                    reinterpret_cast<float*>(p.out)[(size_t)r * p.ldo + n] = x;
                  } else {
                    reinterpret_cast<bf16*>(p.out)[(size_t)r * p.ldo + n] = __float2bfloat16_rn(x);
                  }
                }
              }
            }
          }
        }
      } else {
        // lane = token row of the tile, columns = weight rows
        const int r = un.row0 + lrow;
        const bool rvalid = lrow < un.rows;
        const float sa = (FP8 && rvalid) ? p.a_scale[r] : 1.f;
        if (MODE == 1) {
          for (int c = 0; c < 128; c += 16) {
            float g[16], up[16];
            tmem_ld16(tbase + c, g);
            tmem_ld16(tbase + 128 + c, up);
            tmem_ld_wait();
            const int n0 = un.nt * 128 + c;
            if (rvalid) {
              uint32_t pk[8];
#pragma unroll
              for (int t = 0; t < 16; t += 2) {
                float o[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int n = min(n0 + t + h, p.I - 1);
                  const float gs = FP8 ? sa * p.w_scale[wrow0 + n] : 1.f;
                  const float us = FP8 ? sa * p.w_scale[wrow0 + p.I + n] : 1.f;
                  o[h] = silu_f(g[t + h] * gs) * (up[t + h] * us);
                }
                pk[t / 2] = pack2_bf16(o[0], o[1]);
              }
              bf16* dst = reinterpret_cast<bf16*>(p.out) + (size_t)r * p.ldo + n0;
              if (n0 + 16 <= p.I) {
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
              } else {
                for (int t = 0; t < 16 && n0 + t < p.I; ++t) {
                  const uint32_t w2 = pk[t / 2];
                  const uint16_t h = (t & 1) ? (uint16_t)(w2 >> 16) : (uint16_t)(w2 & 0xffffu);
                  reinterpret_cast<uint16_t*>(dst)[t] = h;
                }
              }
            }
          }
        } else {
          const float tw = (IS_FC2 && rvalid && p.topk_w) ? p.topk_w[p.row_src[r]] : 1.f;
          for (int c = 0; c < 256; c += 16) {
            float v[16];
            tmem_ld16(tbase + c, v);
            tmem_ld_wait();
            const int n0 = un.nt * 256 + c;
            if (rvalid && n0 < p.n_out) {
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                const float ws = FP8 ? p.w_scale[wrow0 + min(n0 + t, p.n_out - 1)] : 1.f;
                v[t] = v[t] * ws * sa * tw;
              }
              if (OUT_F32) {
                float* dst = reinterpret_cast<float*>(p.out) + (size_t)r * p.ldo + n0;
                if (n0 + 16 <= p.n_out) {
#pragma unroll
                  for (int t = 0; t < 16; t += 4)
                    reinterpret_cast<float4*>(dst)[t / 4] = make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]);
                } else {
                  for (int t = 0; t < 16 && n0 + t < p.n_out; ++t) dst[t] = v[t];
                }
              } else {
                bf16* dst = reinterpret_cast<bf16*>(p.out) + (size_t)r * p.ldo + n0;
                if (n0 + 16 <= p.n_out) {
                  uint32_t pk[8];
#pragma unroll
                  for (int t = 0; t < 16; t += 2) pk[t / 2] = pack2_bf16(v[t], v[t + 1]);
                  reinterpret_cast<uint4*>(dst)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                  reinterpret_cast<uint4*>(dst)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                } else {
                  for (int t = 0; t < 16 && n0 + t < p.n_out; ++t) dst[t] = __float2bfloat16_rn(v[t]);
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      if (++acc == 2) { acc = 0; aph ^= 1; }
    }
  }

  // ---- teardown: every role is done; release TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 2 * kAccCols);
}

// ------------------------------------------------------------------ host --
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                        &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool make_map(CUtensorMap* m, const void* base, bool fp8, int64_t rows, int64_t cols,
              int box_rows) {
  if (!g_encode) return false;
  const int elem = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * elem)};
  cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / elem), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool SWAP, int MODE, bool FP8>
cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& tx, const Params& p, int grid,
                       size_t smem, cudaStream_t st) {
  auto k = moe_tc_gemm_kernel<SWAP, MODE, FP8>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(k, dim3(grid), dim3(kThreads), smem, st, tw, tx, p);
}

template <bool SWAP, bool FP8>
cudaError_t launch_mode(int mode, const CUtensorMap& tw, const CUtensorMap& tx, const Params& p,
                        int grid, size_t smem, cudaStream_t st) {
  if (mode == 0) return launch_one<SWAP, 0, FP8>(tw, tx, p, grid, smem, st);
  if (mode == 1) return launch_one<SWAP, 1, FP8>(tw, tx, p, grid, smem, st);
  if (mode == 2) return launch_one<SWAP, 2, FP8>(tw, tx, p, grid, smem, st);
  return launch_one<SWAP, 3, FP8>(tw, tx, p, grid, smem, st);
}

}  // namespace

void engine_init_device() { std::call_once(g_encode_once, load_encode); }

cudaError_t launch_gemm_tc(int mode, bool fp8, bool decode, const void* a, const float* a_scale,
                           const void* w, const float* w_scale, const int32_t* offsets,
                           const int32_t* row_src, const float* topk_w, void* c, int E, int K,
                           int I, int N_out, int R_max, int T, int sms, int* status,
                           cudaStream_t st) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode || R_max == 0) return R_max == 0 ? cudaSuccess : cudaErrorNotSupported;
  if (E > kMaxExperts || K % 64 != 0) return cudaErrorNotSupported;
  const int elem = fp8 ? 1 : 2;
  const int N_w = (mode >= 2) ? N_out : 2 * I;  // weight rows per expert
  Params p{};
  p.offsets = offsets;
  p.row_src = row_src;
  p.topk_w = topk_w;
  p.a_scale = a_scale;
  p.w_scale = w_scale;
  p.out = c;
  p.ldo = N_out;
  p.E = E;
  p.R_max = R_max;
  p.I = I;
  p.N_w = N_w;
  p.n_out = N_out;
  p.kst = (K * elem + kRowBytes - 1) / kRowBytes;
  p.status = status;
  if (decode) {
    // Token rows per unit: an expert normally holds <= T rows (distinct
    // experts per token); larger segments are split into more units, so the
    // B tile of a unit always fits its ring slot.
    int chunk = T < kDecodeMaxN ? T : kDecodeMaxN;
    chunk = ((chunk < 1 ? 1 : chunk) + kDecodeBoxRows - 1) / kDecodeBoxRows * kDecodeBoxRows;
    if (mode == 1 && I % 64 != 0) return cudaErrorNotSupported;
    p.chunk = chunk;
    p.nt = (mode == 1) ? I / 64 : (N_out + 127) / 128;
    p.a_bytes = kTileBytes;
    p.stage_bytes = p.a_bytes + chunk * kRowBytes;
  } else {
    p.chunk = kTileRows;
    p.nt = (mode == 1) ? (I + 127) / 128 : (N_out + 255) / 256;
    p.a_bytes = kTileBytes;
    p.stage_bytes = 3 * kTileBytes;
  }
  const int static_smem = 8 * 1024;
  int stages = (kSmemLimit - static_smem - 1024) / p.stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorNotSupported;
  p.stages = stages;
  const size_t smem = (size_t)stages * p.stage_bytes + 1024;

  CUtensorMap tm_w, tm_x;
  if (!make_map(&tm_w, w, fp8, (int64_t)E * N_w, K, decode ? 64 : 128)) return cudaErrorNotSupported;
  if (!make_map(&tm_x, a, fp8, R_max, K, decode ? kDecodeBoxRows : 128)) return cudaErrorNotSupported;
  // upper bound on units: every expert's token chunks times the N tiles
  const int64_t chunks = (int64_t)(R_max + p.chunk - 1) / p.chunk + E;
  int64_t units = chunks * p.nt;
  int grid = (int)(units < sms ? units : sms);
  if (grid < 1) grid = 1;
  if (decode)
    return fp8 ? launch_mode<true, true>(mode, tm_w, tm_x, p, grid, smem, st)
               : launch_mode<true, false>(mode, tm_w, tm_x, p, grid, smem, st);
  return fp8 ? launch_mode<false, true>(mode, tm_w, tm_x, p, grid, smem, st)
             : launch_mode<false, false>(mode, tm_w, tm_x, p, grid, smem, st);
}

}  // namespace moe
