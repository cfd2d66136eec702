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

constexpr int kThreads = 192;
// Wide token tiles (256 token rows per unit): the producer, the MMA thread and
// eight epilogue warps (four per 128-row half).
constexpr int kThreadsWide = 320;
constexpr int kRowBytes = 128;       // one swizzle row: K slice of a stage
constexpr int kTileRows = 128;       // MMA M
constexpr int kTileBytes = kTileRows * kRowBytes;  // 16 KB
constexpr int kAccCols = 256;        // TMEM columns per accumulator buffer
constexpr int kMaxStages = 8;
constexpr int kDecodeMaxN = 128;     // token rows per decode unit
constexpr int kDecodeBoxRows = 16;   // token rows per TMA box (decode)
constexpr int kSmemLimit = 227 * 1024;

// One grouped GEMM of a launch.
struct JobP {
  const float* a_scale;  // per token row (E4M3)
  const float* w_scale;  // per weight row (E4M3)
  const int32_t* row_src;
  const float* topk_w;
  void* out;
  int ldo;    // output row stride (elements)
  int N_w;    // weight rows per expert
  int n_out;  // output columns
  int nt;     // N tiles per (expert, token chunk)
  int kst;    // K stages (kw 128-byte K atoms each)
};

struct Params {
  const int32_t* offsets;
  int E, I;
  int R_max;   // rows of the activation operands / outputs
  int chunk;   // token rows per unit (decode: the B tile height; prefill: 128)
  int stages;
  int stage_bytes;
  int a_bytes;  // bytes of the A region of a stage (kw atoms of a_atom bytes)
  int kw;       // 128-byte K atoms per stage (wider stages: longer runs per weight row)
  int a_atom;   // bytes of one A atom (128 rows x 128 B)
  int b_atom;   // bytes of one B atom
  int njobs;    // 1, or 2 for FC1 -> FC2 in one launch
  // Split-K (one job, fp32 rows): every unit is computed ksplit times, split
  // s over K stages [s kst / ksplit, (s + 1) kst / ksplit), into output
  // columns s * n_out ..; 1: no split.
  int ksplit;
  // Dynamic scheduling (fused launch): sched[0] is the unit counter, sched[1 + e]
  // counts finished FC1 epilogue warps (bf16) or units (E4M3) of expert e, and
  // sched[1 + E + e] is set once expert e's FC1 rows are quantised (E4M3).
  // NULL: static schedule.
  int* sched;
  // E4M3 fused launch: the bf16 FC1 rows are quantised per row into these
  // (the FC2 job's A operand and its scales).
  uint8_t* actq;
  float* act_scale;
  int* status;
  JobP job[2];
};


// The whole decode forward in one launch: the arguments (engine.h).
using MegaP = DecodeForward;

constexpr int kUnitRing = 4;  // claimed-unit slots between the roles




// TMA loads of one K slice of a unit into ring slot (a, b).
template <bool SWAP, int MODE>
MOE_DEV void issue_stage(uint8_t* a, uint8_t* b, uint64_t* bar, const CUtensorMap* tw,
                         const CUtensorMap* tx, const Unit& un, int kx, int wrow, int I, int nb,
                         uint64_t pol_w, uint64_t pol_x) {
  if (SWAP) {
    if (MODE == 1) {  // 64 gate rows then 64 up rows of N-slice nt
      tma_load_2d(a, tw, bar, kx, wrow + un.nt * 64, pol_w);
      tma_load_2d(a + 64 * kRowBytes, tw, bar, kx, wrow + I + un.nt * 64, pol_w);
    } else {
      tma_load_2d(a, tw, bar, kx, wrow + un.nt * 128, pol_w);
      tma_load_2d(a + 64 * kRowBytes, tw, bar, kx, wrow + un.nt * 128 + 64, pol_w);
    }
    for (int bb = 0; bb < nb; ++bb)
      tma_load_2d(b + bb * kDecodeBoxRows * kRowBytes, tx, bar, kx,
                  un.row0 + bb * kDecodeBoxRows, pol_x);
  } else {
    tma_load_2d(a, tx, bar, kx, un.row0, pol_x);
    if (MODE == 1) {  // 128 gate rows then 128 up rows of N-slice nt
      tma_load_2d(b, tw, bar, kx, wrow + un.nt * 128, pol_w);
      tma_load_2d(b + kTileBytes, tw, bar, kx, wrow + I + un.nt * 128, pol_w);
    } else {
      tma_load_2d(b, tw, bar, kx, wrow + un.nt * 256, pol_w);
      tma_load_2d(b + kTileBytes, tw, bar, kx, wrow + un.nt * 256 + 128, pol_w);
    }
  }
}

// Epilogue of one weight-streaming unit: TMEM -> registers -> fused op ->
// global memory (token tiles use epilogue_tile below).  Returns false if a
// bounded wait ran out.
template <bool SWAP, int MODE, bool FP8>
MOE_DEV bool epilogue_unit(const Unit& un, const JobP& j, int I, uint32_t tbase, int lrow,
                           float* s_xch, uint64_t* xch_bar, uint32_t& xph, volatile int* abort) {
  constexpr bool IS_FC2 = (MODE == 2 || MODE == 3);  // routing-weight epilogue
  constexpr bool OUT_F32 = (MODE == 2);              // fp32 output (else bf16)
  static_assert(SWAP, "token tiles use epilogue_tile");
  const int wrow0 = un.e * j.N_w;
  {
    // lane = weight row of the slice, columns = the unit's token rows
    const int ncols = ((un.rows + 15) / 16) * 16;
    if (MODE == 1) {
      const bool is_gate = lrow < 64;
      const int n = un.nt * 64 + (lrow & 63);  // output column (intermediate index)
      const float ws = FP8 ? j.w_scale[wrow0 + (is_gate ? n : I + n)] : 1.f;
      for (int c = 0; c < ncols; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
        tmem_ld_wait();
        if (!is_gate) {
#pragma unroll
          for (int t = 0; t < 16; ++t) s_xch[(lrow - 64) * 17 + t] = v[t] * ws;
        }
        // bounded sync of the 128 epilogue threads (up values written)
        mbar_arrive(xch_bar);
        if (!mbar_wait(xch_bar, xph, abort)) return false;
        xph ^= 1;
        if (is_gate && n < I) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int r = un.row0 + c + t;
            if (c + t < un.rows) {
              const float sa = FP8 ? j.a_scale[r] : 1.f;
              const float g = v[t] * ws * sa;
              const float up = s_xch[lrow * 17 + t] * sa;
              reinterpret_cast<bf16*>(j.out)[(size_t)r * j.ldo + n] =
                  __float2bfloat16_rn(silu_f(g) * up);
            }
          }
        }
        // bounded sync (up values consumed before the next chunk)
        mbar_arrive(xch_bar);
        if (!mbar_wait(xch_bar, xph, abort)) return false;
        xph ^= 1;
      }
    } else {
      const int n = un.nt * 128 + lrow;
      const bool nvalid = n < j.n_out;
      const float ws = (FP8 && nvalid) ? j.w_scale[wrow0 + n] : 1.f;
      for (int c = 0; c < ncols; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
        tmem_ld_wait();
        if (nvalid) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int r = un.row0 + c + t;
            if (c + t < un.rows) {
              float x = v[t] * ws * (FP8 ? j.a_scale[r] : 1.f);
              if (IS_FC2 && j.topk_w) x *= j.topk_w[j.row_src[r]];
              if (OUT_F32) {
                reinterpret_cast<float*>(j.out)[(size_t)r * j.ldo + n] = x;
              } else {
                // FC2 bf16 rows go back to (token, slot) order
                const int orow = (MODE == 3 && j.row_src) ? j.row_src[r] : r;
                reinterpret_cast<bf16*>(j.out)[(size_t)orow * j.ldo + n] = __float2bfloat16_rn(x);
              }
            }
          }
        }
      }
    }
  }
  return true;
}


// ------------------------------------------------ token-tile epilogue --
// What a token-tile epilogue thread needs besides the accumulator: its row,
// the row's FP8 activation scale, the routing weight and the output row of
// FC2.  Loaded before the thread waits for the accumulator, so these
// dependent global loads overlap the unit's main loop.
struct TileRow {
  int r;        // activation row
  int orow;     // output row
  bool valid;   // the row belongs to the unit
  float sa;     // E4M3 activation scale (1 for bf16)
  float tw;     // routing weight (FC2; else 1)
};

template <int MODE, bool FP8>
MOE_DEV TileRow tile_row(const Unit& un, const JobP& j, int lrow) {
  constexpr bool IS_FC2 = (MODE == 2 || MODE == 3);
  TileRow t;
  t.r = un.row0 + lrow;
  t.valid = lrow < un.rows;
  t.sa = (FP8 && t.valid) ? j.a_scale[t.r] : 1.f;
  const int src = (IS_FC2 && t.valid && j.row_src) ? j.row_src[t.r] : t.r;
  t.tw = (IS_FC2 && t.valid && j.topk_w) ? j.topk_w[src] : 1.f;
  t.orow = (MODE == 3) ? src : t.r;  // FC2 bf16 rows go back to (token, slot) order
  return t;
}

// Shared-memory staging of one epilogue warp: 32 rows x 32 bf16 columns.
constexpr int kStageWords = 32 * 4;  // uint4 per warp (2 KB)
// E4M3 token tiles: the unit's 256 weight-channel scales, per epilogue warp.
constexpr int kTileScales = 256;

// Loads the E4M3 channel scales of a token-tile unit into the warp's slot
// (FC1: the 128 gate then the 128 up channels of the N tile; else the N
// tile's 256 channels; 0 past the matrix), before the warp waits for the
// accumulator.  Scale rows are 16-byte aligned (the boundary checks it).
template <int MODE>
MOE_DEV void load_tile_scales(const Unit& un, const JobP& j, int I, int lane, float* wsc) {
  const float* base = j.w_scale + (size_t)un.e * j.N_w;
#pragma unroll
  for (int i = lane * 4; i < kTileScales; i += 128) {
    int col, lim;
    if (MODE == 1) {
      col = (i < 128 ? 0 : I) + un.nt * 128 + (i & 127);
      lim = (i < 128 ? 0 : I) + I;
      if (un.nt * 128 + (i & 127) >= I) col = lim;  // past the intermediate
    } else {
      col = un.nt * 256 + i;
      lim = j.n_out;
    }
    const float4 v = col < lim ? *reinterpret_cast<const float4*>(base + col)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(wsc + i) = v;
  }
  __syncwarp();
}

// Writes a warp's 32 rows x 32 bf16 columns to global memory in 64-byte row
// runs: each lane holds its row's 32 values as 16 packed words (pk); they go
// through the warp's shared-memory buffer (16-byte chunks XOR-swizzled by row
// pair, so neither side has bank conflicts) and come back as 8 rows x 64 bytes
// per store instruction -- instead of 32 rows x 16 bytes, a quarter of each
// sector.  dst(row) is the row's first column; rows whose `valid` is false
// are not written.
MOE_DEV void store_rows32(uint4* stg, int lane, const uint32_t (&pk)[16], bool valid, bf16* dst) {
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    stg[lane * 4 + (c ^ sw)] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  __syncwarp();
  const unsigned long long my = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = i * 8 + (lane >> 2), c = lane & 3;
    const uint4 v = stg[row * 4 + (c ^ ((row >> 1) & 3))];
    const unsigned long long base = __shfl_sync(0xffffffffu, my, row);
    const int ok = __shfl_sync(0xffffffffu, valid ? 1 : 0, row);
    if (ok) reinterpret_cast<uint4*>(base)[c] = v;
  }
  __syncwarp();
}

// silu(z) = z / (1 + e^-z) with the fast exponential and divide (the token
// tiles' FC1 epilogue is on the critical path; the result is rounded to bf16).
MOE_DEV float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Epilogue of one token-tile unit: lane = token row of the tile, columns =
// weight rows.  TMEM is read in rounds of 128 columns (64 with E4M3 scales,
// whose per-column loads need registers too) with 32-column loads, one wait
// per round; bf16 rows
// leave through store_rows32 (stg: this warp's staging buffer).
template <int MODE, bool FP8>
MOE_DEV void epilogue_tile(const Unit& un, const JobP& j, int I, uint32_t tbase,
                           const TileRow& t, int lane, uint4* stg, const float* wsc) {
  if (MODE == 1) {
    for (int c2 = 0; c2 < 128; c2 += 64) {
      float gg[64], uu[64];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        tmem_ld32(tbase + c2 + 32 * q, gg + 32 * q);
        tmem_ld32(tbase + 128 + c2 + 32 * q, uu + 32 * q);
      }
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        const int n0 = un.nt * 128 + c2 + cc;  // I % 64 == 0: 32 columns are all in or all out
        if (n0 >= I) continue;
        uint32_t pk[16];
#pragma unroll
        for (int t16 = 0; t16 < 32; t16 += 16) {
          // E4M3: the 16 gate and 16 up channel scales of these columns
          // (16-byte aligned rows; the same addresses in every lane)
          float gs[16], us[16];
#pragma unroll
          for (int v4 = 0; v4 < 16; v4 += 4) {
            if (FP8) {
              const int ci = c2 + cc + t16 + v4;  // column within the N tile
              const float4 a = *reinterpret_cast<const float4*>(wsc + ci);
              const float4 b = *reinterpret_cast<const float4*>(wsc + 128 + ci);
              gs[v4] = a.x * t.sa; gs[v4 + 1] = a.y * t.sa; gs[v4 + 2] = a.z * t.sa; gs[v4 + 3] = a.w * t.sa;
              us[v4] = b.x * t.sa; us[v4 + 1] = b.y * t.sa; us[v4 + 2] = b.z * t.sa; us[v4 + 3] = b.w * t.sa;
            } else {
              gs[v4] = gs[v4 + 1] = gs[v4 + 2] = gs[v4 + 3] = 1.f;
              us[v4] = us[v4 + 1] = us[v4 + 2] = us[v4 + 3] = 1.f;
            }
          }
#pragma unroll
          for (int tt = 0; tt < 16; tt += 2) {
            const int c = cc + t16 + tt;
            pk[(t16 + tt) / 2] = pack2_bf16(silu_fast(gg[c] * gs[tt]) * (uu[c] * us[tt]),
                                            silu_fast(gg[c + 1] * gs[tt + 1]) * (uu[c + 1] * us[tt + 1]));
          }
        }
        store_rows32(stg, lane, pk, t.valid,
                     reinterpret_cast<bf16*>(j.out) + (size_t)t.r * j.ldo + n0);
      }
    }
  } else {
    constexpr int RC = FP8 ? 64 : 128;  // columns per round
    const float f = t.sa * t.tw;
    for (int c4 = 0; c4 < 256; c4 += RC) {
      float vv[RC];
#pragma unroll
      for (int q = 0; q < RC / 32; ++q) tmem_ld32(tbase + c4 + 32 * q, vv + 32 * q);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < RC; cc += 32) {
        float* v = vv + cc;
        // bf16 outputs (FC1 raw 2I, FC2 H columns) are multiples of 64 columns,
        // so 32 columns are all in or all out; fp32 outputs (the router's 3E
        // logit columns among them) may end inside a chunk
        const int n0 = un.nt * 256 + c4 + cc;
        if (n0 >= j.n_out) continue;
        if (FP8) {
          // channel scales from the warp's slot (the same address in every lane)
#pragma unroll
          for (int tt = 0; tt < 32; tt += 4) {
            const float4 w = *reinterpret_cast<const float4*>(wsc + c4 + cc + tt);
            v[tt] *= w.x * f; v[tt + 1] *= w.y * f; v[tt + 2] *= w.z * f; v[tt + 3] *= w.w * f;
          }
        } else {
#pragma unroll
          for (int tt = 0; tt < 32; ++tt) v[tt] *= f;
        }
        if (MODE == 2) {  // fp32 rows (split s of a split-K launch: columns s * n_out ..)
          if (t.valid) {
            const int c0 = un.split * j.n_out;
            float* dst = reinterpret_cast<float*>(j.out) + (size_t)t.r * j.ldo + c0 + n0;
            // vector stores need a 16-byte row pitch (the router's 3E may not give one)
            if (n0 + 32 <= j.n_out && ((j.ldo | c0) & 3) == 0) {
#pragma unroll
              for (int tt = 0; tt < 32; tt += 4)
                reinterpret_cast<float4*>(dst)[tt / 4] =
                    make_float4(v[tt], v[tt + 1], v[tt + 2], v[tt + 3]);
            } else {
              for (int tt = 0; tt < 32 && n0 + tt < j.n_out; ++tt) dst[tt] = v[tt];
            }
          }
        } else {
          uint32_t pk[16];
#pragma unroll
          for (int tt = 0; tt < 32; tt += 2) pk[tt / 2] = pack2_bf16(v[tt], v[tt + 1]);
          store_rows32(stg, lane, pk, t.valid,
                       reinterpret_cast<bf16*>(j.out) + (size_t)t.orow * j.ldo + n0);
        }
      }
    }
  }
}

// ------------------------------------------ whole decode forward phases --
// Grid-wide barrier of a cooperative launch.  bar[0] counts arrivals, bar[1]
// is the generation; `gen` (thread 0) is the generation this CTA waits past.
// The CTA's writes before the barrier are visible to every CTA after it.
// Bounded: a wait that runs out records MOE_ERR_TIMEOUT and returns false.
MOE_DEV bool grid_sync(int* bar, unsigned& gen, int* status, volatile int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = true;
    __threadfence();
    const int g = (int)gen;
    if (atomicAdd(&bar[0], 1) == (int)gridDim.x - 1) {
      atomicExch(&bar[0], 0);
      __threadfence();
      atomicExch(&bar[1], g + 1);
    } else {
      const long long t0 = clock64();
      while (ld_acquire(&bar[1]) == g) {
        if (clock64() - t0 > kSpinLimitCycles) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) flag_status(status, MOE_ERR_TIMEOUT);
    gen = (unsigned)(g + 1);
    *s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return *s_ok != 0;
}

// rms_norm, one CTA per token row (the arithmetic of rmsnorm_kernel); on the
// E4M3 path also the per-token quantisation s = absmax / 448, q = e4m3(y / s).
template <bool FP8>
MOE_DEV void mega_rmsnorm(const MegaP& mp, float* red) {
  const int H = mp.H, nv = H >> 3;
  const uint4* wr = reinterpret_cast<const uint4*>(mp.norm_w);
  for (int t = blockIdx.x; t < mp.T; t += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const bf16*>(mp.x) + (size_t)t * H);
    uint4* yr = reinterpret_cast<uint4*>(static_cast<bf16*>(mp.xhat) + (size_t)t * H);
    float ss = 0.f;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      float f[8];
      unpack8_bf16(xr[v], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)H + mp.eps);
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
      uint2* qr = reinterpret_cast<uint2*>(mp.xq + (size_t)t * H);
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
      if (threadIdx.x == 0) mp.xscale[t] = s;
    }
  }
}

// Routing: from given logits, one warp per token; or a small router (E <=
// blockDim), one CTA per token: thread (g, e) sums the rows h = g, g + G, ...
// of W_r (G = blockDim / E), the G partial sums are added in g order.  Then
// the shared warp top-k.  `scratch` holds H + blockDim + E floats.
MOE_DEV void mega_route(const MegaP& mp, int E, float* scratch) {
  if (mp.ids_in) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int T = mp.T, k = mp.k;
  if (mp.logits) {
    for (int t = blockIdx.x * nw + warp; t < T; t += gridDim.x * nw) {
      float v[kTopkPer];
#pragma unroll
      for (int i = 0; i < kTopkPer; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          float x = 0.f;
          x += mp.logits[(size_t)t * E + e];
          if (mp.bias) x += mp.bias[e];
          v[i] = x;
        } else {
          v[i] = -FLT_MAX;
        }
      }
      warp_topk(v, E, k, lane, mp.ids + (size_t)t * k, mp.tw + (size_t)t * k);
    }
    return;
  }
  const int H = mp.H, tid = threadIdx.x;
  float* xs = scratch;
  float* ps = scratch + H;
  float* lg = ps + blockDim.x;
  const int G = blockDim.x / E, g = tid / E, e = tid % E;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const bf16*>(mp.xhat) + (size_t)t * H);
    for (int v = tid; v < H / 8; v += blockDim.x) {
      float f[8];
      unpack8_bf16(xr[v], f);
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[v * 8 + q] = f[q];
    }
    __syncthreads();
    float acc = 0.f;
    if (g < G)
      for (int h = g; h < H; h += G) acc = fmaf(xs[h], mp.router_w[(size_t)h * E + e], acc);
    ps[tid] = acc;
    __syncthreads();
    for (int ee = tid; ee < E; ee += blockDim.x) {
      float s = 0.f;
      for (int gg = 0; gg < G; ++gg) s += ps[gg * E + ee];
      if (mp.bias) s += mp.bias[ee];
      lg[ee] = s;
    }
    __syncthreads();
    if (warp == 0) {
      float v[kTopkPer];
#pragma unroll
      for (int i = 0; i < kTopkPer; ++i) {
        const int ex = lane + 32 * i;
        v[i] = ex < E ? lg[ex] : -FLT_MAX;
      }
      warp_topk(v, E, k, lane, mp.ids + (size_t)t * k, mp.tw + (size_t)t * k);
    }
    __syncthreads();
  }
}

// Stable counting sort of the T k pairs by expert, in CTA 0: counts with
// shared atomics, an exclusive scan, then warp 0 walks the pairs in order in
// batches of 32 and ranks equal experts inside a batch with __match_any_sync.
// `cnt` holds E + 1 ints.  Pairs with an expert outside [0, E) are dropped
// (row_of_pair = -1) and flagged as MOE_ERR_INVALID_ARG.
MOE_DEV void mega_permute(const MegaP& mp, int E, int* cnt, int* status) {
  if (blockIdx.x != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = mp.T * mp.k;
  const int32_t* ids = mp.ids_in ? mp.ids_in : mp.ids;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int q = threadIdx.x; q < R; q += blockDim.x) {
    const int e = ids[q];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else bad = true;
  }
  if (bad) flag_status(status, MOE_ERR_INVALID_ARG);
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int v = (e < E) ? cnt[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) {
        cnt[e] = carry + incl - v;
        mp.offsets[e] = carry + incl - v;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) mp.offsets[E] = carry;
    __syncwarp();
    const unsigned below = (1u << lane) - 1u;
    for (int pb = 0; pb < R; pb += 32) {
      const int q = pb + lane;
      const bool valid = q < R;
      const int e = valid ? ids[q] : -1;
      const bool ok = valid && e >= 0 && e < E;
      const unsigned grp = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
      if (ok) {
        const int r = cnt[e] + __popc(grp & below);
        mp.row_src[r] = q;
        mp.row_of_pair[q] = r;
      } else if (valid) {
        mp.row_of_pair[q] = -1;
      }
      __syncwarp();
      if (ok && (grp & below) == 0) cnt[e] += __popc(grp);
      __syncwarp();
    }
  }
}

// Row gather xp[r] = x_hat[row_src[r] / k] (E4M3 rows and scales on the FP8
// path), one warp per row, then an async-proxy fence for the TMA readers.
template <bool FP8>
MOE_DEV void mega_gather(const MegaP& mp, int E) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int R = min(mp.offsets[E], mp.T * mp.k);
  const int row_vec = mp.H * (FP8 ? 1 : 2) / 16;
  const uint4* src = reinterpret_cast<const uint4*>(FP8 ? (const void*)mp.xq : (const void*)mp.xhat);
  uint4* dst = reinterpret_cast<uint4*>(mp.xp);
  for (int r = blockIdx.x * nw + warp; r < R; r += gridDim.x * nw) {
    const int t = mp.row_src[r] / mp.k;
    const uint4* s = src + (size_t)t * row_vec;
    uint4* d = dst + (size_t)r * row_vec;
    for (int v = lane; v < row_vec; v += 32) d[v] = s[v];
    if (FP8 && lane == 0) mp.xp_scale[r] = mp.xscale[t];
  }
  fence_proxy_async_global();
}

// out[t, :] = bf16(sum_j y[t k + j, :]) over the pairs kept, fp32 in j order
// (the arithmetic of the combine kernel for (token, slot)-ordered rows).
MOE_DEV void mega_combine(const MegaP& mp) {
  const int H = mp.H, k = mp.k, g8 = H >> 3;
  const int64_t total = (int64_t)mp.T * g8;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = it / g8, g = it % g8;
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      if (mp.row_of_pair[t * k + j] < 0) continue;
      float f[8];
      unpack8_bf16(reinterpret_cast<const uint4*>(static_cast<const bf16*>(mp.y) + (t * k + j) * H)[g], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i] += f[i];
    }
    uint4 o;
    o.x = pack2_bf16(s[0], s[1]);
    o.y = pack2_bf16(s[2], s[3]);
    o.z = pack2_bf16(s[4], s[5]);
    o.w = pack2_bf16(s[6], s[7]);
    reinterpret_cast<uint4*>(mp.out)[it] = o;
  }
}

// Persistent grouped GEMM.  One launch runs job 0 (mode M0) and, when M1 >= 0,
// job 1 (mode M1) after it: units of job 0 come first in the unit order.
// Static schedule (p.sched == NULL): CTA c takes units c, c + grid, ...
// Dynamic schedule: the producer claims units from p.sched[0]; a unit of job 1
// for expert e first waits until every job-0 unit of expert e has finished its
// epilogue (p.sched[1 + e]), so job 1 may read job 0's output with TMA.  Since
// job-0 units are all claimed before any job-1 unit and a producer issues all
// loads of a unit before it claims the next, every wait ends.
// MEGA: the whole decode forward in this launch (cooperative, one CTA per SM):
// rms_norm, routing, permute and row gather before the FFN, the combine after
// it, each phase separated by a grid barrier (MegaP).
// WIDE (token tiles only): a unit is 256 token rows x the N tile, computed as
// two M = 128 MMAs per K step that share the weight slice in shared memory --
// per flop 2/3 of the operand bytes of the 128-row tile.  The two 256-column
// accumulators fill TMEM, so one unit's accumulators are live at a time and
// eight epilogue warps drain both halves at once.
template <bool SWAP, bool FP8, int M0, int M1, bool MEGA = false, bool WIDE = false>
__global__ void __launch_bounds__(WIDE ? kThreadsWide : kThreads, 1) moe_tc_gemm_kernel(
    const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_x0,
    const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_x1,
    const Params p, const MegaP mp) {
  static_assert(!WIDE || (!SWAP && !MEGA && M1 < 0), "wide tiles are single-job token tiles");
  static_assert(SWAP || M1 < 0, "token-tile launches run one job");
  constexpr int NJ = (M1 >= 0) ? 2 : 1;
  constexpr int NE = WIDE ? 8 : 4;     // epilogue warps
  constexpr int NACC = WIDE ? 1 : 2;   // accumulator buffers (each kAccCols; WIDE: both halves)
  extern __shared__ uint8_t dyn_smem[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_up[NJ][kMaxExperts + 1];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t ufull_bar[kUnitRing];
  __shared__ __align__(8) uint64_t uempty_bar[kUnitRing];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t xch_bar;
  __shared__ int s_uring[kUnitRing];
  __shared__ int s_last;  // E4M3 fused: this warpgroup finished an expert's FC1
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_xch[SWAP && (M0 == 1 || M1 == 1) ? 64 * 17 : 1];  // decode FC1: up values
  __shared__ uint4 s_stg[SWAP ? 1 : NE * kStageWords];  // token tiles: epilogue row staging
  __shared__ __align__(16) float s_wsc[(!SWAP && FP8) ? NE * kTileScales : 4];  // E4M3 channel scales
  __shared__ volatile int s_gok;  // MEGA: grid barrier result
  unsigned mega_gen = 0;          // MEGA: grid barrier generation (thread 0)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~(uintptr_t)1023);

  // ---- set-up: barriers and TMEM first (no global memory), then wait for
  // the previous kernel and build the unit tables from the expert offsets
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 32 * NE);
    }
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&ufull_bar[i], 1);
      mbar_init(&uempty_bar[i], 1 + NE);  // MMA thread + the epilogue warps
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&xch_bar, 128);
    s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_w0);
    prefetch_tmap(&tm_x0);
    if (NJ == 2) {
      prefetch_tmap(&tm_w1);
      prefetch_tmap(&tm_x1);
    }
  } else if (warp == 1) {
    tmem_alloc(&s_tmem, 2 * kAccCols);
    tmem_relinquish();
  }
  pdl_trigger();
  pdl_wait();
  if constexpr (MEGA) {
    // the forward's steps before the FFN; s_up and the ring are scratch here
    mega_rmsnorm<FP8>(mp, reinterpret_cast<float*>(&s_up[0][0]));
    grid_sync(mp.bar, mega_gen, p.status, &s_gok);
    mega_route(mp, p.E, reinterpret_cast<float*>(ring));
    grid_sync(mp.bar, mega_gen, p.status, &s_gok);
    mega_permute(mp, p.E, s_off, p.status);
    grid_sync(mp.bar, mega_gen, p.status, &s_gok);
    mega_gather<FP8>(mp, p.E);
    grid_sync(mp.bar, mega_gen, p.status, &s_gok);
    fence_proxy_async_global();  // gathered rows are read by TMA below
  }
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
  if (warp < NJ) {  // warp jb builds job jb's unit prefix
    const int jb = warp;
    const int nt = p.job[jb].nt;
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
      if (e < p.E) s_up[jb][e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_up[jb][p.E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int U0 = s_up[0][p.E];
  const int KS = (NJ == 1 && p.ksplit > 1) ? p.ksplit : 1;  // K splits
  const int U = NJ == 2 ? U0 + s_up[NJ - 1][p.E] : U0 * KS;

  // token tiles: the token chunks of one weight tile are consecutive units,
  // so the CTAs that share the tile start it together
  auto decode_unit = [&](int u) -> Unit {
    if (NJ == 2 && u >= U0) {
      Unit un = unit_of(u - U0, s_off, s_up[NJ - 1], p.E, p.job[NJ - 1].nt, p.chunk, !SWAP);
      un.job = 1;
      return un;
    }
    if (KS > 1) {
      const int sp = u / U0;
      Unit un = unit_of(u - sp * U0, s_off, s_up[0], p.E, p.job[0].nt, p.chunk, !SWAP);
      un.split = sp;
      return un;
    }
    return unit_of(u, s_off, s_up[0], p.E, p.job[0].nt, p.chunk, !SWAP);
  };
  // the unit's K stages [kb, ke)
  auto k_begin = [&](const Unit& un, int kst) -> int {
    return KS > 1 ? (int)(((int64_t)un.split * kst) / KS) : 0;
  };
  auto k_end = [&](const Unit& un, int kst) -> int {
    return KS > 1 ? (int)(((int64_t)(un.split + 1) * kst) / KS) : kst;
  };
  // Consumers read claimed units in order from the unit ring.
  auto next_unit = [&](int i) -> int {
    const int slot = i % kUnitRing;
    if (!mbar_wait(&ufull_bar[slot], (uint32_t)((i / kUnitRing) & 1), &s_abort)) return -2;
    return s_uring[slot];
  };

  if (warp == 0) {
    // ===================================================== TMA producer
    if (lane == 0) {
      const uint64_t pol_w = SWAP ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_x = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      uint32_t armed = 0, armed_ph = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        // claim the next unit and publish it to the other roles
        const int slot = i % kUnitRing;
        if (!mbar_wait(&uempty_bar[slot], (uint32_t)(((i / kUnitRing) & 1) ^ 1), &s_abort)) {
          ok = false;
          break;
        }
        int u = p.sched ? atomicAdd(p.sched, 1) : (int)blockIdx.x + i * (int)gridDim.x;
        if (u >= U) u = -1;
        s_uring[slot] = u;
        mbar_arrive(&ufull_bar[slot]);
        if (u < 0) break;
        const Unit un = decode_unit(u);
        const JobP& j = p.job[un.job];
        if (NJ == 2 && un.job == 1 && p.sched) {
          // wait until job 0 (FC1) has written every row of expert e
          const int cnt = s_off[un.e + 1] - s_off[un.e];
          // bf16: every FC1 epilogue warp of e has published its rows;
          // E4M3: e's rows are quantised
          const int need = FP8 ? 1 : ((cnt + p.chunk - 1) / p.chunk) * p.job[0].nt * 4;
          const int* flag = FP8 ? p.sched + 1 + p.E + un.e : p.sched + 1 + un.e;
          const long long t0 = clock64();
          while (ld_acquire(flag) < need) {
            if (s_abort || clock64() - t0 > kSpinLimitCycles) {
              s_abort = 1;
              ok = false;
              break;
            }
          }
          if (!ok) break;
          fence_proxy_async_global();
        }
        const int nb = SWAP ? (un.rows + kDecodeBoxRows - 1) / kDecodeBoxRows : 0;
        // WIDE: the second 128-row half of the token rows is loaded only when
        // the unit has rows there
        const bool half2 = WIDE && un.rows > kTileRows;
        const uint32_t tx = (uint32_t)p.kw *
                            (SWAP ? (uint32_t)(p.a_atom + nb * kDecodeBoxRows * kRowBytes)
                                  : (uint32_t)((half2 ? 2 : 1) * kTileBytes + 2 * kTileBytes));
        const CUtensorMap* tw = un.job ? &tm_w1 : &tm_w0;
        const CUtensorMap* tx_map = un.job ? &tm_x1 : &tm_x0;
        const int kb = k_begin(un, j.kst), ke = k_end(un, j.kst);
        for (int ks = kb; ks < ke; ++ks) {
          if (!mbar_wait(&empty_bar[s], ph ^ 1, &s_abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&full_bar[s], tx);
          uint8_t* a = ring + (size_t)s * p.stage_bytes;
          uint8_t* b = a + p.a_bytes;
          const int wrow = un.e * j.N_w;
          for (int w = 0; w < p.kw; ++w) {
            const int kx = (ks * p.kw + w) * (FP8 ? 128 : 64);  // element coordinate along K
            if ((un.job == 0 ? M0 : M1) == 1)
              issue_stage<SWAP, 1>(a + w * p.a_atom, b + w * p.b_atom, &full_bar[s], tw, tx_map, un,
                                   kx, wrow, p.I, nb, pol_w, pol_x);
            else
              issue_stage<SWAP, 0>(a + w * p.a_atom, b + w * p.b_atom, &full_bar[s], tw, tx_map, un,
                                   kx, wrow, p.I, nb, pol_w, pol_x);
            if (half2)  // token rows 128..255 of the unit, after the first half
              tma_load_2d(a + w * p.a_atom + kTileBytes, tx_map, &full_bar[s], kx,
                          un.row0 + kTileRows, pol_x);
          }
          armed |= 1u << s;
          armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
          if (++s == p.stages) { s = 0; ph ^= 1; }
        }
      }
      if (ok) ok = producer_tail(empty_bar, p.stages, s, ph, &s_abort);
      if (!ok) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        drain_armed(full_bar, p.stages, armed, armed_ph);
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
      for (int i = 0; ok; ++i) {
        const int u = next_unit(i);
        if (u == -2) { ok = false; break; }
        mbar_arrive(&uempty_bar[i % kUnitRing]);
        if (u < 0) break;
        const Unit un = decode_unit(u);
        const int kst = p.job[un.job].kst;
        const int kb = k_begin(un, kst), ke = k_end(un, kst);
        if (!mbar_wait(&tempty_bar[acc], aph ^ 1, &s_abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * kAccCols;
        const int n = SWAP ? ((un.rows + 15) / 16) * 16 : 256;
        const uint32_t idesc = make_idesc(n, FP8 ? 0u : 1u);
        const bool half2 = WIDE && un.rows > kTileRows;  // WIDE: rows 128..255 -> d + kAccCols
        for (int ks = kb; ks < ke; ++ks) {
          if (!mbar_wait(&full_bar[s], ph, &s_abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + (size_t)s * p.stage_bytes);
          const uint32_t b0 = a0 + p.a_bytes;
          for (int w = 0; w < p.kw; ++w) {
            const uint32_t a = a0 + w * p.a_atom, b = b0 + w * p.b_atom;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // four 32-byte K steps per 128-byte atom
              const uint64_t ad = sw128_desc(a + kk * 32);
              const uint64_t bd = sw128_desc(b + kk * 32);
              const uint32_t accum = ((ks - kb) | w | kk) ? 1u : 0u;
              if (FP8) mma_e4m3(d, ad, bd, idesc, accum);
              else mma_bf16(d, ad, bd, idesc, accum);
              if (half2) {
                const uint64_t ad2 = sw128_desc(a + kTileBytes + kk * 32);
                if (FP8) mma_e4m3(d + kAccCols, ad2, bd, idesc, accum);
                else mma_bf16(d + kAccCols, ad2, bd, idesc, accum);
              }
            }
          }
          issued = true;
          mma_commit(&empty_bar[s]);
          if (++s == p.stages) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[acc]);
        if (++acc == NACC) { acc = 0; aph ^= 1; }
      }
      if (ok) ok = accumulator_tail(tempty_bar, acc, aph, &s_abort, NACC);
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
    const int half = WIDE ? (warp - 2) >> 2 : 0;  // WIDE: token rows 128 * half ..
    int acc = 0;
    uint32_t aph = 0;
    uint32_t xph = 0;  // phase of xch_bar (decode FC1 exchange)
    for (int i = 0;; ++i) {
      const int u = next_unit(i);
      __syncwarp();
      if (lane == 0 && u != -2) mbar_arrive(&uempty_bar[i % kUnitRing]);
      if (u == -2) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      if (u < 0) break;
      Unit un = decode_unit(u);
      if (WIDE) {  // this warp's 128-row half of the unit (possibly empty)
        un.row0 += half * kTileRows;
        un.rows = max(0, min(kTileRows, un.rows - half * kTileRows));
      }
      // token tiles: the row's scale, routing weight and output row first
      TileRow trow{};
      float* wsc = s_wsc + ((!SWAP && FP8) ? (warp - 2) * kTileScales : 0);
      if constexpr (!SWAP) {
        if (un.rows > 0) {
          trow = tile_row<M0, FP8>(un, p.job[0], lrow);
          if constexpr (FP8) load_tile_scales<M0>(un, p.job[0], p.I, lane, wsc);
        }
      }
      if (!mbar_wait(&tfull_bar[acc], aph, &s_abort)) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t tbase =
          tmem + acc * kAccCols + (uint32_t)(half * kAccCols) + ((uint32_t)(q * 32) << 16);
      bool ok = true;
      if constexpr (!SWAP) {
        if (un.rows > 0)
          epilogue_tile<M0, FP8>(un, p.job[0], p.I, tbase, trow, lane,
                                 s_stg + (warp - 2) * kStageWords, wsc);
      } else if (un.job == 0) {
        ok = epilogue_unit<SWAP, M0, FP8>(un, p.job[0], p.I, tbase, lrow, s_xch, &xch_bar, xph,
                                          &s_abort);
      } else {
        ok = epilogue_unit<SWAP, (M1 >= 0 ? M1 : M0), FP8>(un, p.job[1], p.I, tbase, lrow, s_xch,
                                                           &xch_bar, xph, &s_abort);
      }
      if (!ok) {
        flag_status(p.status, MOE_ERR_TIMEOUT);
        break;
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      if (++acc == NACC) { acc = 0; aph ^= 1; }
      if (NJ == 2 && un.job == 0 && p.sched && !FP8) {
        // publish this warp's rows of the FC1 output to later TMA readers
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.sched + 1 + un.e, 1);
      }
      if (NJ == 2 && un.job == 0 && p.sched && FP8) {
        // count this unit; the warpgroup that completes expert e's last FC1
        // unit quantises e's rows (per row: s = absmax / 448, q = e4m3(a / s))
        __threadfence();
        mbar_arrive(&xch_bar);
        if (!mbar_wait(&xch_bar, xph, &s_abort)) { flag_status(p.status, MOE_ERR_TIMEOUT); break; }
        xph ^= 1;
        const int r0 = s_off[un.e], r1 = s_off[un.e + 1];
        if (lrow == 0) {
          const int units_e = ((r1 - r0 + p.chunk - 1) / p.chunk) * p.job[0].nt;
          s_last = (atomicAdd(p.sched + 1 + un.e, 1) + 1 == units_e) ? 1 : 0;
        }
        mbar_arrive(&xch_bar);
        if (!mbar_wait(&xch_bar, xph, &s_abort)) { flag_status(p.status, MOE_ERR_TIMEOUT); break; }
        xph ^= 1;
        if (s_last) {
          __threadfence();  // every CTA's rows of expert e are visible
          const bf16* act = reinterpret_cast<const bf16*>(p.job[0].out);
          for (int r = r0 + q; r < r1; r += 4) {  // warp q: rows q, q+4, ...
            const uint4* row = reinterpret_cast<const uint4*>(act + (size_t)r * p.I);
            float amax = 0.f;
            for (int v = lane; v < p.I / 8; v += 32) {
              float f[8];
              unpack8_bf16(__ldcg(row + v), f);
#pragma unroll
              for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            }
            amax = warp_max(amax);
            const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
            uint2* qrow = reinterpret_cast<uint2*>(p.actq + (size_t)r * p.I);
            for (int v = lane; v < p.I / 8; v += 32) {
              float f[8];
              unpack8_bf16(__ldcg(row + v), f);
              uint32_t lo = 0, hi = 0;
#pragma unroll
              for (int i = 0; i < 4; ++i) lo |= (uint32_t)f_to_e4m3(__fdiv_rn(f[i], sc)) << (8 * i);
#pragma unroll
              for (int i = 0; i < 4; ++i) hi |= (uint32_t)f_to_e4m3(__fdiv_rn(f[4 + i], sc)) << (8 * i);
              qrow[v] = make_uint2(lo, hi);
            }
            if (lane == 0) p.act_scale[r] = sc;
          }
          fence_proxy_async_global();
          __threadfence();
          mbar_arrive(&xch_bar);
          if (!mbar_wait(&xch_bar, xph, &s_abort)) { flag_status(p.status, MOE_ERR_TIMEOUT); break; }
          xph ^= 1;
          if (lrow == 0) atomicExch(p.sched + 1 + p.E + un.e, 1);
        }
      }
    }
  }

  if constexpr (MEGA) {
    grid_sync(mp.bar, mega_gen, p.status, &s_gok);  // every FC2 row is written
    mega_combine(mp);
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

}  // namespace

bool tc::encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
                    int64_t rows, int64_t cols, int box_cols, int box_rows, CUtensorMapSwizzle sw) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * elem_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

bool make_map(CUtensorMap* m, const void* base, bool fp8, int64_t rows, int64_t cols,
              int box_rows) {
  const int elem = fp8 ? 1 : 2;
  return tc::encode_map(m, base, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        elem, rows, cols, kRowBytes / elem, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool SWAP, bool FP8, int M0, int M1, bool WIDE = false>
cudaError_t launch_k(const CUtensorMap* maps, const Params& p, int grid, size_t smem,
                     cudaStream_t st) {
  auto k = moe_tc_gemm_kernel<SWAP, FP8, M0, M1, false, WIDE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(k, dim3(grid), dim3(WIDE ? kThreadsWide : kThreads), smem, st, maps[0],
                       maps[1], maps[2], maps[3], p, MegaP{});
}

template <bool SWAP, bool FP8, bool WIDE = false>
cudaError_t launch_mode(int mode, const CUtensorMap* maps, const Params& p, int grid, size_t smem,
                        cudaStream_t st) {
  if (mode == 0) return launch_k<SWAP, FP8, 0, -1, WIDE>(maps, p, grid, smem, st);
  if (mode == 1) return launch_k<SWAP, FP8, 1, -1, WIDE>(maps, p, grid, smem, st);
  if (mode == 2) return launch_k<SWAP, FP8, 2, -1, WIDE>(maps, p, grid, smem, st);
  return launch_k<SWAP, FP8, 3, -1, WIDE>(maps, p, grid, smem, st);
}

// Token rows per decode unit: an expert normally holds <= T rows (distinct
// experts per token); larger segments are split into more units, so the B
// tile of a unit always fits its ring slot.
int decode_chunk(int T) {
  int chunk = T < kDecodeMaxN ? T : kDecodeMaxN;
  return ((chunk < 1 ? 1 : chunk) + kDecodeBoxRows - 1) / kDecodeBoxRows * kDecodeBoxRows;
}

// Fills one job and its two tensor maps; false if the shape is not covered.
bool make_job(JobP* j, CUtensorMap* tw, CUtensorMap* tx, int mode, bool fp8, bool decode,
              const void* a, const float* a_scale, const void* w, const float* w_scale,
              const int32_t* row_src, const float* topk_w, void* c, int E, int K, int I,
              int N_out, int R_max) {
  if (K % 64 != 0) return false;
  const int elem = fp8 ? 1 : 2;
  j->a_scale = a_scale;
  j->w_scale = w_scale;
  j->row_src = row_src;
  j->topk_w = topk_w;
  j->out = c;
  j->ldo = N_out;
  j->N_w = (mode >= 2) ? N_out : 2 * I;
  j->n_out = N_out;
  j->kst = K * elem;  // bytes of K; set_ring() turns it into stages
  if (decode) {
    if (mode == 1 && I % 64 != 0) return false;
    j->nt = (mode == 1) ? I / 64 : (N_out + 127) / 128;
  } else {
    j->nt = (mode == 1) ? (I + 127) / 128 : (N_out + 255) / 256;
  }
  return make_map(tw, w, fp8, (int64_t)E * j->N_w, K, decode ? 64 : 128) &&
         make_map(tx, a, fp8, R_max, K, decode ? kDecodeBoxRows : 128);
}

// Ring geometry shared by the launches; converts each job's K bytes into
// stages of kw atoms.  wide: 256-row token tiles (two 16 KB token-row boxes
// and the 32 KB weight slice per K slice).
bool set_ring(Params* p, bool decode, int T, size_t* smem, bool wide = false) {
  // static shared memory: barriers and tables, plus the token tiles'
  // epilogue staging (2 KB per epilogue warp)
  const int static_smem =
      8 * 1024 + (decode ? 0 : (wide ? 8 : 4) * (kStageWords * 16 + kTileScales * 4));
  p->chunk = decode ? decode_chunk(T) : (wide ? 2 * kTileRows : kTileRows);
  p->a_atom = wide ? 2 * kTileBytes : kTileBytes;
  p->b_atom = decode ? p->chunk * kRowBytes : 2 * kTileBytes;
  int kw = 1;
  if (decode) {
    kw = 2;
    const char* env = getenv("MOE_DECODE_KW");
    if (env && (env[0] == '1' || env[0] == '2' || env[0] == '4')) kw = env[0] - '0';
    while (kw > 1 && (kSmemLimit - static_smem - 1024) / (kw * (p->a_atom + p->b_atom)) < 3) kw /= 2;
  }
  p->kw = kw;
  p->a_bytes = kw * p->a_atom;
  p->stage_bytes = kw * (p->a_atom + p->b_atom);
  int stages = (kSmemLimit - static_smem - 1024) / p->stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return false;
  p->stages = stages;
  *smem = (size_t)stages * p->stage_bytes + 1024;
  const int atom_bytes = kw * kRowBytes;
  for (int jb = 0; jb < p->njobs; ++jb)
    p->job[jb].kst = (p->job[jb].kst + atom_bytes - 1) / atom_bytes;
  return true;
}

// Self-test of the bounded waits: one thread waits on an mbarrier that no
// thread arrives on, for at most `limit` cycles, and records the timeout.
__global__ void wait_selftest_kernel(long long limit, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    if (!mbar_wait_limit(&bar, 0, &abort_flag, limit)) flag_status(status, MOE_ERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(long long limit_cycles, int* status, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(limit_cycles, status);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

void engine_init_device() { std::call_once(g_encode_once, load_encode); }

cudaError_t launch_gemm_tc(int mode, bool fp8, bool decode, const void* a, const float* a_scale,
                           const void* w, const float* w_scale, const int32_t* offsets,
                           const int32_t* row_src, const float* topk_w, void* c, int E, int K,
                           int I, int N_out, int R_max, int T, int sms, int* status,
                           cudaStream_t st, int* sched, int ksplit) {
  std::call_once(g_encode_once, load_encode);
  if (R_max == 0) return cudaSuccess;
  if (!g_encode || E > kMaxExperts) return cudaErrorNotSupported;
  if (ksplit < 1 || (ksplit > 1 && (decode || mode != MOE_GEMM_FC2))) return cudaErrorNotSupported;
  // prefill tiles start only after their predecessor has completed
  PdlOff no_pdl(!decode);
  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.I = I;
  p.R_max = R_max;
  p.njobs = 1;
  p.ksplit = 1;
  p.sched = decode ? nullptr : sched;  // one launch, one job: only the unit counter is used
  p.status = status;
  CUtensorMap maps[4];
  if (!make_job(&p.job[0], &maps[0], &maps[1], mode, fp8, decode, a, a_scale, w, w_scale, row_src,
                topk_w, c, E, K, I, N_out, R_max))
    return cudaErrorNotSupported;
  maps[2] = maps[0];
  maps[3] = maps[1];
  // Token tiles of 256 rows when the batch gives every SM at least two of
  // them (256-row units in the plain rows-per-expert estimate); else 128.
  bool wide = false;
  if (!decode) {
    const int64_t est = ((int64_t)R_max / (2 * kTileRows)) * p.job[0].nt;
    wide = est >= 2LL * sms;
    const char* env = getenv("MOE_WIDE_TILES");
    if (env && env[0] == '0') wide = false;
    if (env && env[0] == '1') wide = true;
  }
  size_t smem = 0;
  if (!set_ring(&p, decode, T, &smem, wide)) return cudaErrorNotSupported;
  if (ksplit > 1) {
    if (ksplit > p.job[0].kst) return cudaErrorNotSupported;  // every split has a K stage
    p.ksplit = ksplit;
    p.job[0].ldo = N_out * ksplit;
  }
  p.job[1] = p.job[0];
  // upper bound on units: every expert's token chunks times the N tiles
  const int64_t chunks = (int64_t)(R_max + p.chunk - 1) / p.chunk + E;
  const int64_t units = chunks * p.job[0].nt * p.ksplit;
  int grid = (int)(units < sms ? units : sms);
  if (grid < 1) grid = 1;
  if (decode)
    return fp8 ? launch_mode<true, true>(mode, maps, p, grid, smem, st)
               : launch_mode<true, false>(mode, maps, p, grid, smem, st);
  if (wide)
    return fp8 ? launch_mode<false, true, true>(mode, maps, p, grid, smem, st)
               : launch_mode<false, false, true>(mode, maps, p, grid, smem, st);
  return fp8 ? launch_mode<false, true>(mode, maps, p, grid, smem, st)
             : launch_mode<false, false>(mode, maps, p, grid, smem, st);
}

cudaError_t launch_decode_ffn_fused(bool fp8, const void* xp, const float* xp_scale,
                                    const void* w13, const float* w13_scale, const void* w2,
                                    const float* w2_scale, void* act, uint8_t* actq,
                                    float* act_scale, void* y, const int32_t* offsets,
                                    const int32_t* row_src, const float* topk_w, int* sched, int E,
                                    int H, int I, int R_max, int T, int sms, int* status,
                                    cudaStream_t st) {
  std::call_once(g_encode_once, load_encode);
  if (R_max == 0) return cudaSuccess;
  if (!g_encode || E > kMaxExperts || !sched || I % 8 != 0) return cudaErrorNotSupported;
  if (fp8 && (!actq || !act_scale || ((uintptr_t)actq & 15u))) return cudaErrorNotSupported;
  Params p{};
  p.offsets = offsets;
  p.E = E;
  p.I = I;
  p.R_max = R_max;
  p.njobs = 2;
  p.sched = sched;
  p.status = status;
  p.actq = actq;
  p.act_scale = act_scale;
  CUtensorMap maps[4];
  // FC1 reads x rows (E4M3 with per-row scales on the FP8 path) and writes bf16
  // rows; FC2 reads those rows (E4M3 copies and scales on the FP8 path)
  if (!make_job(&p.job[0], &maps[0], &maps[1], 1, fp8, true, xp, xp_scale, w13, w13_scale,
                row_src, nullptr, act, E, H, I, I, R_max) ||
      !make_job(&p.job[1], &maps[2], &maps[3], 3, fp8, true, fp8 ? (const void*)actq : act,
                act_scale, w2, w2_scale, row_src, topk_w, y, E, I, I, H, R_max))
    return cudaErrorNotSupported;
  size_t smem = 0;
  if (!set_ring(&p, true, T, &smem)) return cudaErrorNotSupported;
  return fp8 ? launch_k<true, true, 1, 3>(maps, p, sms, smem, st)
             : launch_k<true, false, 1, 3>(maps, p, sms, smem, st);
}

// Opt-in (MOE_MEGA=1): on GB300 the separate launches with programmatic
// dependent launch are faster for the decode workloads measured (a grid
// barrier costs about as much as a programmatic launch boundary, and the
// cooperative launch cannot overlap the previous kernel's tail).
bool decode_forward_mega_covers(int T, int H, int E, int k, bool logits, bool routed) {
  const char* env = getenv("MOE_MEGA");
  if (!(env && env[0] == '1')) return false;
  if (T < 1 || T > 64 || T * k > 512 || E > kMaxExperts) return false;
  if (logits || routed) return true;
  // small router: one CTA per token, W_r rows read by consecutive threads
  return H <= 8192 && (int64_t)H * E <= 65536 && E <= kThreads;
}

cudaError_t launch_decode_forward_mega(bool fp8, const DecodeForward& f, const void* w13,
                                       const float* w13_scale, const void* w2,
                                       const float* w2_scale, void* act, uint8_t* actq,
                                       float* act_scale, int* sched, int E, int I, int sms,
                                       int* status, cudaStream_t st) {
  std::call_once(g_encode_once, load_encode);
  const int T = f.T, H = f.H, R_max = T * f.k;
  if (!g_encode || !sched || !f.bar || I % 8 != 0 || R_max == 0 ||
      !decode_forward_mega_covers(T, H, E, f.k, f.logits != nullptr, f.ids_in != nullptr))
    return cudaErrorNotSupported;
  if (fp8 && (!actq || !act_scale || ((uintptr_t)actq & 15u))) return cudaErrorNotSupported;
  Params p{};
  p.offsets = f.offsets;
  p.E = E;
  p.I = I;
  p.R_max = R_max;
  p.njobs = 2;
  p.sched = sched;
  p.status = status;
  p.actq = actq;
  p.act_scale = act_scale;
  const float* topk_w = f.ids_in ? f.tw_in : f.tw;
  CUtensorMap maps[4];
  if (!make_job(&p.job[0], &maps[0], &maps[1], 1, fp8, true, f.xp, f.xp_scale, w13, w13_scale,
                f.row_src, nullptr, act, E, H, I, I, R_max) ||
      !make_job(&p.job[1], &maps[2], &maps[3], 3, fp8, true, fp8 ? (const void*)actq : act,
                act_scale, w2, w2_scale, f.row_src, topk_w, f.y, E, I, I, H, R_max))
    return cudaErrorNotSupported;
  size_t smem = 0;
  if (!set_ring(&p, true, T, &smem)) return cudaErrorNotSupported;
  auto k = fp8 ? moe_tc_gemm_kernel<true, true, 1, 3, true>
               : moe_tc_gemm_kernel<true, false, 1, 3, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // every CTA must be resident (grid barriers): one per SM
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorNotSupported;
  // scheduler counters and grid barrier words start at zero
  if (f.bar == sched + 2 * E + 1) {
    e = cudaMemsetAsync(sched, 0, (size_t)(2 * E + 3) * sizeof(int), st);
  } else {
    e = cudaMemsetAsync(sched, 0, (size_t)(2 * E + 1) * sizeof(int), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(f.bar, 0, 2 * sizeof(int), st);
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, maps[0], maps[1], maps[2], maps[3], p, f);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace moe
