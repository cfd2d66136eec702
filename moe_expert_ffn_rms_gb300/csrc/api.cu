// extern "C" entry points of libmoeffn.so: argument checks, workspace layout
// and the launch sequence of the MoE expert FFN forward.  No entry point
// allocates device memory or synchronises the host (except
// moe_device_status, which documents that it does).
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <string>

#include "common.cuh"
#include "engine.h"
#include "kernels.h"
#include "api_internal.h"

// Device status word: MOE_OK, or the first error a kernel flagged.
__device__ int g_moe_status = 0;

namespace {

thread_local std::string g_err;

moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = std::string(moe_status_string(s)) + ": " + buf;
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
struct DevInfo {
  bool checked = false;
  bool ok = false;
  int sms = 0;
  int* status = nullptr;  // device address of g_moe_status
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

#define MOE_REQ(cond, code, ...) \
  do {                           \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

#define MOE_CUDA(call, what)                 \
  do {                                       \
    cudaError_t _e = (call);                 \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

moe_status device_info(DevInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED_DEVICE, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.ok = (major == 10 && minor == 3);
    d.sms = sms;
    if (d.ok) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_moe_status)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(g_moe_status)");
      d.status = (int*)p;
      moe::engine_init_device();
    }
    d.checked = true;
    if (!d.ok)
      return fail(MOE_ERR_UNSUPPORTED_DEVICE, "device %d is compute capability %d.%d, need 10.3",
                  dev, major, minor);
  }
  if (!d.ok) return fail(MOE_ERR_UNSUPPORTED_DEVICE, "device %d is not compute capability 10.3", dev);
  *out = &d;
  return MOE_OK;
}

// ------------------------------------------------------------ shapes / ws --
moe_status check_shape(const moe_shape* s) {
  MOE_REQ(s != nullptr, MOE_ERR_INVALID_ARG, "shape is NULL");
  MOE_REQ(s->T >= 0 && s->H > 0 && s->E > 0 && s->I > 0 && s->top_k > 0, MOE_ERR_INVALID_ARG,
          "shape fields must be positive (T >= 0): T=%d H=%d E=%d I=%d top_k=%d", s->T, s->H,
          s->E, s->I, s->top_k);
  MOE_REQ(s->H % 64 == 0 && s->I % 64 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
          "H=%d and I=%d must be multiples of 64", s->H, s->I);
  MOE_REQ(s->E <= kMaxExperts, MOE_ERR_UNSUPPORTED_SHAPE, "E=%d > %d", s->E, kMaxExperts);
  MOE_REQ(s->top_k <= kMaxTopK && s->top_k <= s->E, MOE_ERR_UNSUPPORTED_SHAPE,
          "top_k=%d must be <= min(E=%d, %d)", s->top_k, s->E, kMaxTopK);
  MOE_REQ(s->wdtype == MOE_W_BF16 || s->wdtype == MOE_W_FP8_E4M3 || s->wdtype == MOE_W_NVFP4 ||
              s->wdtype == MOE_W_FP8_BLOCK,
          MOE_ERR_INVALID_ARG, "wdtype=%d", s->wdtype);
  MOE_REQ(s->wdtype != MOE_W_FP8_BLOCK ||
              (s->H % 256 == 0 && s->I % 128 == 0 && s->H <= 8192 && s->I <= 8192),
          MOE_ERR_UNSUPPORTED_SHAPE,
          "block-wise FP8 weights need H=%d a multiple of 256, I=%d a multiple of 128, both <= 8192",
          s->H, s->I);
  MOE_REQ(s->wdtype != MOE_W_NVFP4 || (s->H % 256 == 0 && s->I % 256 == 0),
          MOE_ERR_UNSUPPORTED_SHAPE, "NVFP4 weights need H=%d and I=%d to be multiples of 256", s->H,
          s->I);
  MOE_REQ(s->engine >= MOE_ENGINE_AUTO && s->engine <= MOE_ENGINE_PREFILL, MOE_ERR_INVALID_ARG,
          "engine=%d", s->engine);
  MOE_REQ((int64_t)s->T * s->top_k <= (1 << 24), MOE_ERR_UNSUPPORTED_SHAPE, "T*top_k too large");
  MOE_REQ(s->eps >= 0.f, MOE_ERR_INVALID_ARG, "eps < 0");
  return MOE_OK;
}

size_t router_ws_bytes(int T, int H, int E);

struct Ws {
  size_t xhat, xq, xscale, part, ids, tw, offsets, row_src, row_of_pair, perm_cnt, sched, xp,
      xp_scale, act, actq, act_scale, y, total;
};

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

Ws layout(const moe_shape* s) {
  const size_t T = s->T, H = s->H, E = s->E, I = s->I, k = s->top_k, R = T * k;
  const bool fb = s->wdtype == MOE_W_FP8_BLOCK;
  const bool f8 = s->wdtype == MOE_W_FP8_E4M3 || fb;
  // scales per row: one (per-token FP8) or one per 128-element group (block-wise)
  const size_t hs = fb ? H / 128 : 1, is = fb ? I / 128 : 1;
  Ws w{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += up256(bytes); return at; };
  w.xhat = take(T * H * 2);
  w.xq = take(f8 ? T * H : 0);
  w.xscale = take(f8 ? T * hs * 4 : 0);
  w.part = take(router_ws_bytes(s->T, s->H, s->E));
  w.ids = take(R * 4);
  w.tw = take(R * 4);
  w.offsets = take((E + 1) * 4);
  w.row_src = take(R * 4);
  w.row_of_pair = take(R * 4);
  w.perm_cnt = take(moe::permute_workspace_bytes(s->T, s->E, s->top_k));
  // fused decode FFN: unit counter + per-expert progress; then the two grid
  // barrier words of the one-launch decode forward
  w.sched = take((2 * E + 3) * 4);
  w.xp = take(R * H * (f8 ? 1 : 2));
  w.xp_scale = take(f8 ? R * hs * 4 : 0);
  w.act = take(R * I * 2);
  w.actq = take(f8 ? R * I : 0);
  w.act_scale = take(f8 ? R * is * 4 : 0);
  w.y = take(R * H * 2);  // FC2 output in bf16
  w.total = o;
  return w;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(base) + off);
}

// ---------------------------------------------------------------- router --
// Large batches compute the router logits on the tensor cores (W_r split into
// three bf16 pieces, one grouped GEMM with fp32 rows [T, 3E]); small ones use
// the fp32 SIMT router with split-K partial sums.
bool router_on_tensor_cores(int T) {
  const char* env = getenv("MOE_ROUTER_TC");
  if (env && env[0] == '0') return false;
  return T >= 256;
}

// K splits of the tensor-core router GEMM.  Its [T, 3E] output gives few
// token tiles (ceil(T / 128) units at 3E <= 256), each over all of K, so K is
// split until the units about fill the SMs, keeping at least 8 K stages of 64
// per split; top-k adds the splits' partial logits.
constexpr int kMaxRouterSplits = 8;

int router_ksplit(int T, int H, int E, int sms) {
  const int tiles = ((T + 127) / 128) * ((3 * E + 255) / 256);
  int s = sms / (tiles > 0 ? tiles : 1);
  const int kst = (H + 63) / 64;
  if (s > kst / 8) s = kst / 8;
  if (s > kMaxRouterSplits) s = kMaxRouterSplits;
  return s < 1 ? 1 : s;
}

size_t router_tc_bytes(int T, int H, int E) {
  return up256((size_t)3 * E * H * 2) + up256(2 * 4) +
         up256((size_t)T * 3 * E * kMaxRouterSplits * 4);
}

size_t router_ws_bytes(int T, int H, int E) {
  const int Tc = T > 0 ? T : 1;
  size_t n = (size_t)moe::route_splits(Tc, H, E) * Tc * E * 4;
  if (router_on_tensor_cores(T)) {
    const size_t tc = router_tc_bytes(T, H, E);
    if (tc > n) n = tc;
  }
  return up256(n);
}

// Enqueues the router logits of xhat into `ws` and returns how top-k reads
// them: logit(t, e) = sum_z part[z*zstride + t*tstride + e].
moe_status compute_router_logits(const void* xhat, const float* router_w, int T, int H, int E, void* ws,
                         DevInfo* dev, cudaStream_t st, const float** part, int* ks,
                         size_t* zstride, size_t* tstride) {
  if (router_on_tensor_cores(T)) {
    void* wt = ws;
    int32_t* seg = at<int32_t>(ws, up256((size_t)3 * E * H * 2));
    float* d = at<float>(ws, up256((size_t)3 * E * H * 2) + up256(2 * 4));
    MOE_CUDA(moe::launch_router_split(router_w, H, E, T, wt, seg, st), "router split launch");
    const int S = router_ksplit(T, H, E, dev->sms);
    cudaError_t e = moe::launch_gemm_tc(MOE_GEMM_FC2, false, false, xhat, nullptr, wt, nullptr,
                                        seg, nullptr, nullptr, d, 1, H, H, 3 * E, T, T, dev->sms,
                                        dev->status, st, nullptr, S);
    if (e == cudaSuccess) {  // row t: S splits x (hi, mid, lo) x E partial logits
      *part = d;
      *ks = 3 * S;
      *zstride = (size_t)E;
      *tstride = (size_t)3 * E * S;
      return MOE_OK;
    }
    if (e != cudaErrorNotSupported) return cuda_fail(e, "router GEMM launch");
  }
  *ks = moe::route_splits(T, H, E);
  MOE_CUDA(moe::launch_router_logits(xhat, router_w, T, H, E, *ks, (float*)ws, st),
           "router launch");
  *part = (const float*)ws;
  *zstride = (size_t)T * E;
  *tstride = (size_t)E;
  return MOE_OK;
}

// Router (when router_w is given) + softmax / top-k / renorm into ids, w.
moe_status route_topk_impl(const void* xhat, const float* router_w, const float* logits_in,
                           const float* bias, int T, int H, int E, int k, int32_t* ids, float* w,
                           float* logits_out, void* ws, DevInfo* dev, cudaStream_t st) {
  if (!logits_in && !router_on_tensor_cores(T) && moe::route_small(H, E)) {
    MOE_CUDA(moe::launch_route_small(xhat, router_w, bias, T, H, E, k, ids, w, logits_out, st),
             "router launch");
    return MOE_OK;
  }
  const float* part = logits_in;
  int ks = 1;
  size_t zs = 0, ts = 0;
  if (!logits_in) {
    moe_status rc = compute_router_logits(xhat, router_w, T, H, E, ws, dev, st, &part, &ks, &zs, &ts);
    if (rc != MOE_OK) return rc;
  }
  MOE_CUDA(moe::launch_topk(part, ks, bias, T, E, k, ids, w, logits_out, st, zs, ts),
           "top-k launch");
  return MOE_OK;
}

int pick_engine(const moe_shape* s) {
  if (s->engine != MOE_ENGINE_AUTO) return s->engine;
  const char* env = getenv("MOE_FORCE_ENGINE");
  if (env && !strcmp(env, "decode")) return MOE_ENGINE_DECODE;
  if (env && !strcmp(env, "prefill")) return MOE_ENGINE_PREFILL;
  // Average rows per expert; the decode engine streams weights with the
  // tokens as the narrow operand, the prefill engine tiles the tokens.
  const double rows_per_expert = (double)s->T * s->top_k / s->E;
  return rows_per_expert <= 96.0 ? MOE_ENGINE_DECODE : MOE_ENGINE_PREFILL;
}

// Grouped GEMM dispatch: tcgen05 engines where the shape allows, else SIMT.
// `sched`: NULL, or a zeroed int the token-tile engine claims its units from.
moe_status run_gemm(const moe_shape* s, int mode, int engine, const void* a, const float* a_scale,
                    const void* w, const float* w_scale, const int32_t* offsets,
                    const int32_t* row_src, const float* topk_w, void* c, int R_max, int sms,
                    int* status, cudaStream_t st, int32_t* sched = nullptr) {
  const bool f8 = s->wdtype == MOE_W_FP8_E4M3;
  const bool fc2 = mode >= MOE_GEMM_FC2;
  const int K = fc2 ? s->I : s->H;
  const int N_out = fc2 ? s->H : (mode == MOE_GEMM_FC1_SILU ? s->I : 2 * s->I);
  cudaError_t e = cudaErrorNotSupported;
  const char* env = getenv("MOE_FORCE_SIMT");
  const bool simt_only = env && env[0] == '1';
  if (!simt_only)
    e = moe::launch_gemm_tc(mode, f8, engine == MOE_ENGINE_DECODE, a, a_scale, w, w_scale,
                            offsets, row_src, topk_w, c, s->E, K, s->I, N_out, R_max, s->T, sms,
                            status, st, sched);
  if (e == cudaErrorNotSupported)
    e = moe::launch_gemm_simt(mode, f8, a, a_scale, w, w_scale, offsets, row_src, topk_w, c, s->E,
                              K, s->I, N_out, R_max, st);
  if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM launch");
  return MOE_OK;
}

// FC1 + silu_and_mul then FC2 + routing weight (bf16 rows in (token, slot)
// order).  `sched` (1 + 2E ints) must be zero: the fused decode launch uses
// all of it, the token-tile engine sched[0] (FC1) and sched[1] (FC2) as unit
// counters; actq / act_scale are the FP8 path's scratch.
moe_status ffn_impl(const moe_shape* s, int engine, bool fuse, const void* xp,
                    const float* xp_scale, const void* w13, const float* w13_scale, const void* w2,
                    const float* w2_scale, const int32_t* offsets, const int32_t* row_src,
                    const float* tw, void* act, void* y, int32_t* sched, uint8_t* actq,
                    float* act_scale, DevInfo* dev, cudaStream_t st) {
  const bool f8 = s->wdtype == MOE_W_FP8_E4M3;
  const int T = s->T, H = s->H, E = s->E, I = s->I, R = s->T * s->top_k;
  if (s->wdtype == MOE_W_FP8_BLOCK) {
    // block-wise FP8; the FC2 input is E4M3 codes (actq) with one scale per
    // 128 columns.  Decode engine: one persistent launch (FC1 quantises in
    // its epilogue).  Prefill engine: FC1 tiles -> bf16 act, quantisation,
    // FC2 tiles.
    if (engine == MOE_ENGINE_PREFILL)
      MOE_CUDA(moe::launch_prefill_ffn_fp8b(static_cast<const uint8_t*>(xp), xp_scale,
                                            static_cast<const uint8_t*>(w13), w13_scale,
                                            static_cast<const uint8_t*>(w2), w2_scale, act, actq,
                                            act_scale, y, offsets, row_src, tw, E, H, I, R,
                                            dev->sms, dev->status, st),
               "block-wise FP8 FFN launch");
    else
      MOE_CUDA(moe::launch_decode_ffn_fp8b(static_cast<const uint8_t*>(xp), xp_scale,
                                           static_cast<const uint8_t*>(w13), w13_scale,
                                           static_cast<const uint8_t*>(w2), w2_scale, actq,
                                           act_scale, y, offsets, row_src, tw, sched, E, H, I, R, T,
                                           dev->sms, dev->status, st),
               "block-wise FP8 FFN launch");
    return MOE_OK;
  }
  if (fuse) {
    // one persistent launch (FC2 units wait per expert for FC1)
    cudaError_t e = moe::launch_decode_ffn_fused(f8, xp, xp_scale, w13, w13_scale, w2, w2_scale,
                                                 act, actq, act_scale, y, offsets, row_src, tw,
                                                 sched, E, H, I, R, T, dev->sms, dev->status, st);
    if (e == cudaSuccess) return MOE_OK;
    if (e != cudaErrorNotSupported) return cuda_fail(e, "fused decode FFN launch");
  }
  int32_t* sched_fc1 = (engine == MOE_ENGINE_PREFILL && sched) ? sched : nullptr;
  int32_t* sched_fc2 = sched_fc1 ? sched + 1 : nullptr;
  moe_status rc = run_gemm(s, MOE_GEMM_FC1_SILU, engine, xp, xp_scale, w13, w13_scale, offsets,
                           row_src, nullptr, act, R, dev->sms, dev->status, st, sched_fc1);
  if (rc != MOE_OK) return rc;
  // FP8: per-row quantisation of the bf16 intermediate before FC2
  const void* a2 = act;
  if (f8) {
    MOE_CUDA(moe::launch_quant_rows(act, R, I, actq, act_scale, offsets + E, st), "quant launch");
    a2 = actq;
  }
  return run_gemm(s, MOE_GEMM_FC2_BF16, engine, a2, act_scale, w2, w2_scale, offsets, row_src, tw,
                  y, R, dev->sms, dev->status, st, sched_fc2);
}

bool fuse_decode(const moe_shape* s, int engine) {
  const char* fuse_env = getenv("MOE_FUSE");
  const char* simt_env = getenv("MOE_FORCE_SIMT");
  return engine == MOE_ENGINE_DECODE && !(fuse_env && fuse_env[0] == '0') &&
         !(simt_env && simt_env[0] == '1');
}

// Block and matrix scales of NVFP4 expert weights (moe_ffn_forward_nvfp4).
struct Nvfp4Scales {
  const uint8_t* w13_sb;
  const float* w13_sg;
  const uint8_t* w2_sb;
  const float* w2_sg;
};

moe_status forward_impl(const moe_shape* s, const void* x, const void* norm_w, const float* router_w,
                        const float* router_logits, const float* router_bias,
                        const int32_t* ids_in, const float* tw_in, const void* w13, const void* w2,
                        const float* w13_scale, const float* w2_scale, void* out,
                        int32_t* ids_out, float* tw_out, void* workspace, size_t ws_bytes,
                        moe_stream_t stream, const Nvfp4Scales* nv = nullptr) {
  moe_status rc = check_shape(s);
  if (rc != MOE_OK) return rc;
  const bool fb = s->wdtype == MOE_W_FP8_BLOCK;
  const bool f8 = s->wdtype == MOE_W_FP8_E4M3 || fb;  // E4M3 activations
  MOE_REQ((nv != nullptr) == (s->wdtype == MOE_W_NVFP4), MOE_ERR_INVALID_ARG,
          "NVFP4 weights (wdtype=2) go through moe_ffn_forward_nvfp4, other formats do not");
  MOE_REQ(!nv || (nv->w13_sb && nv->w13_sg && nv->w2_sb && nv->w2_sg), MOE_ERR_INVALID_ARG,
          "NVFP4 block and matrix scales must be non-NULL");
  MOE_REQ(!nv || (aligned16(nv->w13_sb) && aligned16(nv->w2_sb)), MOE_ERR_INVALID_ARG,
          "NVFP4 block scales must be 16-byte aligned");
  const bool routed = ids_in != nullptr;
  MOE_REQ(x && norm_w && w13 && w2 && out && workspace, MOE_ERR_INVALID_ARG,
          "x, norm_w, w13, w2, out and workspace must be non-NULL");
  if (routed) {
    MOE_REQ(tw_in != nullptr, MOE_ERR_INVALID_ARG, "topk_w is NULL");
  } else {
    MOE_REQ((router_w != nullptr) != (router_logits != nullptr), MOE_ERR_INVALID_ARG,
            "give exactly one of router_w and router_logits");
  }
  MOE_REQ(!f8 || (w13_scale && w2_scale), MOE_ERR_INVALID_ARG, "FP8 weights need w13_scale and w2_scale");
  MOE_REQ(aligned16(x) && aligned16(norm_w) && aligned16(w13) && aligned16(w2) && aligned16(out),
          MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  MOE_REQ(!f8 || (aligned16(w13_scale) && aligned16(w2_scale)), MOE_ERR_INVALID_ARG,
          "FP8 weight scales must be 16-byte aligned");
  MOE_REQ(((uintptr_t)workspace & 255u) == 0, MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const Ws L = layout(s);
  MOE_REQ(ws_bytes >= L.total, MOE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", ws_bytes,
          L.total);
  DevInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  if (s->T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int T = s->T, H = s->H, E = s->E, I = s->I, k = s->top_k, R = T * k;
  const int engine = pick_engine(s);
  // The prefill forward runs without programmatic dependent launch: each
  // kernel starts after its predecessor has completed (the launch overlap is
  // worth ~1% there; decode, where it matters, keeps it).
  PdlOff no_pdl(engine == MOE_ENGINE_PREFILL);

  bf16* xhat = at<bf16>(workspace, L.xhat);
  uint8_t* xq = f8 ? at<uint8_t>(workspace, L.xq) : nullptr;
  float* xscale = f8 ? at<float>(workspace, L.xscale) : nullptr;
  int32_t* ids = ids_out ? ids_out : at<int32_t>(workspace, L.ids);
  float* tw = tw_out ? tw_out : at<float>(workspace, L.tw);
  int32_t* offsets = at<int32_t>(workspace, L.offsets);
  int32_t* row_src = at<int32_t>(workspace, L.row_src);
  int32_t* row_of_pair = at<int32_t>(workspace, L.row_of_pair);
  void* xp = at<void>(workspace, L.xp);
  float* xp_scale = f8 ? at<float>(workspace, L.xp_scale) : nullptr;
  bf16* act = at<bf16>(workspace, L.act);
  uint8_t* actq = f8 ? at<uint8_t>(workspace, L.actq) : nullptr;
  float* act_scale = f8 ? at<float>(workspace, L.act_scale) : nullptr;
  bf16* y = at<bf16>(workspace, L.y);
  int32_t* perm_cnt = at<int32_t>(workspace, L.perm_cnt);
  int32_t* sched = at<int32_t>(workspace, L.sched);
  // FC1 and FC2 run in one persistent launch on the decode engine (bf16),
  // unless MOE_FUSE=0 or the SIMT engine is forced.
  const bool fuse = fuse_decode(s, engine);

  // Small decode batches, opt-in: a1..a8 in one cooperative launch
  if (!nv && !fb && fuse &&
      moe::decode_forward_mega_covers(T, H, E, k, router_logits != nullptr, routed)) {
    moe::DecodeForward f{};
    f.x = x;
    f.norm_w = norm_w;
    f.eps = s->eps;
    f.T = T;
    f.H = H;
    f.k = k;
    f.logits = routed ? nullptr : router_logits;
    f.router_w = routed ? nullptr : router_w;
    f.bias = routed ? nullptr : router_bias;
    f.ids_in = routed ? ids_in : nullptr;
    f.tw_in = routed ? tw_in : nullptr;
    f.xhat = xhat;
    f.xq = xq;
    f.xscale = xscale;
    f.ids = ids;
    f.tw = tw;
    f.offsets = offsets;
    f.row_src = row_src;
    f.row_of_pair = row_of_pair;
    f.xp = xp;
    f.xp_scale = xp_scale;
    f.y = y;
    f.out = out;
    f.bar = sched + 2 * E + 1;
    cudaError_t e = moe::launch_decode_forward_mega(f8, f, w13, w13_scale, w2, w2_scale, act, actq,
                                                    act_scale, sched, E, I, dev->sms, dev->status, st);
    if (e == cudaSuccess) return MOE_OK;
    if (e != cudaErrorNotSupported) return cuda_fail(e, "decode forward launch");
  }
  // a1: rms_norm (+ E4M3 quantisation of x_hat: per token on the FP8 path,
  // per 128-element group on the block-wise FP8 path)
  if (fb)
    MOE_CUDA(moe::launch_rmsnorm_q128(x, norm_w, T, H, s->eps, xhat, xq, xscale, st),
             "rmsnorm launch");
  else
    MOE_CUDA(moe::launch_rmsnorm(x, norm_w, T, H, s->eps, xhat, xq, xscale, st), "rmsnorm launch");
  // a2 + a3: router logits, softmax, top-k, renorm
  if (routed) {
    ids = const_cast<int32_t*>(ids_in);
    tw = const_cast<float*>(tw_in);
  } else {
    rc = route_topk_impl(xhat, router_w, router_logits, router_bias, T, H, E, k, ids, tw, nullptr,
                         at<void>(workspace, L.part), dev, st);
    if (rc != MOE_OK) return rc;
  }
  // a4: permute + gather of the (quantised) token rows
  MOE_CUDA(moe::launch_permute_any(ids, T, E, k, offsets, row_src, row_of_pair, perm_cnt,
                                   dev->status, st, sched, 2 * E + 1),
           "permute launch");
  if (nv) {
    // NVFP4 weights: fp16 rows for the fp16 tensor-core GEMMs, one fused launch
    MOE_CUDA(moe::launch_gather_rows_f16(offsets, E, row_src, k, R, H, xhat, xp, st),
             "gather launch");
    MOE_CUDA(moe::launch_decode_ffn_nvfp4(xp, static_cast<const uint8_t*>(w13), nv->w13_sb, nv->w13_sg,
                                          static_cast<const uint8_t*>(w2), nv->w2_sb, nv->w2_sg, act,
                                          y, offsets, row_src, tw, sched, E, H, I, R, T, dev->sms,
                                          dev->status, st),
             "NVFP4 FFN launch");
  } else {
    MOE_CUDA(moe::launch_gather_rows(offsets, E, row_src, k, R, f8 ? (const void*)xq : (const void*)xhat,
                                     xp, H * (f8 ? 1 : 2), xscale, xp_scale, st, fb ? H / 128 : 1),
             "gather launch");
    // a5 + a6 + a7: FC1 + silu_and_mul, FC2 + routing weight
    rc = ffn_impl(s, engine, fuse, xp, xp_scale, w13, w13_scale, w2, w2_scale, offsets, row_src, tw,
                  act, y, sched, actq, act_scale, dev, st);
    if (rc != MOE_OK) return rc;
  }
  // a8: combine (fp32 sum in slot order, one bf16 rounding)
  MOE_CUDA(moe::launch_combine(y, true, true, row_of_pair, T, k, H, out, st), "combine launch");
  return MOE_OK;
}

}  // namespace

namespace moe {
moe_status api_fail(moe_status s, const char* msg) { return fail(s, "%s", msg); }
moe_status api_check_shape(const moe_shape* shape) { return check_shape(shape); }
}  // namespace moe

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

int64_t moe_launch_count(void) { return (int64_t)launch_count(); }

const char* moe_last_error(void) { return g_err.c_str(); }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "MOE_ERR_UNSUPPORTED_DEVICE";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_check_device(void) {
  DevInfo* d = nullptr;
  return device_info(&d);
}

moe_status moe_device_status(int32_t* status_out, int32_t clear) {
  MOE_REQ(status_out != nullptr, MOE_ERR_INVALID_ARG, "status_out is NULL");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  int v = 0;
  MOE_CUDA(cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost), "read status word");
  *status_out = v;
  if (clear) {
    int z = 0;
    MOE_CUDA(cudaMemcpy(d->status, &z, sizeof(int), cudaMemcpyHostToDevice), "clear status word");
  }
  return MOE_OK;
}

moe_status moe_selftest_wait_timeout(int64_t limit_cycles, moe_stream_t stream) {
  MOE_REQ(limit_cycles > 0 && limit_cycles <= (int64_t)1 << 32, MOE_ERR_INVALID_ARG,
          "limit_cycles must be in (0, 2^32]");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_wait_selftest(limit_cycles, d->status, (cudaStream_t)stream),
           "self-test launch");
  return MOE_OK;
}

size_t moe_ffn_workspace_size(const moe_shape* shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  return layout(shape).total;
}

moe_status moe_ffn_forward(const moe_shape* shape, const void* x, const void* norm_w,
                           const float* router_w, const float* router_logits,
                           const float* router_bias, const void* w13, const void* w2,
                           const float* w13_scale, const float* w2_scale, void* out,
                           int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream) {
  return forward_impl(shape, x, norm_w, router_w, router_logits, router_bias, nullptr, nullptr,
                      w13, w2, w13_scale, w2_scale, out, topk_ids_out, topk_w_out, workspace,
                      workspace_bytes, stream);
}

moe_status moe_ffn_forward_routed(const moe_shape* shape, const void* x, const void* norm_w,
                                  const int32_t* topk_ids, const float* topk_w, const void* w13,
                                  const void* w2, const float* w13_scale, const float* w2_scale,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream) {
  if (topk_ids == nullptr) return fail(MOE_ERR_INVALID_ARG, "topk_ids is NULL");
  return forward_impl(shape, x, norm_w, nullptr, nullptr, nullptr, topk_ids, topk_w, w13, w2,
                      w13_scale, w2_scale, out, nullptr, nullptr, workspace, workspace_bytes,
                      stream);
}

moe_status moe_ffn_forward_nvfp4(const moe_shape* shape, const void* x, const void* norm_w,
                                 const float* router_w, const float* router_logits,
                                 const float* router_bias, const uint8_t* w13, const uint8_t* w13_sb,
                                 const float* w13_sg, const uint8_t* w2, const uint8_t* w2_sb,
                                 const float* w2_sg, void* out, int32_t* topk_ids_out,
                                 float* topk_w_out, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  MOE_REQ(shape != nullptr && shape->wdtype == MOE_W_NVFP4, MOE_ERR_INVALID_ARG,
          "shape->wdtype must be MOE_W_NVFP4");
  const Nvfp4Scales nv{w13_sb, w13_sg, w2_sb, w2_sg};
  return forward_impl(shape, x, norm_w, router_w, router_logits, router_bias, nullptr, nullptr, w13,
                      w2, nullptr, nullptr, out, topk_ids_out, topk_w_out, workspace,
                      workspace_bytes, stream, &nv);
}

moe_status moe_quantize_nvfp4(const void* w, int32_t M, int32_t N, int32_t K, uint8_t* q,
                              uint8_t* sb, float* sg, moe_stream_t stream) {
  MOE_REQ(w && q && sb && sg, MOE_ERR_INVALID_ARG, "w, q, sb and sg must be non-NULL");
  MOE_REQ(M >= 0 && N >= 0 && K > 0 && K % 16 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
          "M=%d N=%d K=%d (K %% 16 == 0)", M, N, K);
  MOE_REQ(aligned16(w) && aligned16(q) && ((uintptr_t)sb & 3u) == 0 && ((uintptr_t)sg & 3u) == 0,
          MOE_ERR_INVALID_ARG, "misaligned pointer");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_quantize_nvfp4(w, M, N, K, q, sb, sg, (cudaStream_t)stream), "NVFP4 quantise");
  return MOE_OK;
}

moe_status moe_quantize_fp8_blocks(const void* x, int32_t N, int32_t K, int32_t block_rows,
                                   uint8_t* q, float* scale, moe_stream_t stream) {
  MOE_REQ(x && q && scale, MOE_ERR_INVALID_ARG, "x, q and scale must be non-NULL");
  MOE_REQ(block_rows == 1 || block_rows == 128, MOE_ERR_INVALID_ARG, "block_rows=%d (1 or 128)",
          block_rows);
  MOE_REQ(N >= 0 && K > 0 && K % 128 == 0 && N % block_rows == 0, MOE_ERR_UNSUPPORTED_SHAPE,
          "N=%d K=%d block_rows=%d (K %% 128 == 0, N %% block_rows == 0)", N, K, block_rows);
  MOE_REQ(aligned16(x) && aligned16(q) && ((uintptr_t)scale & 3u) == 0, MOE_ERR_INVALID_ARG,
          "misaligned pointer");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_quantize_fp8_blocks(x, N, K, block_rows, q, scale, (cudaStream_t)stream),
           "block-wise FP8 quantise");
  return MOE_OK;
}

moe_status moe_rmsnorm(const void* x, const void* w, int32_t T, int32_t H, float eps, void* y,
                       void* yq, float* yscale, moe_stream_t stream) {
  MOE_REQ(x && w && y, MOE_ERR_INVALID_ARG, "x, w and y must be non-NULL");
  MOE_REQ((yq == nullptr) == (yscale == nullptr), MOE_ERR_INVALID_ARG,
          "yq and yscale must both be given or both NULL");
  MOE_REQ(T >= 0 && H > 0 && H % 8 == 0, MOE_ERR_UNSUPPORTED_SHAPE, "T=%d H=%d (H %% 8 == 0)", T, H);
  MOE_REQ(aligned16(x) && aligned16(w) && aligned16(y) && (!yq || ((uintptr_t)yq & 7u) == 0),
          MOE_ERR_INVALID_ARG, "misaligned pointer");
  MOE_REQ(eps >= 0.f, MOE_ERR_INVALID_ARG, "eps < 0");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_rmsnorm(x, w, T, H, eps, y, yq, yscale, (cudaStream_t)stream), "rmsnorm launch");
  return MOE_OK;
}

size_t moe_route_workspace_size(int32_t T, int32_t H, int32_t E) {
  if (T < 0 || H <= 0 || H % 64 || E <= 0 || E > kMaxExperts) return 0;
  return router_ws_bytes(T, H, E);
}

moe_status moe_route_topk(const void* xhat, const float* router_w, const float* router_bias,
                          const float* logits_in, int32_t T, int32_t H, int32_t E, int32_t k,
                          int32_t* ids, float* weights, float* logits_out, void* workspace,
                          size_t workspace_bytes, moe_stream_t stream) {
  MOE_REQ(ids && weights, MOE_ERR_INVALID_ARG, "ids and weights must be non-NULL");
  MOE_REQ(T >= 0 && E > 0 && E <= kMaxExperts && k > 0 && k <= E && k <= kMaxTopK,
          MOE_ERR_UNSUPPORTED_SHAPE, "T=%d E=%d k=%d (E <= 256, k <= min(E, 8))", T, E, k);
  if (logits_in == nullptr) {
    MOE_REQ(xhat && router_w && workspace, MOE_ERR_INVALID_ARG,
            "xhat, router_w and workspace are needed when logits_in is NULL");
    MOE_REQ(H > 0 && H % 64 == 0, MOE_ERR_UNSUPPORTED_SHAPE, "H=%d must be a multiple of 64", H);
    MOE_REQ(aligned16(xhat), MOE_ERR_INVALID_ARG, "xhat must be 16-byte aligned");
    MOE_REQ(workspace_bytes >= moe_route_workspace_size(T, H, E), MOE_ERR_WORKSPACE_TOO_SMALL,
            "workspace %zu < %zu bytes", workspace_bytes, moe_route_workspace_size(T, H, E));
  }
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (!logits_in)
    MOE_REQ(((uintptr_t)workspace & 255u) == 0, MOE_ERR_INVALID_ARG,
            "workspace must be 256-byte aligned");
  return route_topk_impl(xhat, router_w, logits_in, router_bias, T, H, E, k, ids, weights,
                         logits_out, workspace, d, st);
}

size_t moe_permute_workspace_size(int32_t T, int32_t E, int32_t k) {
  if (T < 0 || E <= 0 || E > kMaxExperts || k <= 0 || k > kMaxTopK) return 0;
  return moe::permute_workspace_bytes(T, E, k);
}

moe_status moe_permute(const int32_t* ids, int32_t T, int32_t E, int32_t k, int32_t* offsets,
                       int32_t* row_src, int32_t* row_of_pair, const void* xhat, void* xp,
                       int32_t row_bytes, const float* xscale, float* xp_scale, void* workspace,
                       size_t workspace_bytes, moe_stream_t stream) {
  MOE_REQ(ids && offsets && row_src && row_of_pair, MOE_ERR_INVALID_ARG,
          "ids, offsets, row_src and row_of_pair must be non-NULL");
  MOE_REQ(T >= 0 && E > 0 && E <= kMaxExperts && k > 0 && k <= kMaxTopK,
          MOE_ERR_UNSUPPORTED_SHAPE, "T=%d E=%d k=%d", T, E, k);
  MOE_REQ((xhat == nullptr) == (xp == nullptr), MOE_ERR_INVALID_ARG, "give both xhat and xp or neither");
  MOE_REQ((xscale == nullptr) == (xp_scale == nullptr), MOE_ERR_INVALID_ARG,
          "give both xscale and xp_scale or neither");
  MOE_REQ(!xp_scale || xp, MOE_ERR_INVALID_ARG, "a scale gather needs the row gather");
  if (xp) {
    MOE_REQ(row_bytes > 0 && row_bytes % 16 == 0 && aligned16(xhat) && aligned16(xp),
            MOE_ERR_INVALID_ARG, "row_bytes=%d must be a positive multiple of 16, pointers aligned",
            row_bytes);
  }
  const size_t need = moe::permute_workspace_bytes(T, E, k);
  MOE_REQ(workspace_bytes >= need && (need == 0 || workspace != nullptr),
          MOE_ERR_WORKSPACE_TOO_SMALL, "permute workspace %zu < %zu bytes", workspace_bytes, need);
  MOE_REQ(need == 0 || ((uintptr_t)workspace & 15u) == 0, MOE_ERR_INVALID_ARG,
          "workspace must be 16-byte aligned");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  MOE_CUDA(moe::launch_permute_any(ids, T, E, k, offsets, row_src, row_of_pair, (int32_t*)workspace,
                                   d->status, st),
           "permute launch");
  if (xp)
    MOE_CUDA(moe::launch_gather_rows(offsets, E, row_src, k, T * k, xhat, xp, row_bytes, xscale,
                                     xp_scale, st),
             "gather launch");
  return MOE_OK;
}

moe_status moe_grouped_gemm(const moe_shape* shape, int32_t mode, const void* a,
                            const float* a_scale, const void* w, const float* w_scale,
                            const int32_t* offsets, const int32_t* row_src, const float* topk_w,
                            void* c, moe_stream_t stream) {
  moe_status rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  MOE_REQ(mode >= MOE_GEMM_FC1_RAW && mode <= MOE_GEMM_FC2_BF16, MOE_ERR_INVALID_ARG, "mode=%d", mode);
  MOE_REQ(shape->wdtype != MOE_W_NVFP4, MOE_ERR_INVALID_ARG,
          "NVFP4 weights run through moe_ffn_forward_nvfp4");
  MOE_REQ(shape->wdtype != MOE_W_FP8_BLOCK, MOE_ERR_INVALID_ARG,
          "block-wise FP8 weights run through moe_grouped_ffn or the forward");
  MOE_REQ(a && w && offsets && c, MOE_ERR_INVALID_ARG, "a, w, offsets and c must be non-NULL");
  MOE_REQ(aligned16(a) && aligned16(w) && aligned16(c), MOE_ERR_INVALID_ARG, "misaligned pointer");
  const bool f8 = shape->wdtype == MOE_W_FP8_E4M3;
  MOE_REQ(!f8 || (a_scale && w_scale), MOE_ERR_INVALID_ARG, "FP8 needs a_scale and w_scale");
  MOE_REQ(!f8 || aligned16(w_scale), MOE_ERR_INVALID_ARG, "FP8 weight scales must be 16-byte aligned");
  MOE_REQ(!(topk_w && !row_src), MOE_ERR_INVALID_ARG, "topk_w needs row_src");
  DevInfo* d = nullptr;
  if ((rc = device_info(&d)) != MOE_OK) return rc;
  const int R_max = shape->T * shape->top_k;
  return run_gemm(shape, mode, pick_engine(shape), a, a_scale, w, w_scale, offsets, row_src,
                  mode >= MOE_GEMM_FC2 ? topk_w : nullptr, c, R_max, d->sms, d->status,
                  (cudaStream_t)stream);
}

size_t moe_grouped_ffn_workspace_size(const moe_shape* shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  const size_t R = (size_t)shape->T * shape->top_k;
  size_t n = up256((size_t)(2 * shape->E + 1) * 4);
  if (shape->wdtype == MOE_W_FP8_E4M3) n += up256(R * shape->I) + up256(R * 4);
  if (shape->wdtype == MOE_W_FP8_BLOCK)  // group scales of act, and its bf16 values
    n += up256(R * (shape->I / 128) * 4) + up256(R * shape->I * 2);
  return n;
}

moe_status moe_grouped_ffn(const moe_shape* shape, const void* xp, const float* xp_scale,
                           const void* w13, const float* w13_scale, const void* w2,
                           const float* w2_scale, const int32_t* offsets, const int32_t* row_src,
                           const float* topk_w, void* act, void* y, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream) {
  moe_status rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  const bool fb = shape->wdtype == MOE_W_FP8_BLOCK;
  const bool f8 = shape->wdtype == MOE_W_FP8_E4M3 || fb;
  MOE_REQ(shape->wdtype != MOE_W_NVFP4, MOE_ERR_INVALID_ARG,
          "NVFP4 weights run through moe_ffn_forward_nvfp4");
  MOE_REQ(xp && w13 && w2 && offsets && row_src && topk_w && act && y && workspace,
          MOE_ERR_INVALID_ARG, "xp, w13, w2, offsets, row_src, topk_w, act, y and workspace must be non-NULL");
  MOE_REQ(!f8 || (xp_scale && w13_scale && w2_scale), MOE_ERR_INVALID_ARG,
          "FP8 needs xp_scale, w13_scale and w2_scale");
  MOE_REQ(!f8 || (aligned16(w13_scale) && aligned16(w2_scale)), MOE_ERR_INVALID_ARG,
          "FP8 weight scales must be 16-byte aligned");
  MOE_REQ(aligned16(xp) && aligned16(w13) && aligned16(w2) && aligned16(act) && aligned16(y),
          MOE_ERR_INVALID_ARG, "misaligned pointer");
  MOE_REQ(((uintptr_t)workspace & 255u) == 0, MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = moe_grouped_ffn_workspace_size(shape);
  MOE_REQ(workspace_bytes >= need, MOE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes",
          workspace_bytes, need);
  DevInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t R = (size_t)shape->T * shape->top_k;
  const size_t sched_bytes = (size_t)(2 * shape->E + 1) * 4;
  int32_t* sched = at<int32_t>(workspace, 0);
  uint8_t* actq = f8 ? at<uint8_t>(workspace, up256(sched_bytes)) : nullptr;
  float* act_scale = f8 ? at<float>(workspace, up256(sched_bytes) + up256(R * shape->I)) : nullptr;
  void* act_mid = act;
  if (fb) {
    // the E4M3 intermediate goes to the caller's act; its group scales and
    // (prefill engine) its bf16 values to the workspace
    actq = static_cast<uint8_t*>(act);
    act_scale = at<float>(workspace, up256(sched_bytes));
    act_mid = at<void>(workspace, up256(sched_bytes) + up256(R * (shape->I / 128) * 4));
    MOE_CUDA(cudaMemsetAsync(sched, 0, sched_bytes, st), "scheduler reset");
  }
  const int engine = pick_engine(shape);
  PdlOff no_pdl(engine == MOE_ENGINE_PREFILL);  // as in the forward
  const bool fuse = fuse_decode(shape, engine);
  // the fused decode launch and the token tiles' unit counters start at zero
  if (!fb && (fuse || engine == MOE_ENGINE_PREFILL))
    MOE_CUDA(cudaMemsetAsync(sched, 0, sched_bytes, st), "scheduler reset");
  return ffn_impl(shape, engine, fuse, xp, xp_scale, w13, w13_scale, w2, w2_scale, offsets,
                  row_src, topk_w, act_mid, y, sched, actq, act_scale, dev, st);
}

moe_status moe_grouped_ffn_nvfp4(const moe_shape* shape, const void* xp, const uint8_t* w13,
                                 const uint8_t* w13_sb, const float* w13_sg, const uint8_t* w2,
                                 const uint8_t* w2_sb, const float* w2_sg, const int32_t* offsets,
                                 const int32_t* row_src, const float* topk_w, void* act, void* y,
                                 void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  moe_status rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  MOE_REQ(shape->wdtype == MOE_W_NVFP4, MOE_ERR_INVALID_ARG, "shape->wdtype must be MOE_W_NVFP4");
  MOE_REQ(xp && w13 && w13_sb && w13_sg && w2 && w2_sb && w2_sg && offsets && row_src && topk_w &&
              act && y && workspace,
          MOE_ERR_INVALID_ARG, "every pointer must be non-NULL");
  MOE_REQ(aligned16(xp) && aligned16(w13) && aligned16(w2) && aligned16(act) && aligned16(y) &&
              aligned16(w13_sb) && aligned16(w2_sb),
          MOE_ERR_INVALID_ARG, "misaligned pointer");
  MOE_REQ(((uintptr_t)workspace & 255u) == 0, MOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = moe_grouped_ffn_workspace_size(shape);
  MOE_REQ(workspace_bytes >= need, MOE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes",
          workspace_bytes, need);
  DevInfo* dev = nullptr;
  if ((rc = device_info(&dev)) != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* sched = at<int32_t>(workspace, 0);
  const int R = shape->T * shape->top_k;
  MOE_CUDA(cudaMemsetAsync(sched, 0, (size_t)(2 * shape->E + 1) * 4, st), "scheduler reset");
  MOE_CUDA(moe::launch_decode_ffn_nvfp4(xp, w13, w13_sb, w13_sg, w2, w2_sb, w2_sg, act, y, offsets,
                                        row_src, topk_w, sched, shape->E, shape->H, shape->I, R,
                                        shape->T, dev->sms, dev->status, st),
           "NVFP4 FFN launch");
  return MOE_OK;
}

moe_status moe_silu_and_mul(const void* h, int32_t R, int32_t I, void* a, moe_stream_t stream) {
  MOE_REQ(h && a, MOE_ERR_INVALID_ARG, "h and a must be non-NULL");
  MOE_REQ(R >= 0 && I > 0 && I % 8 == 0, MOE_ERR_UNSUPPORTED_SHAPE, "R=%d I=%d (I %% 8 == 0)", R, I);
  MOE_REQ(aligned16(h) && aligned16(a), MOE_ERR_INVALID_ARG, "misaligned pointer");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_silu_and_mul(h, R, I, a, (cudaStream_t)stream), "silu_and_mul launch");
  return MOE_OK;
}

moe_status moe_combine(const void* y, int32_t y_bf16, int32_t y_pair_order,
                       const int32_t* row_of_pair, int32_t T, int32_t k, int32_t H, void* out,
                       moe_stream_t stream) {
  MOE_REQ(y && row_of_pair && out, MOE_ERR_INVALID_ARG, "y, row_of_pair and out must be non-NULL");
  MOE_REQ(T >= 0 && k > 0 && k <= kMaxTopK && H > 0 && H % 8 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
          "T=%d k=%d H=%d (H %% 8 == 0)", T, k, H);
  MOE_REQ(aligned16(y) && aligned16(out), MOE_ERR_INVALID_ARG, "misaligned pointer");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_combine(y, y_bf16 != 0, y_pair_order != 0, row_of_pair, T, k, H, out,
                               (cudaStream_t)stream),
           "combine launch");
  return MOE_OK;
}

moe_status moe_quantize_fp8_rows(const void* x, int64_t rows, int32_t cols, void* q, float* scale,
                                 moe_stream_t stream) {
  MOE_REQ(x && q && scale, MOE_ERR_INVALID_ARG, "x, q and scale must be non-NULL");
  MOE_REQ(rows >= 0 && cols > 0 && cols % 16 == 0, MOE_ERR_UNSUPPORTED_SHAPE,
          "rows=%lld cols=%d (cols %% 16 == 0)", (long long)rows, cols);
  MOE_REQ(aligned16(x) && aligned16(q), MOE_ERR_INVALID_ARG, "misaligned pointer");
  DevInfo* d = nullptr;
  moe_status rc = device_info(&d);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(moe::launch_quant_rows(x, rows, cols, q, scale, nullptr, (cudaStream_t)stream),
           "quantise launch");
  return MOE_OK;
}

}  // extern "C"
