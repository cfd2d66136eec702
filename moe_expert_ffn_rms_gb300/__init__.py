"""Python binding of libmoeffn.so -- the MoE expert FFN forward on a GB300.

Argument marshalling only: every step runs in the library's CUDA kernels.
Functions take torch tensors (device memory) and enqueue work on the current
torch CUDA stream unless a stream is given.  They have the same names as the
C entry points in include/moe_ffn.h.

Importing the package loads the library; if it has not been built
(``python -m moe_expert_ffn_rms_gb300.build`` or ``__graft_entry__.build()``)
the import fails with an ImportError -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeffn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run moe_expert_ffn_rms_gb300.build.build()")

lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
                3: "MOE_ERR_UNSUPPORTED_DEVICE", 4: "MOE_ERR_WORKSPACE_TOO_SMALL",
                5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT"}
W_BF16, W_FP8_E4M3, W_NVFP4, W_FP8_BLOCK = 0, 1, 2, 3
GEMM_FC1_RAW, GEMM_FC1_SILU, GEMM_FC2, GEMM_FC2_BF16 = 0, 1, 2, 3
ENGINE_AUTO, ENGINE_DECODE, ENGINE_PREFILL = 0, 1, 2


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("I", ctypes.c_int32), ("top_k", ctypes.c_int32), ("eps", ctypes.c_float),
                ("wdtype", ctypes.c_int32), ("engine", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t

_SIGS = {
    "moe_abi_version": (_I32, []),
    "moe_launch_count": (ctypes.c_int64, []),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_check_device": (ctypes.c_int, []),
    "moe_device_status": (ctypes.c_int, [ctypes.POINTER(_I32), _I32]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int64, _P]),
    "moe_ffn_workspace_size": (_SZ, [ctypes.POINTER(MoeShape)]),
    "moe_ffn_forward": (ctypes.c_int, [ctypes.POINTER(MoeShape), _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _P, _SZ, _P]),
    "moe_ffn_forward_routed": (ctypes.c_int, [ctypes.POINTER(MoeShape), _P, _P, _P, _P, _P, _P, _P,
                                              _P, _P, _P, _SZ, _P]),
    "moe_ffn_forward_static_ws": (ctypes.c_int, [ctypes.POINTER(MoeShape), _P, _P, _P, _P, _P, _P,
                                                 _P, _P, _P, _P, _P, _P, _P]),
    "moe_rmsnorm": (ctypes.c_int, [_P, _P, _I32, _I32, ctypes.c_float, _P, _P, _P, _P]),
    "moe_route_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "moe_route_topk": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ,
                                      _P]),
    "moe_permute_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "moe_permute": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ,
                                   _P]),
    "moe_grouped_gemm": (ctypes.c_int, [ctypes.POINTER(MoeShape), _I32, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P]),
    "moe_grouped_ffn_workspace_size": (_SZ, [ctypes.POINTER(MoeShape)]),
    "moe_grouped_ffn": (ctypes.c_int, [ctypes.POINTER(MoeShape), _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _SZ, _P]),
    "moe_silu_and_mul": (ctypes.c_int, [_P, _I32, _I32, _P, _P]),
    "moe_combine": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _I32, _I32, _P, _P]),
    "moe_quantize_fp8_rows": (ctypes.c_int, [_P, ctypes.c_int64, _I32, _P, _P, _P]),
    "moe_ffn_forward_nvfp4": (ctypes.c_int, [ctypes.POINTER(MoeShape), _P, _P, _P, _P, _P, _P, _P, _P,
                                             _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_quantize_nvfp4": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P, _P]),
    "moe_grouped_ffn_nvfp4": (ctypes.c_int, [ctypes.POINTER(MoeShape), _P, _P, _P, _P, _P, _P, _P, _P,
                                             _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_quantize_fp8_blocks": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def last_error() -> str:
    return lib.moe_last_error().decode()


def _check(rc: int):
    if rc != MOE_OK:
        raise MoeError(rc, last_error() or STATUS_NAMES.get(rc, str(rc)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_shape(T, H, E, I, top_k, eps=1e-6, fp8=False, engine=ENGINE_AUTO, nvfp4=False) -> MoeShape:
    """fp8: False (bf16), True (per-channel E4M3) or "block" (block-wise E4M3)."""
    wd = W_NVFP4 if nvfp4 else (W_FP8_BLOCK if fp8 == "block" else (W_FP8_E4M3 if fp8 else W_BF16))
    return MoeShape(T, H, E, I, top_k, eps, wd, engine)


def abi_version() -> int:
    return lib.moe_abi_version()


def check_device():
    _check(lib.moe_check_device())


def device_status(clear: bool = True) -> int:
    v = _I32(0)
    _check(lib.moe_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


def moe_selftest_wait_timeout(limit_cycles: int, stream=None):
    _check(lib.moe_selftest_wait_timeout(limit_cycles, _stream(stream)))


def moe_ffn_workspace_size(shape: MoeShape) -> int:
    n = lib.moe_ffn_workspace_size(ctypes.byref(shape))
    if n == 0:
        raise MoeError(1, last_error())
    return n


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Device workspace (torch owns the memory; 256-byte aligned)."""
    return torch.empty(nbytes + 256, dtype=torch.uint8, device=device)


def _ws_ptr(ws: torch.Tensor) -> int:
    p = ws.data_ptr()
    return (p + 255) & ~255


def _ws_bytes(ws: torch.Tensor) -> int:
    return ws.numel() - (_ws_ptr(ws) - ws.data_ptr())


def moe_ffn_forward(shape: MoeShape, x, norm_w, w13, w2, out, workspace, router_w=None,
                    router_logits=None, router_bias=None, w13_scale=None, w2_scale=None,
                    topk_ids_out=None, topk_w_out=None, stream=None):
    _check(lib.moe_ffn_forward(ctypes.byref(shape), _ptr(x), _ptr(norm_w), _ptr(router_w),
                               _ptr(router_logits), _ptr(router_bias), _ptr(w13), _ptr(w2),
                               _ptr(w13_scale), _ptr(w2_scale), _ptr(out), _ptr(topk_ids_out),
                               _ptr(topk_w_out), _ws_ptr(workspace), _ws_bytes(workspace),
                               _stream(stream)))
    return out


def moe_ffn_forward_static_ws(shape: MoeShape, x, norm_w, w13, w2, out, router_w=None,
                              router_logits=None, router_bias=None, w13_scale=None,
                              w2_scale=None, topk_ids_out=None, topk_w_out=None, stream=None):
    """moe_ffn_forward with the library's fixed 32 MiB device scratch instead
    of a caller workspace (for callers that cannot allocate device memory)."""
    _check(lib.moe_ffn_forward_static_ws(ctypes.byref(shape), _ptr(x), _ptr(norm_w), _ptr(router_w),
                                         _ptr(router_logits), _ptr(router_bias), _ptr(w13),
                                         _ptr(w2), _ptr(w13_scale), _ptr(w2_scale), _ptr(out),
                                         _ptr(topk_ids_out), _ptr(topk_w_out), _stream(stream)))
    return out


def moe_ffn_forward_routed(shape: MoeShape, x, norm_w, topk_ids, topk_w, w13, w2, out, workspace,
                           w13_scale=None, w2_scale=None, stream=None):
    _check(lib.moe_ffn_forward_routed(ctypes.byref(shape), _ptr(x), _ptr(norm_w), _ptr(topk_ids),
                                      _ptr(topk_w), _ptr(w13), _ptr(w2), _ptr(w13_scale),
                                      _ptr(w2_scale), _ptr(out), _ws_ptr(workspace),
                                      _ws_bytes(workspace), _stream(stream)))
    return out


def moe_rmsnorm(x, w, eps, y, yq=None, yscale=None, stream=None):
    T, H = x.shape
    _check(lib.moe_rmsnorm(_ptr(x), _ptr(w), T, H, eps, _ptr(y), _ptr(yq), _ptr(yscale),
                           _stream(stream)))
    return y


def moe_route_workspace_size(T, H, E) -> int:
    return lib.moe_route_workspace_size(T, H, E)


def moe_route_topk(T, H, E, k, ids, weights, xhat=None, router_w=None, router_bias=None,
                   logits_in=None, logits_out=None, workspace=None, stream=None):
    wsp = _ws_ptr(workspace) if workspace is not None else None
    wsb = _ws_bytes(workspace) if workspace is not None else 0
    _check(lib.moe_route_topk(_ptr(xhat), _ptr(router_w), _ptr(router_bias), _ptr(logits_in), T, H,
                              E, k, _ptr(ids), _ptr(weights), _ptr(logits_out), wsp, wsb,
                              _stream(stream)))


def moe_permute_workspace_size(T, E, k) -> int:
    return lib.moe_permute_workspace_size(T, E, k)


def moe_permute(ids, T, E, k, offsets, row_src, row_of_pair, xhat=None, xp=None, row_bytes=0,
                xscale=None, xp_scale=None, workspace=None, stream=None):
    wsp = _ws_ptr(workspace) if workspace is not None else None
    wsb = _ws_bytes(workspace) if workspace is not None else 0
    _check(lib.moe_permute(_ptr(ids), T, E, k, _ptr(offsets), _ptr(row_src), _ptr(row_of_pair),
                           _ptr(xhat), _ptr(xp), row_bytes, _ptr(xscale), _ptr(xp_scale), wsp,
                           wsb, _stream(stream)))


def moe_grouped_gemm(shape: MoeShape, mode, a, w, offsets, c, a_scale=None, w_scale=None,
                     row_src=None, topk_w=None, stream=None):
    _check(lib.moe_grouped_gemm(ctypes.byref(shape), mode, _ptr(a), _ptr(a_scale), _ptr(w),
                                _ptr(w_scale), _ptr(offsets), _ptr(row_src), _ptr(topk_w), _ptr(c),
                                _stream(stream)))
    return c


def moe_grouped_ffn_workspace_size(shape: MoeShape) -> int:
    return lib.moe_grouped_ffn_workspace_size(ctypes.byref(shape))


def moe_grouped_ffn(shape: MoeShape, xp, w13, w2, offsets, row_src, topk_w, act, y, workspace,
                    xp_scale=None, w13_scale=None, w2_scale=None, stream=None):
    _check(lib.moe_grouped_ffn(ctypes.byref(shape), _ptr(xp), _ptr(xp_scale), _ptr(w13),
                               _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(offsets),
                               _ptr(row_src), _ptr(topk_w), _ptr(act), _ptr(y), _ws_ptr(workspace),
                               _ws_bytes(workspace), _stream(stream)))
    return y


def moe_silu_and_mul(h, a, stream=None):
    R, I2 = h.shape
    _check(lib.moe_silu_and_mul(_ptr(h), R, I2 // 2, _ptr(a), _stream(stream)))
    return a


def moe_combine(y, row_of_pair, T, k, out, pair_order=False, stream=None):
    H = y.shape[1]
    y_bf16 = 1 if y.dtype == torch.bfloat16 else 0
    _check(lib.moe_combine(_ptr(y), y_bf16, 1 if pair_order else 0, _ptr(row_of_pair), T, k, H,
                           _ptr(out), _stream(stream)))
    return out


def moe_ffn_forward_nvfp4(shape: MoeShape, x, norm_w, w13, w13_sb, w13_sg, w2, w2_sb, w2_sg, out,
                          workspace, router_w=None, router_logits=None, router_bias=None,
                          topk_ids_out=None, topk_w_out=None, stream=None):
    """The forward with NVFP4 expert weights (codes, E4M3 block scales, fp32
    matrix scales from moe_quantize_nvfp4) and bf16 activations."""
    _check(lib.moe_ffn_forward_nvfp4(ctypes.byref(shape), _ptr(x), _ptr(norm_w), _ptr(router_w),
                                     _ptr(router_logits), _ptr(router_bias), _ptr(w13), _ptr(w13_sb),
                                     _ptr(w13_sg), _ptr(w2), _ptr(w2_sb), _ptr(w2_sg), _ptr(out),
                                     _ptr(topk_ids_out), _ptr(topk_w_out), _ws_ptr(workspace),
                                     _ws_bytes(workspace), _stream(stream)))
    return out


def moe_grouped_ffn_nvfp4(shape: MoeShape, xp, w13, w13_sb, w13_sg, w2, w2_sb, w2_sg, offsets,
                          row_src, topk_w, act, y, workspace, stream=None):
    """The NVFP4 FFN step: xp fp16 [R, H] -> act fp16 [R, I] -> y bf16 [R, H]."""
    _check(lib.moe_grouped_ffn_nvfp4(ctypes.byref(shape), _ptr(xp), _ptr(w13), _ptr(w13_sb),
                                     _ptr(w13_sg), _ptr(w2), _ptr(w2_sb), _ptr(w2_sg), _ptr(offsets),
                                     _ptr(row_src), _ptr(topk_w), _ptr(act), _ptr(y),
                                     _ws_ptr(workspace), _ws_bytes(workspace), _stream(stream)))


def moe_quantize_nvfp4(w, q, sb, sg, stream=None):
    """NVFP4 quantisation of w bf16 [M, N, K] (or [N, K]) into q uint8
    [.., N, K/2], sb uint8 [.., N, K/16], sg fp32 [M]."""
    K = w.shape[-1]
    N = w.shape[-2]
    M = w.numel() // (N * K) if w.numel() else 0
    _check(lib.moe_quantize_nvfp4(_ptr(w), M, N, K, _ptr(q), _ptr(sb), _ptr(sg), _stream(stream)))


def moe_quantize_fp8_rows(x, q, scale, stream=None):
    cols = x.shape[-1]
    rows = x.numel() // cols
    _check(lib.moe_quantize_fp8_rows(_ptr(x), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))
    return q, scale


def moe_quantize_fp8_blocks(x, q, scale, block_rows, stream=None):
    """Block-wise E4M3 quantisation of x bf16 [..., K] viewed as [N, K]:
    q uint8 [N, K], scale fp32 [N / block_rows, K / 128] (block_rows 1 or 128)."""
    K = x.shape[-1]
    N = x.numel() // K if x.numel() else 0
    _check(lib.moe_quantize_fp8_blocks(_ptr(x), N, K, block_rows, _ptr(q), _ptr(scale),
                                       _stream(stream)))
    return q, scale
