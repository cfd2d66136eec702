"""The allocation-free forward (moe_ffn_forward_static_ws) against the
workspace forward and against the oracle.

Callers that cannot allocate device memory (a plug-in whose host owns the
memory budget, a latency-critical path, plain C / FFI code holding only its
input and output buffers) use moe_ffn_forward_static_ws, which keeps its
scratch in a fixed 32 MiB device array inside the library.  The skewed decode
shape (T=64, H=7168, E=256, top_k=8, I=2048) is the largest here that must
fit, at about 26 of the 32 MiB, and runs at full size.  This file runs last so
that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import workloads
from tests.parity_util import (TOL_BF16, TOL_FP8, assert_close, check_routing_e2e, f64,
                               forward_xhat)

pytestmark = pytest.mark.gpu
STATIC_BYTES = 32 << 20


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_ffn_rms_gb300 as M
    M.check_device()
    return M


def _call_static(M, shape, inp, w13, w2, s13, s2, out, ids, tw):
    p = lambda t: None if t is None else t.data_ptr()
    return M.lib.moe_ffn_forward_static_ws(
        ctypes.byref(shape), p(inp["x"]), p(inp["norm_w"]), p(inp["router_w"]),
        p(inp["router_logits"]), p(inp["router_bias"]), p(w13), p(w2), p(s13), p(s2),
        p(out), p(ids), p(tw), torch.cuda.current_stream().cuda_stream)


def _fp8_weights(M, inp):
    E, H, I = inp["E"], inp["H"], inp["I"]
    q13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device="cuda")
    s13 = torch.empty((E, 2 * I), dtype=torch.float32, device="cuda")
    q2 = torch.empty((E, H, I), dtype=torch.uint8, device="cuda")
    s2 = torch.empty((E, H), dtype=torch.float32, device="cuda")
    M.moe_quantize_fp8_rows(inp["w13"], q13, s13)
    M.moe_quantize_fp8_rows(inp["w2"], q2, s2)
    return q13, s13, q2, s2


@pytest.mark.parametrize("cfg,sample", [("c1_tiny", None), ("c2_decode_balanced", None),
                                        ("c3_decode_skewed", 8), ("c4_decode_fp8", None)])
def test_static_scratch_forward_matches_workspace_forward_and_oracle(M, cfg, sample):
    inp = workloads.make_inputs(cfg, "cuda")
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    fp8 = bool(inp["fp8"])
    shape = M.make_shape(T, H, E, I, k, inp["eps"], fp8=fp8)
    need = M.moe_ffn_workspace_size(shape)
    assert need <= STATIC_BYTES
    if cfg == "c3_decode_skewed":
        assert need > (20 << 20)        # the size bound is exercised, not only asserted
    if fp8:
        w13, s13, w2, s2 = _fp8_weights(M, inp)
    else:
        w13, s13, w2, s2 = inp["w13"], None, inp["w2"], None
    ws = M.alloc_workspace(need, "cuda")
    ref = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ref_ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ref_tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    M.moe_ffn_forward(shape, inp["x"], inp["norm_w"], w13, w2, ref, ws,
                      router_w=inp["router_w"], router_logits=inp["router_logits"],
                      router_bias=inp["router_bias"], w13_scale=s13, w2_scale=s2,
                      topk_ids_out=ref_ids, topk_w_out=ref_tw)
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row share (and reuse) the static scratch
        out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        tw = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        rc = _call_static(M, shape, inp, w13, w2, s13, s2, out, ids, tw)
        assert rc == 0, M.last_error()
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the same bits as the workspace forward
        assert torch.equal(ids, ref_ids), f"call {call}: routing differs"
        assert torch.equal(tw, ref_tw), f"call {call}: routing weights differ"
        assert torch.equal(out, ref), f"call {call}: outputs differ"
    assert M.device_status() == 0
    # and against the oracle: routing bit-exact outside the tie bands, outputs
    # within the stated tolerance (on every token, or a sample at the skewed shape)
    xg = f64(forward_xhat(M, ws, T, H))
    ids_use, w_use, xhat, _ = check_routing_e2e(
        ids.cpu().numpy(), tw.cpu().double().numpy(), f64(inp["x"]), f64(inp["norm_w"]),
        inp["eps"], k, xhat_gpu=xg,
        router_w=None if inp["router_w"] is None else f64(inp["router_w"]),
        router_bias=None if inp["router_bias"] is None else f64(inp["router_bias"]),
        logits=None if inp["router_logits"] is None else f64(inp["router_logits"]))
    toks = np.arange(T)
    if sample is not None:
        toks = np.sort(np.random.default_rng(1).choice(T, size=sample, replace=False))
    if fp8:
        q13 = {int(e): O.quantize_rows_e4m3(f64(inp["w13"][e])) for e in np.unique(ids_use[toks])}
        q2 = {int(e): O.quantize_rows_e4m3(f64(inp["w2"][e])) for e in np.unique(ids_use[toks])}
        oref = O.ffn_token_outputs(xhat[toks], ids_use[toks], w_use[toks], None, None, I, fp8=True,
                                   wq13_of=q13.get, wq2_of=q2.get)
    else:
        oref = O.ffn_token_outputs(xhat[toks], ids_use[toks], w_use[toks],
                                   lambda e: f64(inp["w13"][e]), lambda e: f64(inp["w2"][e]), I)
    assert_close(f64(out)[toks], oref, TOL_FP8 if fp8 else TOL_BF16, f"static scratch {cfg}")
    del inp, ws
    torch.cuda.empty_cache()


def test_static_scratch_rejects_shapes_beyond_its_size(M):
    shape = M.make_shape(4096, 4096, 64, 1536, 8)   # prefill batch: ~1 GB of scratch
    assert M.moe_ffn_workspace_size(shape) > STATIC_BYTES
    fake = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    rc = M.lib.moe_ffn_forward_static_ws(ctypes.byref(shape), fake.data_ptr(), fake.data_ptr(),
                                         fake.data_ptr(), None, None, fake.data_ptr(),
                                         fake.data_ptr(), None, None, fake.data_ptr(), None, None,
                                         None)
    assert rc == 4                                   # MOE_ERR_WORKSPACE_TOO_SMALL
    assert "static scratch" in M.last_error()
