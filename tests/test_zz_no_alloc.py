"""The allocation-free forward (moe_ffn_forward_static_ws) against the
workspace forward.

Callers that cannot allocate device memory (a plug-in whose host owns the
memory budget, a latency-critical path, plain C / FFI code holding only its
input and output buffers) use moe_ffn_forward_static_ws, which keeps its
scratch in a fixed 32 MiB device array inside the library.  This file runs
last so that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests.parity_util import TOL_BF16, assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_ffn_rms_gb300 as M
    M.check_device()
    return M


def _call_static(M, shape, inp, out, ids, tw):
    p = lambda t: None if t is None else t.data_ptr()
    return M.lib.moe_ffn_forward_static_ws(
        ctypes.byref(shape), p(inp["x"]), p(inp["norm_w"]), p(inp["router_w"]),
        p(inp["router_logits"]), p(inp["router_bias"]), p(inp["w13"]), p(inp["w2"]), None, None,
        p(out), p(ids), p(tw), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cfg", ["c1_tiny", "c2_decode_balanced", "c3_small"])
def test_static_scratch_forward_matches_workspace_forward(M, cfg):
    if cfg == "c3_small":
        inp = workloads.make_inputs("c3_decode_skewed", "cuda",
                                    shape=workloads.Shape(T=64, H=1024, E=256, k=8, I=512))
    else:
        inp = workloads.make_inputs(cfg, "cuda")
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    shape = M.make_shape(T, H, E, I, k, inp["eps"])
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), "cuda")
    ref = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ref_ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ref_tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    M.moe_ffn_forward(shape, inp["x"], inp["norm_w"], inp["w13"], inp["w2"], ref, ws,
                      router_w=inp["router_w"], router_logits=inp["router_logits"],
                      router_bias=inp["router_bias"], topk_ids_out=ref_ids, topk_w_out=ref_tw)
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row share (and reuse) the static scratch
        out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        tw = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        rc = _call_static(M, shape, inp, out, ids, tw)
        assert rc == 0, M.last_error()
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids), f"call {call}: routing differs"
        np.testing.assert_allclose(f64(tw), f64(ref_tw), rtol=1e-6, atol=0)
        assert_close(f64(out), f64(ref), TOL_BF16, f"static scratch call {call}")
    assert M.device_status() == 0


def test_static_scratch_rejects_shapes_beyond_its_size(M):
    shape = M.make_shape(4096, 4096, 64, 1536, 8)   # prefill batch: ~1 GB of scratch
    assert M.moe_ffn_workspace_size(shape) > (32 << 20)
    fake = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    rc = M.lib.moe_ffn_forward_static_ws(ctypes.byref(shape), fake.data_ptr(), fake.data_ptr(),
                                         fake.data_ptr(), None, None, fake.data_ptr(),
                                         fake.data_ptr(), None, None, fake.data_ptr(), None, None,
                                         None)
    assert rc == 4                                   # MOE_ERR_WORKSPACE_TOO_SMALL
    assert "static scratch" in M.last_error()
