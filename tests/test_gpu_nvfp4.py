"""NVFP4 expert weights (E2M1 codes, E4M3 block scales of 16, fp32 matrix
scales) on the GPU: the quantiser bit-exact against the oracle, and the
NVFP4 forward against the oracle's forward on the oracle-dequantised weights
(the GEMMs of the NVFP4 path are those of the bf16 path on those weights)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads
from tests.parity_util import (TOL_BF16, assert_close, check_routing_e2e, f64, forward_xhat,
                               o1_weights)

pytestmark = pytest.mark.gpu
DEV = "cuda"
E2M1 = np.array([O.e2m1_decode(c) for c in range(16)])
E4M3 = np.array([O.e4m3_decode(c) for c in range(256)])


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_ffn_rms_gb300 as M
    return M


def quantize_gpu(M, w):
    E, N, K = w.shape
    q = torch.empty((E, N, K // 2), dtype=torch.uint8, device=DEV)
    sb = torch.empty((E, N, K // 16), dtype=torch.uint8, device=DEV)
    sg = torch.empty((E,), dtype=torch.float32, device=DEV)
    M.moe_quantize_nvfp4(w, q, sb, sg)
    return q, sb, sg


def codes_to_values(q):
    qn = q.cpu().numpy()
    return np.stack([E2M1[qn & 15], E2M1[qn >> 4]], axis=-1).reshape(*qn.shape[:-1], qn.shape[-1] * 2)


def test_quantize_nvfp4_bit_exact(M):
    g = torch.Generator(device=DEV).manual_seed(31)
    w = (torch.randn((4, 48, 512), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w[1, 5, 32:48] = 0          # an all-zero block
    w[2] = 0                    # an all-zero matrix
    w[0, 7, 100] = 0.9          # one large element: its block reaches 448 and code 6
    w[3, :, :16] *= 1e-4        # blocks far below the matrix maximum (small E4M3 scales)
    q, sb, sg = quantize_gpu(M, w)
    torch.cuda.synchronize()
    for e in range(4):
        qo, sbo, sgo = O.quantize_nvfp4(f64(w[e]))
        np.testing.assert_array_equal(codes_to_values(q[e]), qo)
        np.testing.assert_array_equal(E4M3[sb[e].cpu().numpy()], sbo)
        assert sg[e].item() == sgo
    assert sg[2].item() == 1.0 and int(q[2].max()) == 0 and int(sb[2].max()) == 0


def run_forward(M, inp, wq, ws=None):
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    shape = M.make_shape(T, H, E, I, k, inp["eps"], nvfp4=True)
    if ws is None:
        ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    (q13, sb13, sg13), (q2, sb2, sg2) = wq
    M.moe_ffn_forward_nvfp4(shape, inp["x"], inp["norm_w"], q13, sb13, sg13, q2, sb2, sg2, out, ws,
                            router_w=inp["router_w"], router_logits=inp["router_logits"],
                            router_bias=inp["router_bias"], topk_ids_out=ids, topk_w_out=tw)
    torch.cuda.synchronize()
    return out, ids, tw


def check_nvfp4(M, inp, sample=None, seed=0, name=""):
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    wq = (quantize_gpu(M, inp["w13"]), quantize_gpu(M, inp["w2"]))
    M.device_status(clear=True)
    shape = M.make_shape(T, H, E, I, k, inp["eps"], nvfp4=True)
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    out, ids, tw = run_forward(M, inp, wq, ws=ws)
    ids_g = ids.cpu().numpy()
    xg = f64(forward_xhat(M, ws, T, H))
    ids_use, w_use, xhat, _ = check_routing_e2e(
        ids_g, tw.cpu().double().numpy(), f64(inp["x"]), f64(inp["norm_w"]), inp["eps"], k,
        xhat_gpu=xg, router_w=None if inp["router_w"] is None else f64(inp["router_w"]),
        router_bias=None if inp["router_bias"] is None else f64(inp["router_bias"]),
        logits=None if inp["router_logits"] is None else f64(inp["router_logits"]), name=name)
    toks = np.arange(T)
    if sample is not None and sample < T:
        toks = np.sort(np.random.default_rng(seed).choice(T, size=sample, replace=False))

    def w13_of(e):
        return O.dequantize_nvfp4(*O.quantize_nvfp4(f64(inp["w13"][e])))

    def w2_of(e):
        return O.dequantize_nvfp4(*O.quantize_nvfp4(f64(inp["w2"][e])))
    ref = O.ffn_token_outputs(xhat[toks], ids_use[toks], w_use[toks], w13_of, w2_of, I)
    m = assert_close(f64(out)[toks], ref, TOL_BF16, inp["name"] + " nvfp4")
    assert M.device_status() == 0
    return out, m


SHAPES = {
    # name: (workload the distributions come from, shape, routing)
    "learned_small": ("c1_tiny", workloads.Shape(T=16, H=256, E=8, k=2, I=256), "learned"),
    "zipf": ("c3_decode_skewed", workloads.Shape(T=5, H=512, E=16, k=4, I=512), "zipf"),
    "balanced": ("c2_decode_balanced", workloads.Shape(T=16, H=256, E=64, k=8, I=256), "balanced"),
    "rows_64": ("c1_tiny", workloads.Shape(T=64, H=256, E=4, k=2, I=256), "learned"),
    "two_chunks": ("c1_tiny", workloads.Shape(T=300, H=256, E=2, k=1, I=512), "learned"),
    "single_token": ("c1_tiny", workloads.Shape(T=1, H=768, E=8, k=4, I=256), "learned"),
    "wide_hidden": ("c3_decode_skewed", workloads.Shape(T=8, H=7168, E=16, k=4, I=512), "zipf"),
    "max_experts": ("c3_decode_skewed", workloads.Shape(T=40, H=256, E=256, k=8, I=256), "zipf"),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_forward_nvfp4_small(M, name):
    cfg, shape, routing = SHAPES[name]
    for o1 in (False, True):
        inp = workloads.make_inputs(cfg, DEV, shape=shape, routing=routing, seed=13)
        inp["name"] = name + (" o1" if o1 else "")
        if o1:
            o1_weights(inp)
        check_nvfp4(M, inp)


def test_forward_nvfp4_full_decode_workload(M):
    """The decode NVFP4 workload (T=16, H=4096, E=64, k=8, I=1536), every
    token recomputed by the oracle; the run is deterministic."""
    inp = workloads.make_inputs("c6_decode_nvfp4", DEV)
    out, m = check_nvfp4(M, inp, name="c6_decode_nvfp4")
    wq = (quantize_gpu(M, inp["w13"]), quantize_gpu(M, inp["w2"]))
    o1, i1, _ = run_forward(M, inp, wq)
    o2, i2, _ = run_forward(M, inp, wq)
    assert torch.equal(o1, o2) and torch.equal(i1, i2) and torch.equal(o1, out)
    print(f"c6_decode_nvfp4: max scaled error {m:.3e}")


def test_grouped_ffn_nvfp4_matches_forward(M):
    """The FFN step entry point on the forward's own routing gives the
    forward's output after the combine."""
    inp = workloads.make_inputs("c1_tiny", DEV, shape=SHAPES["learned_small"][1], seed=17)
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    wq = (quantize_gpu(M, inp["w13"]), quantize_gpu(M, inp["w2"]))
    out, ids, tw = run_forward(M, inp, wq)
    R = T * k
    xhat = torch.empty_like(inp["x"])
    M.moe_rmsnorm(inp["x"], inp["norm_w"], inp["eps"], xhat)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    row_src = torch.empty((R,), dtype=torch.int32, device=DEV)
    rop = torch.empty((R,), dtype=torch.int32, device=DEV)
    xp = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    M.moe_permute(ids, T, E, k, offsets, row_src, rop, xhat=xhat, xp=xp, row_bytes=H * 2)
    xp16 = xp.to(torch.float16)
    act = torch.empty((R, I), dtype=torch.float16, device=DEV)
    y = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    shape = M.make_shape(T, H, E, I, k, inp["eps"], nvfp4=True)
    ws = M.alloc_workspace(M.moe_grouped_ffn_workspace_size(shape), DEV)
    (q13, sb13, sg13), (q2, sb2, sg2) = wq
    M.moe_grouped_ffn_nvfp4(shape, xp16, q13, sb13, sg13, q2, sb2, sg2, offsets, row_src, tw, act, y, ws)
    out2 = torch.empty_like(out)
    M.moe_combine(y, rop, T, k, out2, pair_order=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_forward_nvfp4_zero_tokens(M):
    shape = M.make_shape(0, 256, 8, 256, 2, nvfp4=True)
    ws = M.alloc_workspace(max(256, M.moe_ffn_workspace_size(shape)), DEV)
    w = torch.ones((256,), dtype=torch.bfloat16, device=DEV)
    q13 = torch.zeros((8, 512, 128), dtype=torch.uint8, device=DEV)
    sb13 = torch.zeros((8, 512, 16), dtype=torch.uint8, device=DEV)
    q2 = torch.zeros((8, 256, 128), dtype=torch.uint8, device=DEV)
    sb2 = torch.zeros((8, 256, 16), dtype=torch.uint8, device=DEV)
    sg = torch.ones((8,), dtype=torch.float32, device=DEV)
    rw = torch.zeros((256, 8), dtype=torch.float32, device=DEV)
    out = torch.empty((1, 256), dtype=torch.bfloat16, device=DEV)
    M.moe_ffn_forward_nvfp4(shape, w, w, q13, sb13, sg, q2, sb2, sg, out, ws, router_w=rw)
    torch.cuda.synchronize()
    assert M.device_status() == 0
