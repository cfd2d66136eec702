"""Block-wise FP8 on the GPU (E4M3 codes, one scale per 128 x 128 weight tile
and per 1 x 128 activation group): the quantiser bit-exact against the
oracle, and the forward against the oracle's block-wise forward."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads
from tests.parity_util import (TOL_FP8, assert_close, check_routing_e2e, covering_tokens, f64,
                               forward_xhat, o1_weights)

pytestmark = pytest.mark.gpu
DEV = "cuda"
E4M3 = np.array([O.e4m3_decode(c) for c in range(256)])


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_ffn_rms_gb300 as M
    return M


def quantize_gpu(M, w, block_rows):
    K = w.shape[-1]
    N = w.numel() // K
    q = torch.empty(w.shape, dtype=torch.uint8, device=DEV)
    lead = w.shape[:-2] + (w.shape[-2] // block_rows,) if w.dim() > 1 else ()
    s = torch.empty(lead + (K // 128,), dtype=torch.float32, device=DEV)
    M.moe_quantize_fp8_blocks(w, q, s, block_rows)
    assert N % block_rows == 0
    return q, s


def test_quantize_fp8_blocks_bit_exact(M):
    g = torch.Generator(device=DEV).manual_seed(41)
    w = (torch.randn((3, 256, 384), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w[1, 128:, 128:256] = 0          # an all-zero tile
    w[2, :128, :128] *= 1e-5         # a tile far below the others
    w[0, 3, 300] = 2.5               # one large element owns its tile's scale
    q, s = quantize_gpu(M, w, 128)
    torch.cuda.synchronize()
    for e in range(3):
        qo, so = O.quantize_blocks_e4m3(f64(w[e]), 128)
        np.testing.assert_array_equal(E4M3[q[e].cpu().numpy()], qo)
        np.testing.assert_array_equal(s[e].cpu().double().numpy(), so)
    assert s[1, 1, 1].item() == 1.0 and int(q[1, 128:, 128:256].max()) == 0
    # activation rows: one scale per row and 128-element group
    x = (torch.randn((37, 512), generator=g, device=DEV) * 3).to(torch.bfloat16)
    x[4] = 0
    x[9, 256:384] = 0
    qa, sa = quantize_gpu(M, x, 1)
    torch.cuda.synchronize()
    qo, so = O.quantize_blocks_e4m3(f64(x), 1)
    np.testing.assert_array_equal(E4M3[qa.cpu().numpy()], qo)
    np.testing.assert_array_equal(sa.cpu().double().numpy(), so)


def quantize_weights(M, inp):
    return quantize_gpu(M, inp["w13"], 128), quantize_gpu(M, inp["w2"], 128)


def run_forward(M, inp, wq, routed=None, engine=None, ws=None):
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    shape = M.make_shape(T, H, E, I, k, inp["eps"], fp8="block",
                         engine=M.ENGINE_AUTO if engine is None else engine)
    if ws is None:
        ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    (q13, s13), (q2, s2) = wq
    if routed is not None:
        ids, tw = routed
        M.moe_ffn_forward_routed(shape, inp["x"], inp["norm_w"], ids, tw, q13, q2, out, ws,
                                 w13_scale=s13, w2_scale=s2)
        torch.cuda.synchronize()
        return out, ids, tw
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    M.moe_ffn_forward(shape, inp["x"], inp["norm_w"], q13, q2, out, ws, router_w=inp["router_w"],
                      router_logits=inp["router_logits"], router_bias=inp["router_bias"],
                      w13_scale=s13, w2_scale=s2, topk_ids_out=ids, topk_w_out=tw)
    torch.cuda.synchronize()
    return out, ids, tw


def check_fp8_block(M, inp, sample=None, seed=0, engine=None, name=""):
    """sample: None = every token, "tiles" = tokens reaching every (expert,
    128-row token tile), an int = that many random tokens."""
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    wq = quantize_weights(M, inp)
    M.device_status(clear=True)
    shape = M.make_shape(T, H, E, I, k, inp["eps"], fp8="block",
                         engine=M.ENGINE_AUTO if engine is None else engine)
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    out, ids, tw = run_forward(M, inp, wq, engine=engine, ws=ws)
    ids_g = ids.cpu().numpy()
    xg = f64(forward_xhat(M, ws, T, H))
    ids_use, w_use, xhat, _ = check_routing_e2e(
        ids_g, tw.cpu().double().numpy(), f64(inp["x"]), f64(inp["norm_w"]), inp["eps"], k,
        xhat_gpu=xg, router_w=None if inp["router_w"] is None else f64(inp["router_w"]),
        router_bias=None if inp["router_bias"] is None else f64(inp["router_bias"]),
        logits=None if inp["router_logits"] is None else f64(inp["router_logits"]), name=name)
    toks = np.arange(T)
    if sample == "tiles":
        toks, ntiles = covering_tokens(ids_use, E, k, tile=128, n_min=256, seed=seed)
        print(f"{inp['name']}: {len(toks)} tokens cover all {ntiles} (expert, token tile) pairs")
    elif sample is not None and sample < T:
        toks = np.sort(np.random.default_rng(seed).choice(T, size=sample, replace=False))
    used = np.unique(ids_use[toks])
    b13 = {int(e): O.quantize_blocks_e4m3(f64(inp["w13"][e]), 128) for e in used}
    b2 = {int(e): O.quantize_blocks_e4m3(f64(inp["w2"][e]), 128) for e in used}
    ref = O.ffn_token_outputs(xhat[toks], ids_use[toks], w_use[toks], None, None, I, fp8="block",
                              wq13_of=b13.get, wq2_of=b2.get)
    m = assert_close(f64(out)[toks], ref, TOL_FP8, inp["name"] + " fp8 block")
    assert M.device_status() == 0
    return out, m, wq


SHAPES = {
    # name: (workload the distributions come from, shape, routing)
    "learned_small": ("c1_tiny", workloads.Shape(T=16, H=256, E=8, k=2, I=256), "learned"),
    "zipf": ("c3_decode_skewed", workloads.Shape(T=5, H=512, E=16, k=4, I=512), "zipf"),
    "balanced": ("c2_decode_balanced", workloads.Shape(T=16, H=256, E=64, k=8, I=256), "balanced"),
    "rows_64": ("c1_tiny", workloads.Shape(T=64, H=256, E=4, k=2, I=256), "learned"),
    "two_chunks": ("c1_tiny", workloads.Shape(T=300, H=256, E=2, k=1, I=384), "learned"),
    "single_token": ("c1_tiny", workloads.Shape(T=1, H=768, E=8, k=4, I=128), "learned"),
    "odd_groups": ("c1_tiny", workloads.Shape(T=7, H=512, E=4, k=2, I=640), "learned"),
    # the largest K of each GEMM: 64 scale groups (H or I = 8192)
    "max_groups_fc1": ("c1_tiny", workloads.Shape(T=6, H=8192, E=4, k=2, I=256), "learned"),
    "max_groups_fc2": ("c1_tiny", workloads.Shape(T=6, H=256, E=4, k=2, I=8192), "learned"),
    "max_experts": ("c3_decode_skewed", workloads.Shape(T=40, H=256, E=256, k=8, I=256), "zipf"),
}


@pytest.mark.parametrize("engine", ["auto", "decode", "prefill"])
@pytest.mark.parametrize("name", list(SHAPES))
def test_forward_fp8_block_small(M, name, engine):
    """Both engines: the weight-streaming launch (decode) and the token tiles
    with a separate group quantisation (prefill); the workloads' own weights
    and weights rescaled to outputs of order one."""
    cfg, shape, routing = SHAPES[name]
    eng = {"auto": None, "decode": M.ENGINE_DECODE, "prefill": M.ENGINE_PREFILL}[engine]
    for o1 in (False, True):
        inp = workloads.make_inputs(cfg, DEV, shape=shape, routing=routing, seed=19)
        inp["name"] = f"{name}/{engine}" + (" o1" if o1 else "")
        if o1:
            o1_weights(inp)
        check_fp8_block(M, inp, engine=eng)


def test_forward_fp8_block_full_decode_workload(M):
    """The block-wise FP8 decode workload (T=16, H=4096, E=64, k=8, I=1536),
    every token recomputed by the oracle; the run is deterministic."""
    inp = workloads.make_inputs("c7_decode_fp8_block", DEV)
    out, m, wq = check_fp8_block(M, inp, name="c7_decode_fp8_block")
    o1, i1, _ = run_forward(M, inp, wq)
    o2, i2, _ = run_forward(M, inp, wq)
    assert torch.equal(o1, o2) and torch.equal(i1, i2) and torch.equal(o1, out)
    print(f"c7_decode_fp8_block: max scaled error {m:.3e}")


def test_forward_fp8_block_prefill_workload(M):
    """Block-wise FP8 at the prefill size (T=4096, H=4096, E=64, k=8, I=1536,
    token tiles); the oracle recomputes tokens that reach every (expert,
    128-row token tile)."""
    inp = workloads.make_inputs("c9_prefill_fp8_block", DEV)
    inp["name"] = "c9_prefill_fp8_block"
    _, m, _ = check_fp8_block(M, inp, sample="tiles", name="c9_prefill_fp8_block")
    print(f"c9_prefill_fp8_block: max scaled error {m:.3e}")
    del inp
    torch.cuda.empty_cache()


def test_forward_fp8_block_zero_tokens(M):
    shape = M.make_shape(0, 256, 8, 128, 2, fp8="block")
    ws = M.alloc_workspace(max(256, M.moe_ffn_workspace_size(shape)), DEV)
    w = torch.ones((256,), dtype=torch.bfloat16, device=DEV)
    q13 = torch.zeros((8, 256, 256), dtype=torch.uint8, device=DEV)
    q2 = torch.zeros((8, 256, 128), dtype=torch.uint8, device=DEV)
    s13 = torch.ones((8, 2, 2), dtype=torch.float32, device=DEV)
    s2 = torch.ones((8, 2, 1), dtype=torch.float32, device=DEV)
    rw = torch.zeros((256, 8), dtype=torch.float32, device=DEV)
    out = torch.empty((1, 256), dtype=torch.bfloat16, device=DEV)
    M.moe_ffn_forward(shape, w, w, q13, q2, out, ws, router_w=rw, w13_scale=s13, w2_scale=s2)
    torch.cuda.synchronize()
    assert M.device_status() == 0


def test_routed_forward_fp8_block_matches_routed_oracle(M):
    inp = workloads.make_inputs("c1_tiny", DEV, shape=SHAPES["rows_64"][1], seed=23)
    inp["name"] = "routed"
    T, k, E = inp["T"], inp["k"], inp["E"]
    g = torch.Generator(device="cpu").manual_seed(5)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    tw = torch.rand((T, k), generator=g, dtype=torch.float32)
    tw /= tw.sum(dim=1, keepdim=True)
    wq = quantize_weights(M, inp)
    out, _, _ = run_forward(M, inp, wq, routed=(ids.to(DEV), tw.to(DEV)))
    res = O.moe_ffn_forward(f64(inp["x"]), f64(inp["norm_w"]), inp["eps"], k, f64(inp["w13"]),
                            f64(inp["w2"]), ids=ids.numpy(), topk_w=tw.double().numpy(), fp8="block")
    assert_close(f64(out), res["out"], TOL_FP8, "routed fp8 block")


@pytest.mark.parametrize("engine", ["decode", "prefill"])
def test_grouped_ffn_fp8_block_matches_forward(M, engine):
    """The FFN step entry point on the forward's own routing and gathered
    E4M3 rows gives the forward's output after the combine."""
    inp = workloads.make_inputs("c1_tiny", DEV, shape=SHAPES["learned_small"][1], seed=29)
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    eng = M.ENGINE_DECODE if engine == "decode" else M.ENGINE_PREFILL
    wq = quantize_weights(M, inp)
    out, ids, tw = run_forward(M, inp, wq, engine=eng)
    R = T * k
    xhat = torch.empty_like(inp["x"])
    M.moe_rmsnorm(inp["x"], inp["norm_w"], inp["eps"], xhat)
    xq, xs = quantize_gpu(M, xhat, 1)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    row_src = torch.empty((R,), dtype=torch.int32, device=DEV)
    rop = torch.empty((R,), dtype=torch.int32, device=DEV)
    M.moe_permute(ids, T, E, k, offsets, row_src, rop)
    tok = (row_src.long() // k)
    xp = xq[tok].contiguous()
    xps = xs[tok].contiguous()
    act = torch.empty((R, I), dtype=torch.uint8, device=DEV)
    y = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    shape = M.make_shape(T, H, E, I, k, inp["eps"], fp8="block", engine=eng)
    ws = M.alloc_workspace(M.moe_grouped_ffn_workspace_size(shape), DEV)
    (q13, s13), (q2, s2) = wq
    M.moe_grouped_ffn(shape, xp, q13, q2, offsets, row_src, tw, act, y, ws, xp_scale=xps,
                      w13_scale=s13, w2_scale=s2)
    out2 = torch.empty_like(out)
    M.moe_combine(y, rop, T, k, out2, pair_order=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
