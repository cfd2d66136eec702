"""GPU parity: every C-ABI entry point and the whole forward against the CPU
oracle on the same seeded inputs.

Small ragged shapes span several tiles in every dimension; the five
reference workloads run at full size in the launch configuration the bench
times, with outputs compared on all tokens (tiny, decode) or on a seeded
token sample (skewed decode, prefill)."""
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads
from tests.parity_util import (TOL_BF16, TOL_FP8, assert_close, check_router,
                               check_routing_e2e, covering_tokens, f64, forward_xhat, o1_weights,
                               record,
                               scaled_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_ffn_rms_gb300 as M
    M.check_device()
    M.device_status(clear=True)
    return M


DEV = "cuda"

SMALL = {
    # name: (T, H, E, k, I)
    "ragged_a": workloads.Shape(T=37, H=256, E=6, k=2, I=320),
    "ragged_b": workloads.Shape(T=200, H=512, E=8, k=3, I=384),
    "wide_e": workloads.Shape(T=45, H=320, E=256, k=8, I=192),
    "prefill_like": workloads.Shape(T=300, H=384, E=4, k=2, I=256),
    "single": workloads.Shape(T=1, H=128, E=8, k=4, I=128),
    # > 256 rows per expert: a full 256-row wide tile and a one-half tail
    "two_wide_chunks": workloads.Shape(T=700, H=256, E=2, k=1, I=256),
}

ENGINES = ["auto", "decode", "prefill", "prefill_wide", "simt"]
# decode: FC1 and FC2 fused in one persistent launch; decode_mega: the whole
# forward in one cooperative launch where it is covered (MOE_MEGA=1);
# decode_unfused: FC1 and FC2 in two launches
FWD_ENGINES = ENGINES + ["decode_mega", "decode_unfused"]
# prefill: 128-row token tiles; prefill_wide: 256-row token tiles (two M = 128
# MMAs per K step), which the engine picks by itself at large batches
ENV_SWITCHES = ("MOE_FORCE_SIMT", "MOE_FUSE", "MOE_ROUTER_TC", "MOE_MEGA", "MOE_WIDE_TILES")


def _set_engine(shape_obj, engine, M):
    for v in ENV_SWITCHES:
        os.environ.pop(v, None)
    if engine == "simt":
        os.environ["MOE_FORCE_SIMT"] = "1"
        return M.ENGINE_AUTO
    if engine == "decode_mega":
        os.environ["MOE_MEGA"] = "1"
        return M.ENGINE_DECODE
    if engine == "decode_unfused":
        os.environ["MOE_FUSE"] = "0"
        return M.ENGINE_DECODE
    if engine == "prefill":
        os.environ["MOE_WIDE_TILES"] = "0"
    if engine == "prefill_wide":
        os.environ["MOE_WIDE_TILES"] = "1"
        return M.ENGINE_PREFILL
    return {"auto": M.ENGINE_AUTO, "decode": M.ENGINE_DECODE, "prefill": M.ENGINE_PREFILL}[engine]


@pytest.fixture(autouse=True)
def _clear_env():
    yield
    for v in ENV_SWITCHES:
        os.environ.pop(v, None)


# ----------------------------------------------------------------- steps ---

@pytest.mark.parametrize("T,H", [(1, 64), (5, 256), (37, 4096), (3, 7168)])
def test_rmsnorm(M, T, H):
    g = torch.Generator(device=DEV).manual_seed(T * 1000 + H)
    x = torch.randn((T, H), generator=g, device=DEV).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn((H,), generator=g, device=DEV)).to(torch.bfloat16)
    y = torch.empty_like(x)
    M.moe_rmsnorm(x, w, 1e-6, y)
    ref = O.rms_norm(f64(x), f64(w), 1e-6)
    got = f64(y)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(got - ref) <= ulp + 1e-30)   # at most one bf16 step (fp32 vs fp64)
    assert np.mean(got == ref) > 0.99


def test_rmsnorm_fp8_quant(M):
    T, H = 9, 4096
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randn((T, H), generator=g, device=DEV).to(torch.bfloat16)
    x[3] = 0
    w = (1 + 0.1 * torch.randn((H,), generator=g, device=DEV)).to(torch.bfloat16)
    y = torch.empty_like(x)
    yq = torch.empty((T, H), dtype=torch.uint8, device=DEV)
    ys = torch.empty((T,), dtype=torch.float32, device=DEV)
    M.moe_rmsnorm(x, w, 1e-6, y, yq, ys)
    # the codes are decided from the GPU's bf16 row: quantise that row in the oracle
    q, s = O.quantize_rows_e4m3(f64(y))
    got_q = yq.cpu().view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(got_q, q)
    np.testing.assert_array_equal(ys.cpu().double().numpy(), s)
    assert ys[3].item() == 1.0


def test_quantize_rows_bit_exact(M):
    g = torch.Generator(device=DEV).manual_seed(6)
    x = (0.02 * torch.randn((300, 512), generator=g, device=DEV)).to(torch.bfloat16)
    x[7] = 0
    x[8, 5] = 1e4
    q = torch.empty((300, 512), dtype=torch.uint8, device=DEV)
    s = torch.empty((300,), dtype=torch.float32, device=DEV)
    M.moe_quantize_fp8_rows(x, q, s)
    qr, sr = O.quantize_rows_e4m3(f64(x))
    np.testing.assert_array_equal(q.cpu().view(torch.float8_e4m3fn).double().numpy(), qr)
    np.testing.assert_array_equal(s.cpu().double().numpy(), sr)


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (37, 64, 8), (64, 256, 8), (517, 64, 8), (9, 5, 5)])
def test_route_topk_given_logits_bit_exact(M, T, E, k):
    """Fed fp32 logits, the selection must equal the oracle's top-k on the
    same fp32 values exactly (ids and their order); weights within fp32."""
    g = torch.Generator(device=DEV).manual_seed(T + E + k)
    logits = torch.randn((T, E), generator=g, device=DEV) * 2
    logits[:, : E // 3] = torch.round(logits[:, : E // 3])       # plenty of exact ties
    bias = torch.randn((E,), generator=g, device=DEV)
    for b in (None, bias):
        ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        lo = torch.empty((T, E), dtype=torch.float32, device=DEV)
        M.moe_route_topk(T, 0, E, k, ids, w, logits_in=logits, router_bias=b, logits_out=lo)
        l32 = (logits + b if b is not None else logits)           # fp32 add, as the kernel
        np.testing.assert_array_equal(lo.cpu().numpy(), l32.cpu().numpy())
        ids_ref, w_ref = O.topk_renorm(l32.cpu().double().numpy(), k)
        np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
        np.testing.assert_allclose(w.cpu().double().numpy(), w_ref, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("tc", ["1", "0"])
@pytest.mark.parametrize("cfg", ["c1_tiny", "c3_decode_skewed", "c5_prefill", "wide_prefill",
                                 "small_uneven", "small_bias", "odd_e_prefill", "split_k_uneven",
                                 "split_k_odd_e"])
def test_route_topk_router(M, cfg, tc):
    """Router logits from x_hat and W_r (tensor-core bf16x3 split for >= 256
    tokens unless MOE_ROUTER_TC=0; a one-CTA-per-token router fused with top-k
    when H * E is small; else fp32 SIMT split-K) against the fp64 oracle."""
    os.environ["MOE_ROUTER_TC"] = tc
    if cfg == "wide_prefill":   # E = 256 -> three N tiles of the split router GEMM
        inp = workloads.make_inputs("c3_decode_skewed", DEV,
                                    shape=workloads.Shape(T=600, H=1024, E=256, k=8, I=256))
    elif cfg == "small_uneven":  # E does not divide the 256 threads of the small router
        inp = workloads.make_inputs("c1_tiny", DEV,
                                    shape=workloads.Shape(T=5, H=512, E=24, k=3, I=256))
    elif cfg == "small_bias":    # Zipf bias on a small router, H * E at the size limit
        inp = workloads.make_inputs("c3_decode_skewed", DEV,
                                    shape=workloads.Shape(T=9, H=256, E=256, k=8, I=256))
    elif cfg == "odd_e_prefill":  # tensor-core router with 3E = 21 logit columns (odd row pitch)
        inp = workloads.make_inputs("c1_tiny", DEV,
                                    shape=workloads.Shape(T=300, H=512, E=7, k=2, I=256))
    elif cfg == "split_k_uneven":  # 25 K stages over 3 splits (8, 8, 9)
        inp = workloads.make_inputs("c1_tiny", DEV,
                                    shape=workloads.Shape(T=256, H=1600, E=24, k=2, I=256))
    elif cfg == "split_k_odd_e":  # 4 splits of 3E = 21 columns: odd column offsets per split
        inp = workloads.make_inputs("c1_tiny", DEV,
                                    shape=workloads.Shape(T=400, H=2048, E=7, k=2, I=256))
    else:
        inp = workloads.make_inputs(cfg, DEV)
    T, H, E, k = inp["T"], inp["H"], inp["E"], inp["k"]
    xhat = torch.empty_like(inp["x"])
    M.moe_rmsnorm(inp["x"], inp["norm_w"], inp["eps"], xhat)
    ws = M.alloc_workspace(M.moe_route_workspace_size(T, H, E), DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    lo = torch.empty((T, E), dtype=torch.float32, device=DEV)
    M.moe_route_topk(T, H, E, k, ids, w, xhat=xhat, router_w=inp["router_w"],
                     router_bias=inp["router_bias"], logits_out=lo, workspace=ws)
    torch.cuda.synchronize()
    # the oracle's fp64 logits from the GPU's own x_hat: only the router's
    # summation differs, so the tie band is twice each token's logit error
    l64 = O.router_logits(f64(xhat), f64(inp["router_w"]),
                          None if inp["router_bias"] is None else f64(inp["router_bias"]))
    _, counts = check_router(ids.cpu().numpy(), w.cpu().double().numpy(),
                             lo.cpu().double().numpy(), l64, k)
    record(f"router {cfg} tc={tc}", counts)
    print(f"{cfg} tc={tc}: {counts}")
    os.environ.pop("MOE_ROUTER_TC", None)


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (37, 6, 2), (64, 256, 8), (4096, 64, 8), (333, 7, 7),
                                   (1000, 256, 8), (600, 3, 2)])
def test_permute_bit_exact(M, T, E, k):
    g = torch.Generator().manual_seed(T * 7 + E)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    if T > 10:
        ids[: T // 3] = torch.arange(k, dtype=torch.int32)   # hot experts 0..k-1
    ids_d = ids.to(DEV)
    H = 64
    xhat = torch.randn((T, H), device=DEV).to(torch.bfloat16)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    row_src = torch.empty((T * k,), dtype=torch.int32, device=DEV)
    rop = torch.empty((T * k,), dtype=torch.int32, device=DEV)
    xp = torch.empty((T * k, H), dtype=torch.bfloat16, device=DEV)
    ws = M.alloc_workspace(max(16, M.moe_permute_workspace_size(T, E, k)), DEV)
    M.moe_permute(ids_d, T, E, k, offsets, row_src, rop, xhat=xhat, xp=xp, row_bytes=H * 2,
                  workspace=ws)
    off_ref, rs_ref = O.permute(ids.numpy(), E)
    np.testing.assert_array_equal(offsets.cpu().numpy(), off_ref)
    np.testing.assert_array_equal(row_src.cpu().numpy(), rs_ref)
    inv = np.empty(T * k, dtype=np.int64)
    inv[rs_ref] = np.arange(T * k)
    np.testing.assert_array_equal(rop.cpu().numpy(), inv)
    np.testing.assert_array_equal(f64(xp), f64(xhat)[rs_ref // k])
    assert M.device_status() == 0


@pytest.mark.parametrize("T", [3, 1500])
def test_permute_flags_out_of_range_ids(M, T):
    base = torch.tensor([[0, 1], [2, 9], [1, -1]], dtype=torch.int32)
    ids = base.repeat((T + 2) // 3, 1)[:T].contiguous().to(DEV)
    offsets = torch.empty((5,), dtype=torch.int32, device=DEV)
    rs = torch.empty((2 * T,), dtype=torch.int32, device=DEV)
    rop = torch.empty((2 * T,), dtype=torch.int32, device=DEV)
    ws = M.alloc_workspace(max(16, M.moe_permute_workspace_size(T, 4, 2)), DEV)
    M.moe_permute(ids, T, 4, 2, offsets, rs, rop, workspace=ws)
    assert M.device_status(clear=True) == 1        # MOE_ERR_INVALID_ARG recorded
    n = T // 3
    assert offsets.cpu().tolist() == [0, n, 3 * n, 4 * n, 4 * n]
    assert rop.cpu().tolist()[3] == -1 and rop.cpu().tolist()[5] == -1
    assert M.device_status() == 0


def test_silu_and_mul(M):
    g = torch.Generator(device=DEV).manual_seed(11)
    R, I = 77, 320
    h = (3 * torch.randn((R, 2 * I), generator=g, device=DEV)).to(torch.bfloat16)
    a = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    M.moe_silu_and_mul(h, a)
    ref = O.silu_and_mul(f64(h), I)
    got = f64(a)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(got - ref) <= ulp + 1e-30)
    assert np.mean(got == ref) > 0.99


@pytest.mark.parametrize("ydtype", [torch.float32, torch.bfloat16])
def test_combine(M, ydtype):
    g = torch.Generator(device=DEV).manual_seed(12)
    T, k, H = 29, 3, 192
    y = torch.randn((T * k, H), generator=g, device=DEV).to(ydtype)
    perm = torch.randperm(T * k, generator=torch.Generator().manual_seed(3)).to(torch.int32)
    rop = torch.empty_like(perm)
    rop[perm.long()] = torch.arange(T * k, dtype=torch.int32)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    M.moe_combine(y, rop.to(DEV), T, k, out)
    ref = O.combine(f64(y), perm.numpy(), T, k)
    got = f64(out)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(got - ref) <= ulp + 1e-30)
    # the same rows in (token, slot) order, with one skipped pair
    y_pair = torch.empty_like(y)
    y_pair[perm.long().to(DEV)] = y
    rop2 = rop.clone()
    rop2[4] = -1
    out2 = torch.empty_like(out)
    M.moe_combine(y_pair, rop2.to(DEV), T, k, out2, pair_order=True)
    keep = np.ones(T * k)
    keep[4] = 0
    yp = f64(y_pair) * keep[:, None]
    ref2 = O.bf16_round(yp.reshape(T, k, H).sum(axis=1))
    assert np.all(np.abs(f64(out2) - ref2) <= np.ldexp(1.0, np.frexp(np.abs(ref2))[1] - 8) + 1e-30)


def _grouped_inputs(shape, seed, fp8=False, hot=False):
    T, H, E, k, I = shape.T, shape.H, shape.E, shape.k, shape.I
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    if hot:
        ids[:, 0] = 0
        for t in range(T):
            if (ids[t, 1:] == 0).any():
                ids[t] = torch.tensor(list(range(k)), dtype=torch.int32)
    offsets, row_src = O.permute(ids.numpy(), E)
    gd = torch.Generator(device=DEV).manual_seed(seed)
    xp = torch.randn((T * k, H), generator=gd, device=DEV).to(torch.bfloat16)
    w13 = (0.05 * torch.randn((E, 2 * I, H), generator=gd, device=DEV)).to(torch.bfloat16)
    w2 = (0.05 * torch.randn((E, H, I), generator=gd, device=DEV)).to(torch.bfloat16)
    a = torch.randn((T * k, I), generator=gd, device=DEV).to(torch.bfloat16)
    tw = torch.rand((T * k,), generator=gd, device=DEV)
    return dict(ids=ids, offsets=torch.from_numpy(offsets).to(DEV), offsets_np=offsets,
                row_src=torch.from_numpy(row_src).to(DEV), row_src_np=row_src, xp=xp, w13=w13,
                w2=w2, a=a, tw=tw)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("name", ["ragged_a", "ragged_b", "prefill_like", "single", "hot",
                                  "two_wide_chunks"])
def test_grouped_gemm_modes(M, engine, name):
    shape = SMALL.get(name, workloads.Shape(T=150, H=256, E=5, k=2, I=192))
    d = _grouped_inputs(shape, 21, hot=(name == "hot"))
    T, H, E, k, I = shape.T, shape.H, shape.E, shape.k, shape.I
    R = T * k
    eng = _set_engine(shape, engine, M)
    ms = M.make_shape(T, H, E, I, k, engine=eng)
    off = d["offsets_np"]
    w13_of = lambda e: f64(d["w13"][e])
    w2_of = lambda e: f64(d["w2"][e])
    # FC1 + silu_and_mul
    c1 = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    M.moe_grouped_gemm(ms, M.GEMM_FC1_SILU, d["xp"], d["w13"], d["offsets"], c1)
    ref1 = O.grouped_fc1(f64(d["xp"]), off, w13_of, I)
    assert_close(f64(c1), ref1, TOL_BF16, f"FC1+silu {name}/{engine}")
    # FC1 raw
    c0 = torch.empty((R, 2 * I), dtype=torch.bfloat16, device=DEV)
    M.moe_grouped_gemm(ms, M.GEMM_FC1_RAW, d["xp"], d["w13"], d["offsets"], c0)
    ref0 = np.zeros((R, 2 * I))
    for e in range(E):
        ref0[off[e]:off[e + 1]] = f64(d["xp"])[off[e]:off[e + 1]] @ w13_of(e).T
    assert_close(f64(c0), O.bf16_round(ref0), TOL_BF16, f"FC1 raw {name}/{engine}")
    # FC2 with the routing weight
    c2 = torch.empty((R, H), dtype=torch.float32, device=DEV)
    M.moe_grouped_gemm(ms, M.GEMM_FC2, d["a"], d["w2"], d["offsets"], c2, row_src=d["row_src"],
                       topk_w=d["tw"])
    row_w = f64(d["tw"])[d["row_src_np"]]
    ref2 = O.grouped_fc2(f64(d["a"]), off, w2_of, row_w)
    assert_close(f64(c2), ref2, 1e-3, f"FC2 {name}/{engine}")
    c3 = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    M.moe_grouped_gemm(ms, M.GEMM_FC2_BF16, d["a"], d["w2"], d["offsets"], c3,
                       row_src=d["row_src"], topk_w=d["tw"])
    # rows come back in (token, slot) order: c3[row_src[r]] holds row r
    ref3 = np.empty_like(ref2)
    ref3[d["row_src_np"]] = ref2
    assert_close(f64(c3), O.bf16_round(ref3), TOL_BF16, f"FC2 bf16 {name}/{engine}")
    # bf16 rows are the fp32 rows rounded once (same kernel family, same sums)
    assert torch.equal(c3[d["row_src"].long()], c2.to(torch.bfloat16))
    torch.cuda.synchronize()
    assert M.device_status() == 0


@pytest.mark.parametrize("engine", ENGINES)
def test_grouped_gemm_fp8(M, engine):
    shape = workloads.Shape(T=40, H=256, E=6, k=3, I=192)
    d = _grouped_inputs(shape, 31)
    T, H, E, k, I = shape.T, shape.H, shape.E, shape.k, shape.I
    R = T * k
    eng = _set_engine(shape, engine, M)
    ms = M.make_shape(T, H, E, I, k, fp8=True, engine=eng)
    q13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=DEV)
    s13 = torch.empty((E, 2 * I), dtype=torch.float32, device=DEV)
    q2 = torch.empty((E, H, I), dtype=torch.uint8, device=DEV)
    s2 = torch.empty((E, H), dtype=torch.float32, device=DEV)
    M.moe_quantize_fp8_rows(d["w13"], q13, s13)
    M.moe_quantize_fp8_rows(d["w2"], q2, s2)
    xq = torch.empty((R, H), dtype=torch.uint8, device=DEV)
    xs = torch.empty((R,), dtype=torch.float32, device=DEV)
    M.moe_quantize_fp8_rows(d["xp"], xq, xs)
    aq = torch.empty((R, I), dtype=torch.uint8, device=DEV)
    as_ = torch.empty((R,), dtype=torch.float32, device=DEV)
    M.moe_quantize_fp8_rows(d["a"], aq, as_)
    off = d["offsets_np"]
    c1 = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    M.moe_grouped_gemm(ms, M.GEMM_FC1_SILU, xq, q13, d["offsets"], c1, a_scale=xs, w_scale=s13)
    Oq13 = [O.quantize_rows_e4m3(f64(d["w13"][e])) for e in range(E)]
    Oq2 = [O.quantize_rows_e4m3(f64(d["w2"][e])) for e in range(E)]
    xq_r, xs_r = O.quantize_rows_e4m3(f64(d["xp"]))
    ref1 = O.grouped_fc1_fp8(xq_r, xs_r, off, lambda e: Oq13[e][0], lambda e: Oq13[e][1], I)
    assert_close(f64(c1), ref1, TOL_FP8, f"FP8 FC1 {engine}")
    c2 = torch.empty((R, H), dtype=torch.float32, device=DEV)
    M.moe_grouped_gemm(ms, M.GEMM_FC2, aq, q2, d["offsets"], c2, a_scale=as_, w_scale=s2,
                       row_src=d["row_src"], topk_w=d["tw"])
    row_w = f64(d["tw"])[d["row_src_np"]]
    ref2 = O.grouped_fc2_fp8(f64(d["a"]), off, lambda e: Oq2[e][0], lambda e: Oq2[e][1], row_w)
    assert_close(f64(c2), ref2, 1e-3, f"FP8 FC2 {engine}")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("engine", ["decode", "prefill", "prefill_wide"])
@pytest.mark.parametrize("name", ["ragged_a", "prefill_like", "hot"])
def test_grouped_ffn_matches_steps(M, engine, name, fp8):
    """moe_grouped_ffn (fused on the decode engine for bf16) gives the same bits
    as FC1_SILU then FC2_BF16 through moe_grouped_gemm, and matches the oracle."""
    shape = SMALL.get(name, workloads.Shape(T=150, H=256, E=5, k=2, I=192))
    d = _grouped_inputs(shape, 41, hot=(name == "hot"))
    T, H, E, k, I = shape.T, shape.H, shape.E, shape.k, shape.I
    R = T * k
    eng = _set_engine(shape, engine, M)
    ms = M.make_shape(T, H, E, I, k, fp8=fp8, engine=eng)
    xp, w13, w2, s13, s2, xs = d["xp"], d["w13"], d["w2"], None, None, None
    if fp8:
        w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=DEV)
        s13 = torch.empty((E, 2 * I), dtype=torch.float32, device=DEV)
        w2 = torch.empty((E, H, I), dtype=torch.uint8, device=DEV)
        s2 = torch.empty((E, H), dtype=torch.float32, device=DEV)
        M.moe_quantize_fp8_rows(d["w13"], w13, s13)
        M.moe_quantize_fp8_rows(d["w2"], w2, s2)
        xp = torch.empty((R, H), dtype=torch.uint8, device=DEV)
        xs = torch.empty((R,), dtype=torch.float32, device=DEV)
        M.moe_quantize_fp8_rows(d["xp"], xp, xs)
    act = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    ws = M.alloc_workspace(M.moe_grouped_ffn_workspace_size(ms), DEV)
    for _ in range(2):  # twice: the scheduler counters are reset per call
        M.moe_grouped_ffn(ms, xp, w13, w2, d["offsets"], d["row_src"], d["tw"], act, y, ws,
                          xp_scale=xs, w13_scale=s13, w2_scale=s2)
    act2 = torch.empty_like(act)
    y2 = torch.empty_like(y)
    M.moe_grouped_gemm(ms, M.GEMM_FC1_SILU, xp, w13, d["offsets"], act2, a_scale=xs, w_scale=s13)
    a2, as2 = act2, None
    if fp8:
        a2 = torch.empty((R, I), dtype=torch.uint8, device=DEV)
        as2 = torch.empty((R,), dtype=torch.float32, device=DEV)
        M.moe_quantize_fp8_rows(act2, a2, as2)
    M.moe_grouped_gemm(ms, M.GEMM_FC2_BF16, a2, w2, d["offsets"], y2, a_scale=as2, w_scale=s2,
                       row_src=d["row_src"], topk_w=d["tw"])
    torch.cuda.synchronize()
    assert torch.equal(act, act2) and torch.equal(y, y2)
    if not fp8:
        off = d["offsets_np"]
        ref_a = O.grouped_fc1(f64(d["xp"]), off, lambda e: f64(d["w13"][e]), I)
        assert_close(f64(act), ref_a, TOL_BF16, f"ffn act {name}/{engine}")
        row_w = f64(d["tw"])[d["row_src_np"]]
        ref_y = O.grouped_fc2(ref_a, off, lambda e: f64(d["w2"][e]), row_w)
        ref_pair = np.empty_like(ref_y)
        ref_pair[d["row_src_np"]] = ref_y
        assert_close(f64(y), ref_pair, TOL_BF16, f"ffn y {name}/{engine}")
    assert M.device_status() == 0


# ------------------------------------------------------------ end to end ---

def _run_forward(M, inp, engine=None, fp8_weights=None, out=None, ws=None):
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    eng = M.ENGINE_AUTO if engine is None else engine
    shape = M.make_shape(T, H, E, I, k, inp["eps"], fp8=inp["fp8"], engine=eng)
    if ws is None:
        ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    w13, w2, s13, s2 = inp["w13"], inp["w2"], None, None
    if inp["fp8"]:
        w13, s13, w2, s2 = fp8_weights
    M.moe_ffn_forward(shape, inp["x"], inp["norm_w"], w13, w2, out, ws, router_w=inp["router_w"],
                      router_logits=inp["router_logits"], router_bias=inp["router_bias"],
                      w13_scale=s13, w2_scale=s2, topk_ids_out=ids, topk_w_out=tw)
    torch.cuda.synchronize()
    return out, ids, tw


def quantize_weights_gpu(M, inp):
    E, H, I = inp["E"], inp["H"], inp["I"]
    q13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=DEV)
    s13 = torch.empty((E, 2 * I), dtype=torch.float32, device=DEV)
    q2 = torch.empty((E, H, I), dtype=torch.uint8, device=DEV)
    s2 = torch.empty((E, H), dtype=torch.float32, device=DEV)
    M.moe_quantize_fp8_rows(inp["w13"], q13, s13)
    M.moe_quantize_fp8_rows(inp["w2"], q2, s2)
    return q13, s13, q2, s2


def check_forward(M, inp, sample=None, engine=None, seed=0, name=None):
    """Run the library forward and compare with the oracle.

    sample: None = every token; "tiles" = tokens that reach every (expert,
    128-row token tile) of the permuted order (at least 256); an int = that
    many random tokens.  Routing: bit-exact outside the tie bands
    (parity_util.check_routing_e2e), counts recorded under ``name``."""
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    fp8w = quantize_weights_gpu(M, inp) if inp["fp8"] else None
    shape = M.make_shape(T, H, E, I, k, inp["eps"], fp8=inp["fp8"],
                         engine=M.ENGINE_AUTO if engine is None else engine)
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    out, ids, tw = _run_forward(M, inp, engine, fp8w, ws=ws)
    ids_g = ids.cpu().numpy()
    xg = f64(forward_xhat(M, ws, T, H))
    ids_use, w_use, xhat, _ = check_routing_e2e(
        ids_g, tw.cpu().double().numpy(), f64(inp["x"]), f64(inp["norm_w"]), inp["eps"], k,
        xhat_gpu=xg, router_w=None if inp["router_w"] is None else f64(inp["router_w"]),
        router_bias=None if inp["router_bias"] is None else f64(inp["router_bias"]),
        logits=None if inp["router_logits"] is None else f64(inp["router_logits"]),
        name=name or "")
    toks = np.arange(T)
    if sample == "tiles":
        toks, ntiles = covering_tokens(ids_use, E, k, tile=128, n_min=256, seed=seed)
        print(f"{inp['name']}: {len(toks)} tokens cover all {ntiles} (expert, token tile) pairs")
    elif sample is not None and sample < T:
        toks = np.sort(np.random.default_rng(seed).choice(T, size=sample, replace=False))
    if inp["fp8"]:
        q13, s13, q2, s2 = fp8w
        # weight codes: bit-exact against the oracle's quantisation (a few experts)
        for e in sorted(set(ids_use[toks].reshape(-1).tolist()))[:3]:
            qr, sr = O.quantize_rows_e4m3(f64(inp["w13"][e]))
            np.testing.assert_array_equal(q13[e].cpu().view(torch.float8_e4m3fn).double().numpy(), qr)
            np.testing.assert_array_equal(s13[e].cpu().double().numpy(), sr)
        cache = {}

        def wq13(e):
            if ("13", e) not in cache:
                cache[("13", e)] = O.quantize_rows_e4m3(f64(inp["w13"][e]))
            return cache[("13", e)]

        def wq2(e):
            if ("2", e) not in cache:
                cache[("2", e)] = O.quantize_rows_e4m3(f64(inp["w2"][e]))
            return cache[("2", e)]
        ref = O.ffn_token_outputs(xhat[toks], ids_use[toks], w_use[toks], None, None, I, fp8=True,
                                  wq13_of=wq13, wq2_of=wq2)
        tol = TOL_FP8
    else:
        ref = O.ffn_token_outputs(xhat[toks], ids_use[toks], w_use[toks],
                                  lambda e: f64(inp["w13"][e]), lambda e: f64(inp["w2"][e]), I)
        tol = TOL_BF16
    got = f64(out)[toks]
    m = assert_close(got, ref, tol, inp["name"])
    assert M.device_status() == 0
    return m, len(toks)


@pytest.mark.parametrize("engine", FWD_ENGINES)
@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small_shapes(M, name, engine):
    """Every engine on ragged shapes: the learned and the Zipf-biased router
    with expert weights rescaled to outputs of order one, and the learned
    router with the workloads' own N(0, 0.02) weights."""
    for routing, o1 in (("learned", True), ("zipf", True), ("learned", False)):
        inp = workloads.make_inputs("c1_tiny", DEV, shape=SMALL[name], routing=routing, seed=7)
        if o1:
            o1_weights(inp)
        eng = _set_engine(None, engine, M)
        check_forward(M, inp, engine=eng)


def test_forward_balanced_small(M):
    inp = workloads.make_inputs("c2_decode_balanced", DEV,
                                shape=workloads.Shape(T=16, H=256, E=64, k=8, I=128))
    check_forward(M, inp)
    check_forward(M, o1_weights(inp))


def test_forward_fp8_small(M):
    inp = workloads.make_inputs("c4_decode_fp8", DEV,
                                shape=workloads.Shape(T=24, H=256, E=16, k=4, I=192),
                                routing="learned")
    check_forward(M, inp)
    check_forward(M, o1_weights(inp))


@pytest.mark.parametrize("cfg,sample", [("c1_tiny", None), ("c2_decode_balanced", None),
                                        ("c3_decode_skewed", None), ("c4_decode_fp8", None),
                                        ("c5_prefill", "tiles"), ("c8_prefill_fp8", "tiles")])
def test_forward_reference_workloads(M, cfg, sample):
    """The reference workloads at full size in the bench's launch
    configuration: decode on every token, prefill on tokens that reach every
    (expert, 128-row token tile) of the FC1 and FC2 tiles."""
    inp = workloads.make_inputs(cfg, DEV)
    m, ntok = check_forward(M, inp, sample=sample, name=cfg)
    if cfg in ("c1_tiny", "c2_decode_balanced", "c4_decode_fp8"):
        # the same workload in one cooperative launch
        os.environ["MOE_MEGA"] = "1"
        check_forward(M, inp, sample=sample, name=cfg + " one-launch")
        os.environ.pop("MOE_MEGA", None)
    if cfg in ("c2_decode_balanced", "c3_decode_skewed", "c4_decode_fp8"):
        # the fused and the two-launch FFN give identical bits
        fp8w = quantize_weights_gpu(M, inp) if inp["fp8"] else None
        o1, i1, _ = _run_forward(M, inp, fp8_weights=fp8w)
        os.environ["MOE_FUSE"] = "0"
        o2, i2, _ = _run_forward(M, inp, fp8_weights=fp8w)
        os.environ.pop("MOE_FUSE", None)
        assert torch.equal(i1, i2) and torch.equal(o1, o2)
        if cfg != "c3_decode_skewed":
            # one-launch forward: the routing (given logits) is the same, the
            # outputs agree to a few bf16 ulps (x_hat's sum of squares is
            # reduced in another order)
            os.environ["MOE_MEGA"] = "1"
            o3, i3, _ = _run_forward(M, inp, fp8_weights=fp8w)
            os.environ.pop("MOE_MEGA", None)
            assert torch.equal(i1, i3)
            assert_close(f64(o3), f64(o1), TOL_FP8 if inp["fp8"] else TOL_BF16, "one-launch")
    print(f"{cfg}: max scaled error {m:.3e} over {ntok} tokens")
    del inp
    torch.cuda.empty_cache()


def test_launch_counter_counts_the_forward(M):
    """The forward of the tiny workload enqueues the same number of kernels
    every call: rms_norm, router + top-k, permute, gather, fused FFN, combine."""
    inp = workloads.make_inputs("c1_tiny", DEV)
    _run_forward(M, inp)
    n0 = M.lib.moe_launch_count()
    _run_forward(M, inp)
    n1 = M.lib.moe_launch_count()
    _run_forward(M, inp)
    n2 = M.lib.moe_launch_count()
    assert n1 - n0 == n2 - n1 == 6


def test_forward_is_deterministic(M):
    inp = workloads.make_inputs("c1_tiny", DEV, shape=SMALL["ragged_b"], seed=3)
    o1, i1, w1 = _run_forward(M, inp)
    o2, i2, w2 = _run_forward(M, inp)
    assert torch.equal(o1, o2) and torch.equal(i1, i2) and torch.equal(w1, w2)


def test_forward_routed_matches_forward(M):
    inp = workloads.make_inputs("c1_tiny", DEV, shape=SMALL["ragged_a"], seed=4)
    out, ids, tw = _run_forward(M, inp)
    T, H, E, k, I = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"]
    shape = M.make_shape(T, H, E, I, k, inp["eps"])
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    out2 = torch.empty_like(out)
    M.moe_ffn_forward_routed(shape, inp["x"], inp["norm_w"], ids, tw, inp["w13"], inp["w2"], out2, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_forward_all_tokens_one_expert_and_empty_experts(M):
    T, H, E, k, I = 70, 256, 8, 1, 192
    inp = workloads.make_inputs("c1_tiny", DEV, shape=workloads.Shape(T, H, E, k, I), seed=9)
    ids = torch.full((T, k), 5, dtype=torch.int32, device=DEV)
    tw = torch.ones((T, k), dtype=torch.float32, device=DEV)
    shape = M.make_shape(T, H, E, I, k)
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    M.moe_ffn_forward_routed(shape, inp["x"], inp["norm_w"], ids, tw, inp["w13"], inp["w2"], out, ws)
    torch.cuda.synchronize()
    xhat = O.rms_norm(f64(inp["x"]), f64(inp["norm_w"]), 1e-6)
    ref = O.ffn_token_outputs(xhat, ids.cpu().numpy(), np.ones((T, k)), lambda e: f64(inp["w13"][e]),
                              lambda e: f64(inp["w2"][e]), I)
    assert_close(f64(out), ref, TOL_BF16, "one expert")


def test_forward_routed_invalid_ids_dropped(M):
    """Caller routing with an expert id outside [0, E): the pair is dropped
    and MOE_ERR_INVALID_ARG recorded, in the one-launch forward and in the
    separate launches alike."""
    T, H, E, k, I = 6, 256, 8, 2, 128
    inp = workloads.make_inputs("c1_tiny", DEV, shape=workloads.Shape(T, H, E, k, I), seed=11)
    ids = torch.tensor([[0, 1], [2, 9], [3, 4], [-1, 5], [6, 7], [1, 2]], dtype=torch.int32, device=DEV)
    tw = torch.full((T, k), 0.5, dtype=torch.float32, device=DEV)
    shape = M.make_shape(T, H, E, I, k)
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), DEV)
    outs = []
    for mega in ("1", "0"):
        os.environ["MOE_MEGA"] = mega
        M.device_status(clear=True)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        M.moe_ffn_forward_routed(shape, inp["x"], inp["norm_w"], ids, tw, inp["w13"], inp["w2"], out, ws)
        torch.cuda.synchronize()
        assert M.device_status(clear=True) == 1      # MOE_ERR_INVALID_ARG
        outs.append(f64(out))
    os.environ.pop("MOE_MEGA", None)
    xhat = O.rms_norm(f64(inp["x"]), f64(inp["norm_w"]), 1e-6)
    idn = ids.cpu().numpy()
    wn = np.where((idn >= 0) & (idn < E), 0.5, 0.0)
    ids_ok = np.where((idn >= 0) & (idn < E), idn, 0)
    ref = O.ffn_token_outputs(xhat, ids_ok, wn, lambda e: f64(inp["w13"][e]),
                              lambda e: f64(inp["w2"][e]), I)
    for o in outs:
        assert_close(o, ref, TOL_BF16, "invalid ids dropped")


def test_forward_zero_tokens(M):
    shape = M.make_shape(0, 256, 8, 128, 2)
    ws = M.alloc_workspace(max(1, M.moe_ffn_workspace_size(shape)), DEV)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    w = torch.ones((256,), dtype=torch.bfloat16, device=DEV)
    w13 = torch.zeros((8, 256, 256), dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros((8, 256, 128), dtype=torch.bfloat16, device=DEV)
    rw = torch.zeros((256, 8), dtype=torch.float32, device=DEV)
    out = torch.empty((1, 256), dtype=torch.bfloat16, device=DEV)
    M.moe_ffn_forward(shape, x if x.numel() else w, w, w13, w2, out, ws, router_w=rw)
    torch.cuda.synchronize()


def test_identity_experts_on_gpu(M):
    """Closed form on the GPU: W_gate = W_up = [I_H; 0], W2 = [I_H, 0] for all
    experts gives out = bf16(x_hat^2 * sigmoid(x_hat)) whatever the routing."""
    T, H, E, k, I = 33, 128, 4, 2, 192
    inp = workloads.make_inputs("c1_tiny", DEV, shape=workloads.Shape(T, H, E, k, I), seed=5)
    eye = torch.zeros((I, H), device=DEV)
    eye[:H, :H] = torch.eye(H, device=DEV)
    inp["w13"] = torch.cat([eye, eye]).to(torch.bfloat16).unsqueeze(0).repeat(E, 1, 1).contiguous()
    inp["w2"] = eye.t().contiguous().to(torch.bfloat16).unsqueeze(0).repeat(E, 1, 1).contiguous()
    out, _, _ = _run_forward(M, inp)
    xhat = torch.empty_like(inp["x"])
    M.moe_rmsnorm(inp["x"], inp["norm_w"], 1e-6, xhat)
    xh = f64(xhat)
    import scipy.special
    expect = O.bf16_round(O.bf16_round(xh * xh * scipy.special.expit(xh)))
    err = scaled_err(f64(out), expect)
    assert err.max() <= 1e-2


def test_bounded_wait_times_out_and_context_survives(M):
    """A device wait that nothing completes gives up after its limit, records
    MOE_ERR_TIMEOUT in the status word, and the context keeps working."""
    import time
    M.device_status(clear=True)
    t0 = time.perf_counter()
    M.moe_selftest_wait_timeout(20_000_000)        # ~10 ms of SM cycles
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert M.device_status(clear=True) == 6        # MOE_ERR_TIMEOUT
    inp = workloads.make_inputs("c1_tiny", DEV)
    out, ids, _ = _run_forward(M, inp)
    assert torch.isfinite(out.float()).all()
    assert M.device_status() == 0

