"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself (closed forms, format definitions, library special cases,
invariants, brute force on tiny inputs).  CPU only."""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O
import workloads


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def test_bf16_round_hand_cases():
    # 1 + 2^-8 is exactly half-way between 1 and 1 + 2^-7: ties to even -> 1.
    assert O.bf16_round(1 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 is half-way between 1+2^-7 (odd) and 1+2^-6 (even) -> up.
    assert O.bf16_round(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    # just above the half-way point rounds up
    assert O.bf16_round(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    assert O.bf16_round(-(1 + 2.0 ** -8 + 2.0 ** -30)) == -(1 + 2.0 ** -7)
    assert O.bf16_round(0.0) == 0.0
    # smallest bf16 subnormal is 2^-133; half of it ties to even (0)
    assert O.bf16_round(2.0 ** -133) == 2.0 ** -133
    assert O.bf16_round(2.0 ** -134) == 0.0
    assert O.bf16_round(3 * 2.0 ** -134) == 2.0 ** -132


def test_bf16_round_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(0)
    mant = rng.integers(0, 2 ** 23, size=200000)
    expo = rng.integers(-140, 120, size=200000)
    sign = rng.choice([-1.0, 1.0], size=200000)
    vals = sign * np.ldexp(1.0 + mant / 2.0 ** 23, expo)
    vals = vals.astype(np.float32)
    # include exact ties: force the low 16 bits of finite values to 0x8000
    ties = (vals[:1000].view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    vals = np.concatenate([vals, ties.view(np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(vals.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------

def test_e4m3_code_table_roundtrip_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    vals = np.array([O.e4m3_decode(int(c)) for c in codes])
    finite = ~np.isnan(vals)
    assert finite.sum() == 254                    # 0x7F and 0xFF are NaN
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9       # smallest subnormal
    assert O.e4m3_decode(0x08) == 2.0 ** -6       # smallest normal
    # every finite code round-trips through the rounding function
    np.testing.assert_array_equal(O.e4m3_round(vals[finite]), vals[finite])
    # and torch's float8_e4m3fn agrees on the value of each byte
    tv = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(tv[finite], vals[finite])


def test_e4m3_midpoints_ties_to_even_and_saturation():
    pos = sorted(set(O.e4m3_decode(c) for c in range(0x00, 0x7F)))
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = 0.5 * (lo + hi)
        got = O.e4m3_round(mid)
        # the even neighbour is the one whose code has mantissa LSB 0
        lo_code = [c for c in range(0x7F) if O.e4m3_decode(c) == lo][0]
        expect = lo if lo_code % 2 == 0 else hi
        assert got == expect, (lo, hi, got)
        assert O.e4m3_round(-mid) == -expect
    assert O.e4m3_round(449.0) == 448.0
    assert O.e4m3_round(1e9) == 448.0
    assert O.e4m3_round(-1e9) == -448.0


def test_e4m3_matches_torch_in_range():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(100000) * rng.choice([1e-3, 0.1, 10, 100], 100000)).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.e4m3_round(v.astype(np.float64)), ref)


def test_quantize_rows_matches_torch_recipe_and_zero_row():
    rng = np.random.default_rng(2)
    w = torch.from_numpy((rng.standard_normal((37, 300)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    w[5] = 0
    q, s = O.quantize_rows_e4m3(w.to(torch.float64).numpy())
    wf = w.float()
    amax = wf.abs().amax(dim=1)
    ts = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    tq = (wf / ts[:, None]).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(q, tq)
    np.testing.assert_array_equal(s, ts.double().numpy())
    assert s[5] == 1.0 and np.all(q[5] == 0)
    # each non-zero row reaches +-448 at its absmax
    assert np.all(np.abs(q[np.arange(37) != 5]).max(axis=1) == 448.0)


E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_brute(x):
    """Nearest of the 15 E2M1 values by exhaustive search; on an exact tie
    the value whose code has mantissa bit 0 (1.0, 2.0, 4.0 or 0); beyond 6
    the largest magnitude."""
    mags = E2M1_GRID
    a = abs(x)
    if a >= 6.0:
        return math.copysign(6.0, x)
    best = min(mags, key=lambda m: (abs(a - m), 0 if mags.index(m) % 2 == 0 else 1))
    return math.copysign(best, x) if best != 0 else 0.0


def test_e2m1_rounding_brute_force():
    rng = np.random.default_rng(21)
    xs = np.concatenate([rng.uniform(-8, 8, 4000),
                         [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, -6.0]])
    got = O.e2m1_round(xs)
    for x, g in zip(xs, got):
        assert g == _e2m1_brute(x) or (g == 0 and _e2m1_brute(x) == 0), (x, g)
    # every code value round-trips
    vals = np.array([O.e2m1_decode(c) for c in range(16)])
    np.testing.assert_array_equal(O.e2m1_round(vals), vals)


def test_nvfp4_constructed_weights_round_trip():
    """Weights built as q * s_b * s_g with a +-6 in every block are recovered
    exactly: the block ratio amax_b / (6 s_g) is s_b itself and every element
    quotient is its code."""
    rng = np.random.default_rng(22)
    n, kdim = 12, 64
    sg = 2.0 ** -12
    grid = np.array(E2M1_GRID[1:] + [-v for v in E2M1_GRID[1:]])
    q = rng.choice(grid, (n, kdim))
    q = q.reshape(n, kdim // 16, 16)
    q[:, :, 3] = 6.0                                  # the block maximum
    e4m3_vals = np.array([O.e4m3_decode(c) for c in range(0x08, 0x7F)])  # positive normals
    sb = rng.choice(e4m3_vals, (n, kdim // 16))
    sb[0, 0] = 448.0                                  # the matrix maximum: 6 * 448 * s_g
    w = (q * sb[..., None] * sg).reshape(n, kdim)
    q2, sb2, sg2 = O.quantize_nvfp4(w)
    assert sg2 == sg
    np.testing.assert_array_equal(sb2, sb)
    np.testing.assert_array_equal(q2, q.reshape(n, kdim))
    np.testing.assert_array_equal(O.dequantize_nvfp4(q2, sb2, sg2), w)


def test_nvfp4_recipe_closed_forms_and_nearest_codes():
    rng = np.random.default_rng(23)
    w = (rng.standard_normal((9, 96)) * 0.02).astype(np.float32).astype(np.float64)
    w[4, 16:32] = 0.0                                 # an all-zero block
    q, sb, sg = O.quantize_nvfp4(w)
    amax = np.abs(w).max()
    assert sg == float(np.float32(np.float32(amax) / np.float32(2688.0)))
    i, j = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert sb[i, j // 16] == 448.0 and abs(q[i, j]) == 6.0   # amax maps to 6 * 448 * s_g
    assert np.all(sb[4, 1] == 0) and np.all(q[4, 16:32] == 0)
    # each code is the E2M1 value nearest the fp32 quotient w / (s_b s_g)
    scale = np.repeat((sb.astype(np.float32) * np.float32(sg)).astype(np.float32), 16, axis=1)
    ok = scale > 0
    quot = (w.astype(np.float32) / np.where(ok, scale, 1)).astype(np.float32).astype(np.float64)
    for x, g in zip(quot[ok], q[ok]):
        assert g == _e2m1_brute(x) or (g == 0 and _e2m1_brute(x) == 0)
    # block scales: e4m3 of amax_block / (6 s_g), decided in fp32
    ab = np.abs(w).reshape(9, 6, 16).max(axis=-1).astype(np.float32)
    six_sg = np.float32(np.float32(6.0) * np.float32(sg))
    np.testing.assert_array_equal(sb, O.e4m3_round((ab / six_sg).astype(np.float32).astype(np.float64)))
    # zero matrix
    qz, sbz, sgz = O.quantize_nvfp4(np.zeros((2, 32)))
    assert sgz == 1.0 and np.all(sbz == 0) and np.all(qz == 0)


def test_nvfp4_dequantised_error_bound():
    """|w - w_hat| <= half an E2M1 spacing at |w|'s magnitude times the block
    scale, for blocks whose rounded scale does not clip the block maximum."""
    rng = np.random.default_rng(24)
    w = (rng.standard_normal((16, 128)) * 0.05).astype(np.float32).astype(np.float64)
    q, sb, sg = O.quantize_nvfp4(w)
    wh = O.dequantize_nvfp4(q, sb, sg)
    scale = np.repeat(sb * sg, 16, axis=1)
    r = np.abs(w) / scale
    spacing = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    bound = np.where(r <= 6, 0.5 * spacing * scale, np.abs(w) - 6 * scale) * (1 + 1e-6)
    assert np.all(np.abs(w - wh) <= bound + 1e-30)


def test_fp8_gemm_equals_bf16_gemm_on_representable_inputs():
    """With E4M3-representable values and power-of-two scales the W8A8 FC1
    equals the plain FC1 exactly (pins where each scale is applied)."""
    rng = np.random.default_rng(3)
    grid = np.array(sorted(set(O.e4m3_decode(c) for c in range(0x7F))))
    grid = np.concatenate([-grid[1:], grid])
    H, I, rows = 64, 32, 5

    def rep(shape, p):
        m = rng.choice(grid, size=shape)
        m[..., 0] = 448.0                       # absmax 448 -> scale exactly 2^p
        return m * 2.0 ** p
    x = rep((rows, H), -7)
    w13 = rep((2 * I, H), -12)
    offsets = np.array([0, rows])
    xq, sx = O.quantize_rows_e4m3(x)
    assert np.all(sx == 2.0 ** -7)
    q13, s13 = O.quantize_rows_e4m3(w13)
    assert np.all(s13 == 2.0 ** -12)
    a8 = O.grouped_fc1_fp8(xq, sx, offsets, lambda e: q13, lambda e: s13, I)
    a16 = O.grouped_fc1(x, offsets, lambda e: w13, I)
    np.testing.assert_array_equal(a8, a16)
    w2 = rep((H, I), -11)
    rw = rng.random(rows)
    q2, s2 = O.quantize_rows_e4m3(w2)
    aq, sa = O.quantize_rows_e4m3(a16)
    # FC2's activations are re-quantised per row; compare against the plain
    # FC2 applied to those dequantised rows.
    y8 = O.grouped_fc2_fp8(a16, offsets, lambda e: q2, lambda e: s2, rw)
    y16 = O.grouped_fc2(aq * sa[:, None], offsets, lambda e: w2, rw)
    np.testing.assert_allclose(y8, y16, rtol=1e-13, atol=0)


def _rep_rows(rng, shape, exps):
    """Rows of E4M3 values, each row scaled by its own power of two 2^exps[r]
    and holding one element of magnitude 448 (so its absmax/448 scale is
    exactly 2^exps[r])."""
    grid = np.array(sorted(set(O.e4m3_decode(c) for c in range(0x7F))))
    grid = np.concatenate([-grid[1:], grid])
    m = rng.choice(grid, size=shape)
    m[np.arange(shape[0]), rng.integers(0, shape[1], shape[0])] = 448.0
    return m * np.ldexp(1.0, np.asarray(exps))[:, None]


def test_fp8_per_channel_scales_pin_their_axes():
    """The W8A8 scales belong to different axes: one per token row of the
    activations (s_a) and one per output channel of the weights (s_w); the
    SM-architecture article's scaled GEMM c = (a*s_a)(b*s_b).  With a
    different power of two on every row and every output channel, the FP8
    FC1 and FC2 equal the bf16 ones exactly only if each scale multiplies its
    own axis: a transposed or shifted scale vector fails."""
    rng = np.random.default_rng(33)
    H, I, E, rows = 64, 48, 2, 7
    offsets = np.array([0, 3, rows])
    x = _rep_rows(rng, (rows, H), rng.integers(-9, -4, rows))
    w13 = [_rep_rows(rng, (2 * I, H), rng.integers(-14, -9, 2 * I)) for _ in range(E)]
    w2 = [_rep_rows(rng, (H, I), rng.integers(-13, -8, H)) for _ in range(E)]
    xq, sx = O.quantize_rows_e4m3(x)
    q13 = [O.quantize_rows_e4m3(w) for w in w13]
    q2 = [O.quantize_rows_e4m3(w) for w in w2]
    assert len(set(sx.tolist())) > 1 and len(set(q13[0][1].tolist())) > 1
    a8 = O.grouped_fc1_fp8(xq, sx, offsets, lambda e: q13[e][0], lambda e: q13[e][1], I)
    a16 = O.grouped_fc1(x, offsets, lambda e: w13[e], I)
    np.testing.assert_array_equal(a8, a16)
    rw = rng.random(rows)
    aq, sa = O.quantize_rows_e4m3(a16)
    y8 = O.grouped_fc2_fp8(a16, offsets, lambda e: q2[e][0], lambda e: q2[e][1], rw)
    y16 = O.grouped_fc2(aq * sa[:, None], offsets, lambda e: w2[e], rw)
    np.testing.assert_allclose(y8, y16, rtol=1e-13, atol=0)
    # a planted mistake: the FC2 channel scales reversed
    y_bad = O.grouped_fc2_fp8(a16, offsets, lambda e: q2[e][0], lambda e: q2[e][1][::-1], rw)
    assert not np.allclose(y_bad, y16, rtol=1e-6, atol=0)


def test_fp8_forward_token_definition_matches_grouped_form():
    """ffn_token_outputs(fp8=True), the per-token definition the sampled GPU
    checks of the W8A8 workloads use, equals the grouped W8A8 forward on the
    tiny workload: all columns and a column subset (whose channel scales must
    follow the columns)."""
    inp = workloads.make_inputs("c1_tiny", "cpu")
    x = inp["x"].double().numpy()
    nw = inp["norm_w"].double().numpy()
    Wr = inp["router_w"].double().numpy()
    w13 = inp["w13"].double().numpy()
    w2 = inp["w2"].double().numpy()
    res = O.moe_ffn_forward(x, nw, 1e-6, 2, w13, w2, router_w=Wr, fp8=True)
    q13 = {e: O.quantize_rows_e4m3(w13[e]) for e in range(8)}
    q2 = {e: O.quantize_rows_e4m3(w2[e]) for e in range(8)}
    assert len(set(q2[0][1].tolist())) > 30             # the channel scales differ
    direct = O.ffn_token_outputs(res["xhat"], res["ids"], res["topk_w"], None, None, 512,
                                 fp8=True, wq13_of=q13.get, wq2_of=q2.get)
    np.testing.assert_array_equal(direct, res["out"])
    cols = np.array([0, 5, 77, 128, 255])
    direct_c = O.ffn_token_outputs(res["xhat"], res["ids"], res["topk_w"], None, None, 512,
                                   cols=cols, fp8=True, wq13_of=q13.get, wq2_of=q2.get)
    np.testing.assert_array_equal(direct_c, res["out"][:, cols])
    # a planted mistake: the column subset taken with the scales of other columns
    bad2 = {e: (q2[e][0], np.roll(q2[e][1], 1)) for e in range(8)}
    bad_c = O.ffn_token_outputs(res["xhat"], res["ids"], res["topk_w"], None, None, 512,
                                cols=cols, fp8=True, wq13_of=q13.get, wq2_of=bad2.get)
    assert not np.array_equal(bad_c, res["out"][:, cols])
    # W8A8 stays close to the bf16 forward (E4M3 carries 3 mantissa bits)
    ref = O.moe_ffn_forward(x, nw, 1e-6, 2, w13, w2, router_w=Wr)["out"]
    assert np.max(np.abs(res["out"] - ref)) < 6e-2 * max(1.0, np.max(np.abs(ref)))


# ---------------------------------------------------------------------------
# block-wise FP8 (128 x 128 weight tiles, 1 x 128 activation groups)
# ---------------------------------------------------------------------------

E4M3_NORMALS = np.array(sorted(set(O.e4m3_decode(c) for c in range(0x08, 0x7F))))


def _tiled(rng, n, kdim, bn, scales, bk=128):
    """A matrix whose (bn x bk) tile (i, g) is scales[i, g] times E4M3 normals
    with one element of magnitude 448 (so the tile's scale is scales[i, g])."""
    q = rng.choice(E4M3_NORMALS, (n, kdim)) * rng.choice([-1.0, 1.0], (n, kdim))
    for i in range(n // bn):
        for g in range(kdim // bk):
            r, c = rng.integers(bn), rng.integers(bk)
            q[i * bn + r, g * bk + c] = 448.0 * rng.choice([-1.0, 1.0])
    return q, q * np.repeat(np.repeat(scales, bn, axis=0), bk, axis=1)


def test_fp8_block_quantise_constructed_round_trip():
    """Tiles built as (E4M3 codes) x (scale with few significant bits) come
    back exactly, each scale at its own (row block, K group): pins the tile
    indexing and the absmax/448 scale."""
    rng = np.random.default_rng(40)
    sw = np.array([[1.5, 0.75, 2.0 ** -9], [1.25 * 2.0 ** -6, 3.0, 1.0]]) * 2.0 ** -8
    q, w = _tiled(rng, 256, 384, 128, sw)
    q2, s2 = O.quantize_blocks_e4m3(w, 128)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(s2, sw)
    # activation groups: one scale per (row, 128 K elements)
    sa = rng.choice([0.5, 1.0, 1.5, 0.125, 1.75], (5, 3)) * 2.0 ** -5
    qa, a = _tiled(rng, 5, 384, 1, sa)
    qa2, sa2 = O.quantize_blocks_e4m3(a, 1)
    np.testing.assert_array_equal(qa2, qa)
    np.testing.assert_array_equal(sa2, sa)


def test_fp8_block_quantise_special_cases():
    rng = np.random.default_rng(41)
    w = torch.from_numpy((rng.standard_normal((256, 256)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    w64 = w.to(torch.float64).numpy()
    # one K group and one row per block: the per-row recipe (pinned against torch)
    q1, s1 = O.quantize_blocks_e4m3(w64[:, :128], 1)
    qr, sr = O.quantize_rows_e4m3(w64[:, :128])
    np.testing.assert_array_equal(q1, qr)
    np.testing.assert_array_equal(s1[:, 0], sr)
    # torch's float8_e4m3fn on each tile, tile by tile
    q, s = O.quantize_blocks_e4m3(w64, 128)
    for i in range(2):
        for g in range(2):
            t = w[i * 128:(i + 1) * 128, g * 128:(g + 1) * 128].float()
            ts = t.abs().max() / 448.0
            assert s[i, g] == ts.item()
            tq = (t / ts).to(torch.float8_e4m3fn).to(torch.float64).numpy()
            np.testing.assert_array_equal(q[i * 128:(i + 1) * 128, g * 128:(g + 1) * 128], tq)
    # an all-zero tile: scale 1, codes 0; the other tiles are untouched
    w0 = w64.copy()
    w0[128:, :128] = 0
    qz, sz = O.quantize_blocks_e4m3(w0, 128)
    assert sz[1, 0] == 1.0 and np.all(qz[128:, :128] == 0)
    np.testing.assert_array_equal(sz[0], s[0])


def test_block_scaled_matmul_exact_on_representable_inputs():
    """With tiles that quantise exactly, the block-scaled product equals the
    plain fp64 product x @ w^T exactly (all partial sums are exact in fp64):
    a swapped scale index or a dropped scale fails it."""
    rng = np.random.default_rng(42)
    sw = rng.choice([1.0, 2.0, 0.5, 4.0, 0.25], (2, 3)) * 2.0 ** -10
    sa = rng.choice([1.0, 2.0, 0.5, 0.125], (6, 3)) * 2.0 ** -4
    qw, w = _tiled(rng, 256, 384, 128, sw)
    qa, a = _tiled(rng, 6, 384, 1, sa)
    y = O.block_scaled_matmul(qa, sa, qw, sw)
    np.testing.assert_array_equal(y, a @ w.T)
    # the same through the quantiser
    aq, as_ = O.quantize_blocks_e4m3(a, 1)
    wq, ws = O.quantize_blocks_e4m3(w, 128)
    np.testing.assert_array_equal(O.block_scaled_matmul(aq, as_, wq, ws), a @ w.T)


def test_block_scaled_matmul_error_bound():
    """E4M3 round to nearest: |v - v~| <= 2^-4 |v| + 2^-10 s per element (half
    a normal quantum relative, half the subnormal quantum 2^-9 s absolute), so
    |y - x w^T| <= sum_k |dx| |w~| + |x| |dw|."""
    rng = np.random.default_rng(43)
    x = rng.standard_normal((7, 256)) * np.repeat(rng.choice([0.1, 1.0, 10.0], (7, 2)), 128, axis=1)
    w = rng.standard_normal((256, 256)) * 0.02
    x = x.astype(np.float32).astype(np.float64)
    w = w.astype(np.float32).astype(np.float64)
    xq, sx = O.quantize_blocks_e4m3(x, 1)
    wq, sw = O.quantize_blocks_e4m3(w, 128)
    y = O.block_scaled_matmul(xq, sx, wq, sw)
    xt = xq * np.repeat(sx, 128, axis=1)
    wt = wq * np.repeat(np.repeat(sw, 128, axis=0), 128, axis=1)
    dx = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * np.repeat(sx, 128, axis=1)
    dw = 2.0 ** -4 * np.abs(w) + 2.0 ** -10 * np.repeat(np.repeat(sw, 128, axis=0), 128, axis=1)
    assert np.all(np.abs(xt - x) <= dx) and np.all(np.abs(wt - w) <= dw)
    bound = dx @ np.abs(wt).T + np.abs(x) @ dw.T
    assert np.all(np.abs(y - x @ w.T) <= bound * (1 + 1e-12))
    # and the bound is not vacuous: the error is well below the plain magnitude
    assert np.max(np.abs(y - x @ w.T)) < 0.2 * np.max(np.abs(x @ w.T))


def test_fp8_block_ffn_equals_bf16_ffn_on_representable_inputs():
    """FC1 and FC2 with block-wise FP8 equal the plain FC1/FC2 when the
    activations and weights quantise exactly (FC2 compared on the re-quantised
    FC1 output, the input the block-wise FC2 sees)."""
    rng = np.random.default_rng(44)
    H, I, rows = 256, 256, 5
    s13 = rng.choice([1.0, 2.0, 0.5], (4, 2)) * 2.0 ** -12
    q13, w13 = _tiled(rng, 2 * I, H, 128, s13)
    sx = rng.choice([1.0, 0.5, 2.0], (rows, 2)) * 2.0 ** -6
    qx, x = _tiled(rng, rows, H, 1, sx)
    offsets = np.array([0, rows])
    a8 = O.grouped_fc1_fp8_block(qx, sx, offsets, lambda e: q13, lambda e: s13, I)
    a16 = O.grouped_fc1(x, offsets, lambda e: w13, I)
    np.testing.assert_array_equal(a8, a16)
    s2 = rng.choice([1.0, 2.0, 0.25], (2, 2)) * 2.0 ** -11
    q2, w2 = _tiled(rng, H, I, 128, s2)
    rw = rng.random(rows)
    aq, sa = O.quantize_blocks_e4m3(a16, 1)
    y8 = O.grouped_fc2_fp8_block(a16, offsets, lambda e: q2, lambda e: s2, rw)
    y16 = O.grouped_fc2(aq * np.repeat(sa, 128, axis=1), offsets, lambda e: w2, rw)
    np.testing.assert_allclose(y8, y16, rtol=1e-13, atol=0)


def test_fp8_block_forward_token_definition_matches_grouped_form():
    inp = workloads.make_inputs("c1_tiny", "cpu")
    x = inp["x"].double().numpy()
    nw = inp["norm_w"].double().numpy()
    Wr = inp["router_w"].double().numpy()
    w13 = inp["w13"].double().numpy()
    w2 = inp["w2"].double().numpy()
    res = O.moe_ffn_forward(x, nw, 1e-6, 2, w13, w2, router_w=Wr, fp8="block")
    b13 = {e: O.quantize_blocks_e4m3(w13[e], 128) for e in range(8)}
    b2 = {e: O.quantize_blocks_e4m3(w2[e], 128) for e in range(8)}
    direct = O.ffn_token_outputs(res["xhat"], res["ids"], res["topk_w"], None, None, 512,
                                 fp8="block", wq13_of=b13.get, wq2_of=b2.get)
    np.testing.assert_array_equal(direct, res["out"])
    cols = np.array([0, 127, 128, 200])
    direct_c = O.ffn_token_outputs(res["xhat"], res["ids"], res["topk_w"], None, None, 512,
                                   cols=cols, fp8="block", wq13_of=b13.get, wq2_of=b2.get)
    np.testing.assert_array_equal(direct_c, res["out"][:, cols])
    # block-wise FP8 stays close to the bf16 forward (E4M3 carries 3 mantissa bits)
    ref = O.moe_ffn_forward(x, nw, 1e-6, 2, w13, w2, router_w=Wr)["out"]
    assert np.max(np.abs(res["out"] - ref)) < 6e-2 * max(1.0, np.max(np.abs(ref)))


# ---------------------------------------------------------------------------
# silu / rms_norm
# ---------------------------------------------------------------------------

def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    assert O.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    z = np.linspace(-20, 20, 401)
    np.testing.assert_allclose(O.silu(-z), O.silu(z) - z, atol=1e-12)
    np.testing.assert_allclose(O.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    assert O.silu(60.0) == pytest.approx(60.0, rel=1e-20)
    big_neg = O.silu(-1000.0)
    assert big_neg == 0.0 and not np.isnan(big_neg)


def test_silu_and_mul_halves():
    h = np.array([[1.0, 2.0, 3.0, 4.0]])
    a = O.silu_and_mul(h, 2)
    expect = O.bf16_round(np.array([[1.0 * scipy.special.expit(1.0) * 3.0,
                                     2.0 * scipy.special.expit(2.0) * 4.0]]))
    np.testing.assert_array_equal(a, expect)


def test_rms_norm_constant_vector_and_eps_placement():
    # c*1 with w=1 -> c/sqrt(c^2+eps); c=1e-3, eps=1e-6 gives 1/sqrt(2)
    x = np.full((1, 64), 1e-3)
    y = O.rms_norm(x, np.ones(64), 1e-6)
    assert np.all(y == 0.70703125)              # bf16(1/sqrt(2)) = 1.0110101b * 2^-1
    # a large constant is ~1
    y = O.rms_norm(np.full((1, 8), 3.0), np.ones(8), 1e-6)
    assert np.all(y == 1.0)


def test_rms_norm_weight_linear_and_mean_not_sum():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 128))
    w = O.bf16_round(1 + 0.1 * rng.standard_normal(128))
    y1 = O.rms_norm(x, w, 1e-6)
    y2 = O.rms_norm(x, 2 * w, 1e-6)
    np.testing.assert_array_equal(y2, 2 * y1)
    # duplicating the row keeps mean(x^2) -> same output (a sum would change it)
    y3 = O.rms_norm(np.concatenate([x, x], axis=1), np.concatenate([w, w]), 1e-6)
    np.testing.assert_array_equal(y3[:, :128], y1)


def test_rms_norm_matches_torch_fused_op():
    """The fused library op equals the pow->mean->rsqrt->mul composite (the
    check the V100 article reports with max_abs_diff == 0)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 512))
    w = 1 + 0.1 * rng.standard_normal(512)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (512,), torch.from_numpy(w), eps=1e-6)
    ref = O.bf16_round(ref.numpy())
    got = O.rms_norm(x, w, 1e-6)
    diff = np.abs(got - ref)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(diff <= ulp)                  # at most a 1-ulp flip at a rounding tie
    assert np.mean(diff == 0) > 0.999


# ---------------------------------------------------------------------------
# router / softmax / top-k
# ---------------------------------------------------------------------------

def test_router_logits_brute_force():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 5))
    W = rng.standard_normal((5, 4))
    b = rng.standard_normal(4)
    got = O.router_logits(x, W, b)
    for t in range(3):
        for e in range(4):
            s = b[e]
            for h in range(5):
                s += x[t, h] * W[h, e]
            assert got[t, e] == pytest.approx(s, rel=1e-13)


def test_topk_invariants_and_full_softmax():
    rng = np.random.default_rng(7)
    l = rng.standard_normal((50, 16)) * 3
    for k in (1, 2, 5, 16):
        ids, w = O.topk_renorm(l, k)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
        assert np.all(np.diff(w, axis=1) <= 0)
        assert all(len(set(r)) == k for r in ids)
    ids, w = O.topk_renorm(l, 1)
    np.testing.assert_array_equal(ids[:, 0], np.argmax(l, axis=1))
    assert np.all(w == 1.0)
    ids, w = O.topk_renorm(l, 16)
    full = scipy.special.softmax(l, axis=1)
    np.testing.assert_allclose(np.take_along_axis(full, ids.astype(np.int64), 1), w, rtol=1e-13)


def test_topk_ties_lowest_index_first():
    l = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    ids, w = O.topk_renorm(l, 2)
    assert ids.tolist() == [[1, 2]]
    ids, w = O.topk_renorm(l, 3)
    assert ids.tolist() == [[1, 2, 4]]
    np.testing.assert_allclose(w, [[1 / 3, 1 / 3, 1 / 3]], rtol=1e-15)
    ids, _ = O.topk_renorm(np.zeros((1, 8)), 4)
    assert ids.tolist() == [[0, 1, 2, 3]]


def test_topk_brute_force_tiny_config():
    """Tiny workload (E=8, k=2): enumerate all 28 pairs, take the pair with
    the largest probability mass (lexicographically smallest on ties)."""
    inp = workloads.make_inputs("c1_tiny", "cpu")
    xhat = O.rms_norm(inp["x"].double().numpy(), inp["norm_w"].double().numpy(), inp["eps"])
    l = O.router_logits(xhat, inp["router_w"].double().numpy())
    p = scipy.special.softmax(l, axis=1)
    ids, w = O.topk_renorm(l, 2)
    for t in range(l.shape[0]):
        best = None
        for pair in itertools.combinations(range(8), 2):
            m = p[t, pair[0]] + p[t, pair[1]]
            if best is None or m > best[0]:
                best = (m, pair)
        assert set(ids[t].tolist()) == set(best[1])
        assert p[t, ids[t, 0]] >= p[t, ids[t, 1]]
        assert w[t, 0] == pytest.approx(p[t, ids[t, 0]] / best[0], rel=1e-14)


def test_bias_moves_selection():
    l = np.zeros((2, 6))
    ids, w = O.topk_renorm(l + np.array([0, 0, 0, 0, 0, 5.0]), 2)
    assert ids[:, 0].tolist() == [5, 5]


# ---------------------------------------------------------------------------
# permute / combine
# ---------------------------------------------------------------------------

def test_permute_brute_force_and_invariants():
    rng = np.random.default_rng(8)
    for T, E, k in [(1, 4, 1), (7, 5, 3), (33, 16, 8), (64, 256, 8)]:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        offsets, row_src = O.permute(ids, E)
        assert offsets[0] == 0 and offsets[-1] == T * k
        assert np.all(np.diff(offsets) >= 0)
        assert sorted(row_src.tolist()) == list(range(T * k))
        pairs = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(k))
        assert row_src.tolist() == [t * k + j for (_, t, j) in pairs]
        for e in range(E):
            seg = row_src[offsets[e]:offsets[e + 1]]
            assert np.all(ids.reshape(-1)[seg] == e)


def test_combine_brute_force():
    rng = np.random.default_rng(9)
    T, k, H = 5, 3, 7
    Y = rng.standard_normal((T * k, H))
    row_src = rng.permutation(T * k).astype(np.int32)
    out = O.combine(Y, row_src, T, k)
    for t in range(T):
        s = np.zeros(H)
        for j in range(k):
            r = int(np.where(row_src == t * k + j)[0][0])
            s = s + Y[r]
        np.testing.assert_array_equal(out[t], O.bf16_round(s))


# ---------------------------------------------------------------------------
# whole FFN
# ---------------------------------------------------------------------------

def _ffn_loops(x, norm_w, eps, Wr, w13, w2, k):
    """Pure-Python loops for a tiny shape: an independent restatement of the
    per-token definition (no numpy matmul, no argsort)."""
    T, H = x.shape
    E = Wr.shape[1]
    I = w2.shape[2]
    out = np.zeros((T, H))
    for t in range(T):
        ms = sum(float(v) * float(v) for v in x[t]) / H
        xh = [float(O.bf16_round(x[t, i] / math.sqrt(ms + eps) * norm_w[i])) for i in range(H)]
        lg = [sum(xh[i] * Wr[i, e] for i in range(H)) for e in range(E)]
        chosen = []
        for _ in range(k):
            best = None
            for e in range(E):
                if e in chosen:
                    continue
                if best is None or lg[e] > lg[best]:
                    best = e
            chosen.append(best)
        m = max(lg)
        pe = [math.exp(lg[e] - m) for e in chosen]
        acc = [0.0] * H
        for j, e in enumerate(chosen):
            wj = pe[j] / sum(pe)
            a = []
            for n in range(I):
                g = sum(xh[i] * w13[e, n, i] for i in range(H))
                u = sum(xh[i] * w13[e, I + n, i] for i in range(H))
                a.append(float(O.bf16_round(g / (1 + math.exp(-g)) * u)))
            for h in range(H):
                acc[h] += wj * sum(a[n] * w2[e, h, n] for n in range(I))
        out[t] = O.bf16_round(np.array(acc))
    return out


def test_ffn_matches_pure_python_loops():
    rng = np.random.default_rng(10)
    T, H, E, k, I = 3, 8, 4, 2, 6
    x = O.bf16_round(rng.standard_normal((T, H)))
    nw = O.bf16_round(1 + 0.1 * rng.standard_normal(H))
    Wr = rng.standard_normal((H, E)) * 0.5
    w13 = O.bf16_round(rng.standard_normal((E, 2 * I, H)) * 0.5)
    w2 = O.bf16_round(rng.standard_normal((E, H, I)) * 0.5)
    res = O.moe_ffn_forward(x, nw, 1e-6, k, w13, w2, router_w=Wr)
    ref = _ffn_loops(x, nw, 1e-6, Wr, w13, w2, k)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(res["out"] - ref) <= ulp)
    assert np.mean(res["out"] == ref) > 0.9


def test_identity_experts_reproduce_input_closed_form():
    """W_gate = W_up = [I_H; 0], W2 = [I_H, 0] for every expert gives
    out = bf16(x_hat^2 * sigmoid(x_hat)) elementwise, whatever the routing."""
    rng = np.random.default_rng(11)
    T, H, E, k, I = 6, 16, 4, 2, 24
    x = O.bf16_round(rng.standard_normal((T, H)))
    nw = O.bf16_round(1 + 0.1 * rng.standard_normal(H))
    eye = np.zeros((I, H))
    eye[:H, :H] = np.eye(H)
    w13 = np.stack([np.concatenate([eye, eye])] * E)
    w2 = np.stack([eye.T.copy()] * E)
    ref_xhat = O.bf16_round(torch.nn.functional.rms_norm(
        torch.from_numpy(x), (H,), torch.from_numpy(nw), eps=1e-6).numpy())
    expect = O.bf16_round(ref_xhat * ref_xhat * scipy.special.expit(ref_xhat))
    for seed in range(3):
        Wr = np.random.default_rng(seed).standard_normal((H, E))
        res = O.moe_ffn_forward(x, nw, 1e-6, k, w13, w2, router_w=Wr)
        np.testing.assert_array_equal(res["out"], expect)


def test_token_definition_matches_grouped_form():
    inp = workloads.make_inputs("c1_tiny", "cpu")
    x = inp["x"].double().numpy()
    nw = inp["norm_w"].double().numpy()
    Wr = inp["router_w"].double().numpy()
    w13 = inp["w13"].double().numpy()
    w2 = inp["w2"].double().numpy()
    res = O.moe_ffn_forward(x, nw, 1e-6, 2, w13, w2, router_w=Wr)
    direct = O.ffn_token_outputs(res["xhat"], res["ids"], res["topk_w"],
                                 lambda e: w13[e], lambda e: w2[e], 512)
    np.testing.assert_array_equal(direct, res["out"])
    cols = np.array([0, 5, 255])
    direct_c = O.ffn_token_outputs(res["xhat"], res["ids"], res["topk_w"],
                                   lambda e: w13[e], lambda e: w2[e], 512, cols=cols)
    np.testing.assert_array_equal(direct_c, res["out"][:, cols])


def test_balanced_routing_workload_is_balanced():
    inp = workloads.make_inputs("c2_decode_balanced", "cpu",
                                shape=workloads.Shape(T=16, H=64, E=64, k=8, I=64))
    _, ids, w = O.route(None, logits=inp["router_logits"].double().numpy(), k=8)
    offsets, _ = O.permute(ids, 64)
    assert np.all(np.diff(offsets) == 2)
    for t in range(16):
        assert sorted(ids[t].tolist()) == sorted(((8 * t + j) % 64) for j in range(8))
