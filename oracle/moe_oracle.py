"""CPU oracle for the MoE expert FFN forward (TEST INFRASTRUCTURE ONLY).

This module is the plain, slow, obviously correct definition the CUDA path is
checked against.  Only the test-suite, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import it; the product library never calls it
and shares no code with it.

Arithmetic: fp64 (numpy float64) over inputs that hold bf16 / E4M3 values.
Library primitives used as steps: numpy ``@`` (fp64 matmul), ``argsort``,
``exp``.  No blocking, fusion or reordering beyond what each definition says.

Sources (web pages; titles and sections):
  [V100]  Qiita, "running the latest vLLM on a Tesla V100" (yoheier) --
          sections "2nd wall" (rms_norm / silu_and_mul are the custom ops of
          the FFN path) and "rewrite on torch::stable::Tensor" (rms_norm is
          the pow -> mean -> rsqrt -> mul composite; the fused op matched it
          with max_abs_diff == 0).
  [RUBIN] "vLLM Support for NVIDIA Vera Rubin NVL72" (Chinese summary) --
          section "Locality domain": at small token counts the MoE forward is
          FC1 then FC2 over expert weights read from HBM.
  [SM]    "vLLM's adaptation to different GPU SM architectures" --
          sections 3.1/3.2 (W8A8 scaled GEMM c = (a*s_a)(b*s_b), FP8 E4M3)
          and 4.3 (MoE experts take hidden_states, w1, w2).
The pages do not spell out top-k, renormalisation, permutation, combine, the
FFN formula or the FP8 scale recipe; where they are silent the plain standard
reading is used and named at each function.

Parity status: every function below is pinned by tests in
tests/test_oracle_pins.py and tests/test_golden.py (closed forms, invariants,
brute force, library special cases, hand-derived format tables).  NVFP4
(E2M1 elements, E4M3 block scales) follows the public format definition; the
pages name the format without defining it.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64

# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
E4M3_MAX = 448.0
E2M1_MAX = 6.0
NVFP4_BLOCK = 16


def bf16_round(a) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even).

    bfloat16 keeps 8 significant bits and fp32's exponent range; normal
    numbers |a| >= 2^-126 have quantum 2^(e-8) with a = m*2^e, 0.5<=|m|<1;
    below that the subnormal quantum is 2^-133.  Rounding is done once,
    directly from fp64 (no intermediate fp32 rounding)."""
    a = np.asarray(a, dtype=F64)
    _, e = np.frexp(a)
    q = np.where(e >= -125, e - 8, -133)
    return np.ldexp(np.rint(np.ldexp(a, -q)), q)


def e4m3_round(a) -> np.ndarray:
    """Round float64 values to OCP FP8 E4M3FN, nearest-even, saturating.

    E4M3FN: 4 exponent bits (bias 7), 3 mantissa bits, no infinity, largest
    finite 448 = 1.75*2^8, smallest normal 2^-6, subnormal quantum 2^-9.
    Values beyond +-448 saturate to +-448 (the 'satfinite' conversion)."""
    a = np.asarray(a, dtype=F64)
    _, e = np.frexp(a)
    q = np.where(e >= -5, e - 4, -9)
    r = np.ldexp(np.rint(np.ldexp(a, -q)), q)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def e4m3_decode(code: int) -> float:
    """Value of one E4M3FN byte (NaN for 0x7F / 0xFF), from the format layout."""
    s = -1.0 if code & 0x80 else 1.0
    ex = (code >> 3) & 0xF
    m = code & 0x7
    if ex == 0xF and m == 0x7:
        return float("nan")
    if ex == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (ex - 7)


def e2m1_round(a) -> np.ndarray:
    """Round float64 values to FP4 E2M1, nearest-even, saturating to +-6.

    E2M1: 2 exponent bits (bias 1), 1 mantissa bit, no infinity or NaN:
    magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6.  With a = m*2^e,
    0.5 <= |m| < 1, a normal value (e >= 1) has quantum 2^(e-2); below 1 the
    subnormal quantum is 0.5.  Ties go to the even mantissa (np.rint), and
    values beyond +-6 saturate to +-6."""
    a = np.asarray(a, dtype=F64)
    _, e = np.frexp(a)
    q = np.where(e >= 1, e - 2, -1)
    r = np.ldexp(np.rint(np.ldexp(a, -q)), q)
    return np.clip(r, -E2M1_MAX, E2M1_MAX)


def e2m1_decode(code: int) -> float:
    """Value of one E2M1 nibble, from the format layout (sign, 2-bit exponent
    with bias 1, 1-bit mantissa; exponent 0 is subnormal)."""
    s = -1.0 if code & 0x8 else 1.0
    ex = (code >> 1) & 0x3
    m = code & 0x1
    if ex == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (ex - 1)


def f32(a) -> np.ndarray:
    """Round to IEEE fp32 (used only where fp32 decides an integer code)."""
    return np.asarray(a, dtype=np.float32)


def quantize_rows_e4m3(v: np.ndarray):
    """Per-row dynamic E4M3 quantisation: s = absmax/448, q = e4m3(v/s).

    [SM] 3.1/3.2: W8A8 scaled GEMM with E4M3 operands and per-row scales.
    Reading: the scale and the division are taken in fp32, the precision in
    which the code is decided on the GPU; a row of zeros gets s = 1, q = 0.
    Returns (q as float64 holding E4M3 values, s as float64 holding fp32)."""
    v = np.asarray(v, dtype=F64)
    amax = f32(np.max(np.abs(v), axis=-1))
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    ratio = (f32(v) / s[..., None]).astype(F64)          # correctly rounded fp32 divide
    q = e4m3_round(ratio)
    return q, s.astype(F64)


def quantize_nvfp4(w: np.ndarray):
    """NVFP4 quantisation of a weight matrix [N, K] along K.

    [SM] 4.4 and the support table name NVFP4 expert weights for Blackwell
    MoE but do not define the format.  Reading: the public NVFP4 layout,
    E2M1 elements in blocks of 16 consecutive K elements, one E4M3 scale per
    block and one fp32 scale per matrix:
        s_g = amax|W| / (448 * 6)                (1 for an all-zero matrix)
        s_b = e4m3( amax_block / (6 * s_g) )
        q   = e2m1( w / (s_b * s_g) )            (0 where s_b = 0)
    so that w ~ q * s_b * s_g.  The codes are decided in fp32, the precision
    the GPU decides them in: s_g, 6 * s_g, each block ratio, each product
    s_b * s_g and each element quotient are rounded to fp32.
    Returns (q float64 holding E2M1 values [N, K], s_b float64 holding E4M3
    values [N, K/16], s_g a float holding an fp32 value)."""
    w = np.asarray(w, dtype=F64)
    n, kdim = w.shape
    assert kdim % NVFP4_BLOCK == 0
    amax = f32(np.max(np.abs(w))) if w.size else np.float32(0.0)
    sg = np.float32(amax / np.float32(E4M3_MAX * E2M1_MAX)) if amax > 0 else np.float32(1.0)
    six_sg = np.float32(np.float32(E2M1_MAX) * sg)
    wb = f32(w).reshape(n, kdim // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(wb), axis=-1)
    sb = e4m3_round((amax_b / six_sg).astype(np.float32).astype(F64))
    scale = (sb.astype(np.float32) * sg).astype(np.float32)          # fp32 product
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (wb / scale[..., None]).astype(np.float32).astype(F64)
    q = np.where(scale[..., None] > 0, e2m1_round(ratio), 0.0)
    return q.reshape(n, kdim), sb, float(sg)


def dequantize_nvfp4(q, sb, sg) -> np.ndarray:
    """w = q * s_b * s_g (exact in fp64: at most 5 significant bits times an fp32)."""
    q = np.asarray(q, dtype=F64)
    return q * np.repeat(np.asarray(sb, dtype=F64), NVFP4_BLOCK, axis=-1) * float(sg)


# ---------------------------------------------------------------------------
# Steps of the path
# ---------------------------------------------------------------------------

def silu(z):
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z)).  [V100] 2nd wall names the
    silu_and_mul op; the formula is the standard SiLU."""
    z = np.asarray(z, dtype=F64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def rms_norm(x, w, eps):
    """x_hat = bf16( x / sqrt(mean(x^2) + eps) * w ), per row.

    [V100] "rewrite on torch::stable::Tensor": rms_norm is the composite
    pow -> mean -> rsqrt -> mul; rsqrt is 1/sqrt here, in fp64.  The output is
    rounded once to bf16, the dtype the op writes (its input dtype)."""
    x = np.asarray(x, dtype=F64)
    w = np.asarray(w, dtype=F64)
    ms = np.mean(x ** 2, axis=-1, keepdims=True)
    return bf16_round(x / np.sqrt(ms + eps) * w)


def router_logits(xhat, router_w, router_bias=None):
    """logits[t, e] = sum_h xhat[t, h] * W_r[h, e] (+ b[e]).

    The router is a plain linear layer over the normalised tokens; the
    per-expert bias (skewed workload) is added to the logits before softmax
    and so moves both the selection and the weights (plain reading)."""
    l = np.asarray(xhat, dtype=F64) @ np.asarray(router_w, dtype=F64)
    if router_bias is not None:
        l = l + np.asarray(router_bias, dtype=F64)[None, :]
    return l


def softmax(logits):
    """p = exp(l - max l) / sum exp(l - max l) over the last axis.
    [RUBIN] "Hardware grows": exp throughput matters for softmax."""
    l = np.asarray(logits, dtype=F64)
    z = np.exp(l - l.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def topk_renorm(logits, k):
    """Top-k of the softmax, renormalised.

    ids: the k experts with the largest probability, in descending order,
    ties to the lower expert index.  Because softmax is strictly increasing
    in the logit, the selection is taken on the logits themselves.
    weights: w_j = p_{ids_j} / sum_j' p_{ids_j'} (fp64).
    Returns (ids int32 [T,k], weights float64 [T,k])."""
    l = np.asarray(logits, dtype=F64)
    T, E = l.shape
    assert 1 <= k <= E
    order = np.argsort(-l, axis=-1, kind="stable")      # stable: ties keep index order
    ids = order[:, :k].astype(np.int32)
    p = softmax(l)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=-1)
    w = sel / sel.sum(axis=-1, keepdims=True)
    return ids, w


def permute(ids, E):
    """Group the T*k (token, slot) pairs by expert.

    Rows are ordered by (expert ascending, token ascending); a token uses an
    expert at most once, so the order is unique.  row_src[r] = t*k + j is the
    pair that row r holds; offsets[e] .. offsets[e+1] is expert e's segment.
    Returns (offsets int32 [E+1], row_src int32 [T*k])."""
    ids = np.asarray(ids)
    flat = ids.reshape(-1).astype(np.int64)
    row_src = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets, row_src


def silu_and_mul(h, I):
    """a = bf16( silu(h[:, :I]) * h[:, I:] ) -- [V100] 2nd wall (op name);
    first half is the gate, second half the up projection."""
    h = np.asarray(h, dtype=F64)
    return bf16_round(silu(h[:, :I]) * h[:, I:])


def grouped_fc1(xp, offsets, w13_of, I):
    """FC1 gate/up per expert + silu_and_mul.  [RUBIN] Locality domain (FC1).

    For rows r in expert e's segment: h = xp[r] @ W13[e]^T  (W13[e] is
    [2I, H], rows 0..I-1 gate, I..2I-1 up), then a = silu_and_mul(h)."""
    xp = np.asarray(xp, dtype=F64)
    out = np.zeros((xp.shape[0], I), dtype=F64)
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        h = xp[r0:r1] @ np.asarray(w13_of(e), dtype=F64).T
        out[r0:r1] = silu_and_mul(h, I)
    return out


def grouped_fc2(a, offsets, w2_of, row_weight):
    """FC2 per expert with the routing weight applied: Y[r] = w_r * (a[r] @ W2[e]^T).
    [RUBIN] Locality domain (FC2); W2[e] is [H, I]."""
    a = np.asarray(a, dtype=F64)
    H = None
    Y = None
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        w2 = np.asarray(w2_of(e), dtype=F64)
        if Y is None:
            H = w2.shape[0]
            Y = np.zeros((a.shape[0], H), dtype=F64)
        Y[r0:r1] = (a[r0:r1] @ w2.T) * np.asarray(row_weight[r0:r1], dtype=F64)[:, None]
    if Y is None:
        Y = np.zeros((a.shape[0], 0), dtype=F64)
    return Y


def combine(Y, row_src, T, k):
    """out[t] = bf16( sum_{j=0..k-1} Y[row of (t, j)] ), summed in j order."""
    Y = np.asarray(Y, dtype=F64)
    pos = np.empty(T * k, dtype=np.int64)
    pos[np.asarray(row_src, dtype=np.int64)] = np.arange(T * k)
    out = np.zeros((T, Y.shape[1]), dtype=F64)
    for j in range(k):
        out += Y[pos[np.arange(T) * k + j]]
    return bf16_round(out)


# ---------------------------------------------------------------------------
# FP8 W8A8 pieces
# ---------------------------------------------------------------------------

def grouped_fc1_fp8(xq, sx_rows, offsets, w13q_of, s13_of, I):
    """FC1 on E4M3 operands: h = (xq . W13q^T) * s_x[r] * s_w[e, n], fp64 sums;
    then a = silu_and_mul(h) in bf16.  [SM] 3.1: c = (a*s_a)(b*s_b)."""
    out = np.zeros((xq.shape[0], I), dtype=F64)
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        h = (xq[r0:r1] @ np.asarray(w13q_of(e), dtype=F64).T)
        h = h * sx_rows[r0:r1, None] * np.asarray(s13_of(e), dtype=F64)[None, :]
        out[r0:r1] = silu_and_mul(h, I)
    return out


def grouped_fc2_fp8(a, offsets, w2q_of, s2_of, row_weight):
    """FC2 on E4M3 operands: the bf16 row a[r] is quantised per row
    (s_a = absmax/448), y = (aq . W2q^T) * s_a[r] * s_w[e, h]; Y = w_r * y."""
    aq, sa = quantize_rows_e4m3(a)
    Y = None
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        w2q = np.asarray(w2q_of(e), dtype=F64)
        if Y is None:
            Y = np.zeros((a.shape[0], w2q.shape[0]), dtype=F64)
        y = (aq[r0:r1] @ w2q.T) * sa[r0:r1, None] * np.asarray(s2_of(e), dtype=F64)[None, :]
        Y[r0:r1] = y * np.asarray(row_weight[r0:r1], dtype=F64)[:, None]
    return Y


# ---------------------------------------------------------------------------
# Block-wise FP8 pieces
# ---------------------------------------------------------------------------

FP8_BLOCK = 128


def quantize_blocks_e4m3(v: np.ndarray, block_rows: int, block_cols: int = FP8_BLOCK):
    """Block-wise dynamic E4M3 quantisation of a matrix [N, K]: one fp32
    scale per block_rows x block_cols tile, s = absmax(tile)/448, and
    q = e4m3(v/s) for every element of the tile.

    [SM] support table ("FP8 block-wise" MoE GEMMs) and the Hopper data-flow
    figure ("block-wise FP8 dequant inside GEMM loop") name the scheme
    without defining it.  Reading: 128 x 128 weight tiles (block_rows = 128)
    and per-token groups of 128 consecutive K elements for activations
    (block_rows = 1); the scale and the division are taken in fp32, as in
    quantize_rows_e4m3, and an all-zero tile gets s = 1, q = 0.
    Returns (q float64 holding E4M3 values [N, K], s float64 holding fp32
    values [N / block_rows, K / block_cols])."""
    v = np.asarray(v, dtype=F64)
    n, kdim = v.shape
    assert n % block_rows == 0 and kdim % block_cols == 0
    tiles = f32(v).reshape(n // block_rows, block_rows, kdim // block_cols, block_cols)
    amax = np.max(np.abs(tiles), axis=(1, 3))
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    ratio = (tiles / s[:, None, :, None]).astype(F64)     # correctly rounded fp32 divide
    q = e4m3_round(ratio)
    return q.reshape(n, kdim), s.astype(F64)


def block_scaled_matmul(aq, sa, wq, sw, block_cols: int = FP8_BLOCK):
    """y[r, n] = sum over K groups g of  s_a[r, g] * s_w[n / 128, g] *
    (sum over k in g of aq[r, k] * wq[n, k]).

    The products of each 128-wide K group are summed exactly (fp64 over E4M3
    values) and scaled once; the scaled group sums are added in K order (the
    "dequantise inside the GEMM loop" of the block-wise scheme).  aq [R, K]
    with sa [R, K/128]; wq [N, K] with sw [N/128, K/128]."""
    aq = np.asarray(aq, dtype=F64)
    wq = np.asarray(wq, dtype=F64)
    sa = np.asarray(sa, dtype=F64)
    sw = np.asarray(sw, dtype=F64)
    rows_per_wblock = wq.shape[0] // sw.shape[0]
    y = np.zeros((aq.shape[0], wq.shape[0]), dtype=F64)
    for g in range(aq.shape[1] // block_cols):
        ks = slice(g * block_cols, (g + 1) * block_cols)
        part = aq[:, ks] @ wq[:, ks].T
        y += part * sa[:, g, None] * np.repeat(sw[:, g], rows_per_wblock)[None, :]
    return y


def grouped_fc1_fp8_block(xq, sx_rows, offsets, w13q_of, s13_of, I):
    """FC1 with block-wise FP8: h = block_scaled_matmul(x_q, s_x, W13_q, s_w)
    per expert segment (s_x [R, H/128] per row and K group, s_w
    [2I/128, H/128]), then a = silu_and_mul(h) in bf16."""
    out = np.zeros((xq.shape[0], I), dtype=F64)
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        h = block_scaled_matmul(xq[r0:r1], sx_rows[r0:r1], w13q_of(e), s13_of(e))
        out[r0:r1] = silu_and_mul(h, I)
    return out


def grouped_fc2_fp8_block(a, offsets, w2q_of, s2_of, row_weight):
    """FC2 with block-wise FP8: the bf16 row a[r] is quantised in groups of
    128 (quantize_blocks_e4m3 with block_rows = 1), y = block_scaled_matmul
    (a_q, s_a, W2_q, s_w) with s_w [H/128, I/128]; Y = w_r * y."""
    aq, sa = quantize_blocks_e4m3(a, 1)
    Y = None
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        w2q = np.asarray(w2q_of(e), dtype=F64)
        if Y is None:
            Y = np.zeros((a.shape[0], w2q.shape[0]), dtype=F64)
        y = block_scaled_matmul(aq[r0:r1], sa[r0:r1], w2q, s2_of(e))
        Y[r0:r1] = y * np.asarray(row_weight[r0:r1], dtype=F64)[:, None]
    return Y


# ---------------------------------------------------------------------------
# Whole forward
# ---------------------------------------------------------------------------

def route(xhat, router_w=None, router_bias=None, logits=None, k=1):
    """Router step: logits (given, or x_hat @ W_r + b), then top-k renorm."""
    if logits is None:
        logits = router_logits(xhat, router_w, router_bias)
    ids, w = topk_renorm(logits, k)
    return logits, ids, w


def moe_ffn_forward(x, norm_w, eps, k, w13, w2, router_w=None, router_bias=None,
                    logits=None, ids=None, topk_w=None, fp8=False):
    """The full path: rms_norm -> router/top-k -> permute -> FC1+silu_and_mul
    -> FC2 (x routing weight) -> combine.

    ``w13``/``w2`` are [E,2I,H] / [E,H,I] arrays (or callables e -> expert
    matrix).  Routing is computed from ``router_w`` or ``logits`` unless
    ``ids``/``topk_w`` are given.  With fp8=True the weights are quantised
    per output channel and the activations per row, as quantize_rows_e4m3;
    with fp8="block" in 128 x 128 weight tiles and 1 x 128 activation groups,
    as quantize_blocks_e4m3.  Returns a dict with every intermediate."""
    x = np.asarray(x, dtype=F64)
    T, H = x.shape
    w13_of = w13 if callable(w13) else (lambda e, _w=w13: _w[e])
    w2_of = w2 if callable(w2) else (lambda e, _w=w2: _w[e])
    E = (np.asarray(router_w).shape[1] if router_w is not None else
         np.asarray(logits).shape[1] if logits is not None else
         (np.asarray(w13).shape[0] if not callable(w13) else None))
    xhat = rms_norm(x, norm_w, eps)
    if ids is None:
        logits, ids, topk_w = route(xhat, router_w, router_bias, logits, k)
    ids = np.asarray(ids, dtype=np.int32)
    topk_w = np.asarray(topk_w, dtype=F64)
    offsets, row_src = permute(ids, E)
    tok = row_src // k
    row_w = topk_w.reshape(-1)[row_src]
    I = np.asarray(w2_of(int(ids.flat[0]))).shape[1]  # any expert in use gives I
    if not fp8:
        xp = xhat[tok]
        A = grouped_fc1(xp, offsets, w13_of, I)
        Y = grouped_fc2(A, offsets, w2_of, row_w)
    elif fp8 == "block":
        xq, sx = quantize_blocks_e4m3(xhat, 1)
        cache13, cache2 = {}, {}

        def b13(e):
            if e not in cache13:
                cache13[e] = quantize_blocks_e4m3(w13_of(e), FP8_BLOCK)
            return cache13[e]

        def b2(e):
            if e not in cache2:
                cache2[e] = quantize_blocks_e4m3(w2_of(e), FP8_BLOCK)
            return cache2[e]
        A = grouped_fc1_fp8_block(xq[tok], sx[tok], offsets, lambda e: b13(e)[0],
                                  lambda e: b13(e)[1], I)
        Y = grouped_fc2_fp8_block(A, offsets, lambda e: b2(e)[0], lambda e: b2(e)[1], row_w)
    else:
        xq, sx = quantize_rows_e4m3(xhat)
        cache13, cache2 = {}, {}

        def q13(e):
            if e not in cache13:
                cache13[e] = quantize_rows_e4m3(w13_of(e))
            return cache13[e]

        def q2(e):
            if e not in cache2:
                cache2[e] = quantize_rows_e4m3(w2_of(e))
            return cache2[e]
        A = grouped_fc1_fp8(xq[tok], sx[tok], offsets, lambda e: q13(e)[0],
                            lambda e: q13(e)[1], I)
        Y = grouped_fc2_fp8(A, offsets, lambda e: q2(e)[0], lambda e: q2(e)[1], row_w)
    out = combine(Y, row_src, T, k)
    return dict(xhat=xhat, logits=logits, ids=ids, topk_w=topk_w, offsets=offsets,
                row_src=row_src, A=A, Y=Y, out=out)


def ffn_token_outputs(xhat_rows, ids, topk_w, w13_of, w2_of, I, cols=None, fp8=False,
                      wq13_of=None, wq2_of=None):
    """Direct per-token definition, out_t = bf16( sum_j w_j * FFN_{ids_j}(x_hat_t) ),
    for a subset of tokens (and optionally a subset of output columns).

    Used for sampled checks at full size: it needs only the experts the
    sampled tokens use.  Work is grouped by expert so each expert's weights
    are converted once.  For fp8=True (or "block"), ``wq13_of``/``wq2_of``
    return (codes, scales) of the quantised expert weights (per-channel, or
    per 128 x 128 tile).  NVFP4 weights with bf16
    activations are the bf16 path on the dequantised weights: pass
    ``w13_of``/``w2_of`` returning dequantize_nvfp4(...)."""
    xhat_rows = np.asarray(xhat_rows, dtype=F64)
    ids = np.asarray(ids)
    topk_w = np.asarray(topk_w, dtype=F64)
    n, k = ids.shape
    nc = len(cols) if cols is not None else None
    acc = None
    if fp8 == "block":
        xq, sx = quantize_blocks_e4m3(xhat_rows, 1)
    elif fp8:
        xq, sx = quantize_rows_e4m3(xhat_rows)
    for e in np.unique(ids):
        tj = np.argwhere(ids == e)                      # (token-in-subset, slot) pairs
        rows = tj[:, 0]
        if not fp8:
            h = xhat_rows[rows] @ np.asarray(w13_of(int(e)), dtype=F64).T
            a = silu_and_mul(h, I)
            w2 = np.asarray(w2_of(int(e)), dtype=F64)
            if cols is not None:
                w2 = w2[cols]
            y = a @ w2.T
        elif fp8 == "block":
            q13, s13 = wq13_of(int(e))
            h = block_scaled_matmul(xq[rows], sx[rows], q13, s13)
            a = silu_and_mul(h, I)
            aq, sa = quantize_blocks_e4m3(a, 1)
            q2, s2 = wq2_of(int(e))
            q2 = np.asarray(q2, dtype=F64)
            s2 = np.asarray(s2, dtype=F64)
            if cols is not None:
                # the weight scale of output column n is s2[n / 128]
                s2 = np.repeat(s2, q2.shape[0] // s2.shape[0], axis=0)[cols]
                q2 = q2[cols]
            y = block_scaled_matmul(aq, sa, q2, s2)
        else:
            q13, s13 = wq13_of(int(e))
            h = (xq[rows] @ np.asarray(q13, dtype=F64).T) * sx[rows, None] * np.asarray(s13)[None, :]
            a = silu_and_mul(h, I)
            aq, sa = quantize_rows_e4m3(a)
            q2, s2 = wq2_of(int(e))
            q2 = np.asarray(q2, dtype=F64)
            s2 = np.asarray(s2, dtype=F64)
            if cols is not None:
                q2, s2 = q2[cols], s2[cols]
            y = (aq @ q2.T) * sa[:, None] * s2[None, :]
        if acc is None:
            acc = np.zeros((n, k, y.shape[1]), dtype=F64)
        acc[tj[:, 0], tj[:, 1]] = y * topk_w[tj[:, 0], tj[:, 1]][:, None]
    out = np.zeros((n, acc.shape[2]), dtype=F64)
    for j in range(k):                                  # j order, as combine()
        out += acc[:, j]
    return bf16_round(out)
