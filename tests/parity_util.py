"""Helpers shared by the GPU parity tests: compare the library with the oracle
(routing bit-exact outside the stated tie bands, outputs within the stated
tolerances), choose sampled tokens that reach every tile, and record how many
tokens each workload exempted from the bit-exact routing check."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle as O

TOL_BF16 = 2e-2
TOL_FP8 = 6e-2

# Routing tie band (the set of selected experts): a token whose k-th and
# (k+1)-th fp64 logits are closer than TAU * max(1, |l_k|, |l_k+1|) may
# select either expert; every other token must select exactly the oracle's
# experts, in the oracle's order (descending logit, ties to the lower index).
TAU = 1e-4
# The router's own arithmetic error bound.  The GPU sums the logits in fp32
# (or on the tensor cores with fp32 accumulation); the oracle in fp64 from the
# same bf16 x_hat.  Measured |l_gpu - l_fp64| <= 3.2e-5 on every routing
# workload here; the checks below assert that bound per token, so a tie band
# of twice a token's own logit error is below TAU.
ROUTER_ERR = 5e-5


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def scaled_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(got - ref) / np.maximum(1.0, np.abs(ref))


def row_scaled_err(got, ref):
    """|got - ref| / max(|ref|, rms of ref's row): the tolerance form that keeps
    its teeth when outputs are much smaller than 1."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True)) if ref.ndim > 1 else \
        np.sqrt(np.mean(ref * ref))
    return np.abs(got - ref) / np.maximum(np.maximum(np.abs(ref), rms), 1e-30)


def assert_close(got, ref, tol, what="", rows=True):
    """Both forms must hold: |got - ref| <= tol * max(1, |ref|) (the stated
    tolerance) and |got - ref| <= tol * max(|ref|, rms(ref row)) (relative to
    the row's own magnitude).  Returns the first form's maximum."""
    err = scaled_err(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err.max() <= tol, f"{what}: max scaled error {err.max():.3e} > {tol} at {np.unravel_index(err.argmax(), err.shape)}"
    if rows:
        rel = row_scaled_err(got, ref)
        assert rel.max() <= tol, (f"{what}: max row-relative error {rel.max():.3e} > {tol} at "
                                  f"{np.unravel_index(rel.argmax(), rel.shape)}")
    return err.max()


# ----------------------------------------------------------------- routing --

def _boundary_gap(l, k):
    """Per token: the gap between the k-th and (k+1)-th largest logit, and the
    tie band TAU * max(1, |l_k|, |l_k+1|) (an infinite gap when k == E)."""
    s = -np.sort(-l, axis=1)
    if s.shape[1] == k:
        return np.full(l.shape[0], np.inf), np.full(l.shape[0], TAU)
    gap = s[:, k - 1] - s[:, k]
    band = TAU * np.maximum(1.0, np.maximum(np.abs(s[:, k - 1]), np.abs(s[:, k])))
    return gap, band


def _order_gap(l, ids):
    """Per token: the smallest gap between adjacent selected logits (in the
    oracle's order), i.e. how close the ordering inside the selection is."""
    sel = np.take_along_axis(l, ids.astype(np.int64), axis=1)
    if sel.shape[1] < 2:
        return np.full(l.shape[0], np.inf)
    return np.min(sel[:, :-1] - sel[:, 1:], axis=1)


def compare_routing(ids_gpu, l_ref, k, band_of=None):
    """ids_gpu against the oracle's top-k of l_ref.

    The set must be the oracle's wherever the k / (k+1) gap is at least the
    band; the order inside the set must be the oracle's wherever adjacent
    selected logits differ by at least the band.  Inside a band the GPU's
    choice must still be a valid top-k of l_ref within that band.
    band_of: optional per-token band (default TAU * max(1, |l|)).
    Returns (ids_ref, counts) with counts of tokens exempted by each band."""
    ids_ref, _ = O.topk_renorm(l_ref, k)
    gap, band = _boundary_gap(l_ref, k)
    if band_of is not None:
        band = band_of
    ogap = _order_gap(l_ref, ids_ref)
    T = ids_gpu.shape[0]
    set_g = np.sort(ids_gpu, axis=1)
    set_r = np.sort(ids_ref, axis=1)
    set_diff = np.any(set_g != set_r, axis=1)
    order_diff = ~set_diff & np.any(ids_gpu != ids_ref, axis=1)
    set_tie = gap < band
    order_tie = ogap < band
    bad_set = set_diff & ~set_tie
    assert not bad_set.any(), (f"routing set differs outside the tie band for tokens "
                               f"{np.where(bad_set)[0][:10]} (gaps {gap[bad_set][:5]})")
    bad_order = order_diff & ~order_tie
    assert not bad_order.any(), (f"routing order differs outside the tie band for tokens "
                                 f"{np.where(bad_order)[0][:10]}")
    for t in np.where(set_diff | order_diff)[0]:
        sel = ids_gpu[t].astype(np.int64)
        assert len(set(sel.tolist())) == k and sel.min() >= 0 and sel.max() < l_ref.shape[1]
        kth = -np.sort(-l_ref[t])[k - 1]
        assert np.all(l_ref[t, sel] >= kth - band[t]), f"token {t}: a GPU pick lies outside the band"
        # the GPU's own order is descending within the band
        assert np.all(np.diff(l_ref[t, sel]) <= band[t]), f"token {t}: GPU order not descending"
    counts = dict(tokens=int(T), set_ties=int(set_tie.sum()), set_ties_routed_apart=int(set_diff.sum()),
                  order_ties=int((order_tie & ~set_tie).sum()), order_ties_routed_apart=int(order_diff.sum()),
                  min_gap=float(np.min(gap)) if T else None)
    return ids_ref, counts


def topk_weights(l, ids):
    """Renormalised softmax weights of the given selection (fp64)."""
    sel = np.take_along_axis(l, ids.astype(np.int64), axis=1)
    z = np.exp(sel - np.max(l, axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def check_router(ids_gpu, w_gpu, l_gpu, l64, k):
    """The router step fed the GPU's own x_hat: l64 is the oracle's fp64 logit
    from that same x_hat, l_gpu the kernel's fp32 logit.

    - the logits agree to ROUTER_ERR * max(1, |l|);
    - the selection equals the oracle's top-k of the GPU's own fp32 logits
      bit-exactly (the decision in the kernel's precision);
    - against the fp64 logits, a token may differ only where a gap is below
      twice its own logit error (<= 2 * ROUTER_ERR, below TAU)."""
    err = np.abs(l_gpu - l64)
    scale = np.maximum(1.0, np.abs(l64))
    assert np.all(err <= ROUTER_ERR * scale), f"router logit error {np.max(err / scale):.2e}"
    ids32, _ = O.topk_renorm(l_gpu, k)
    np.testing.assert_array_equal(ids_gpu, ids32)
    band = 2.0 * np.max(err, axis=1) + 1e-12
    ids_ref, counts = compare_routing(ids_gpu, l64, k, band_of=band)
    np.testing.assert_allclose(w_gpu, topk_weights(l64, ids_gpu), rtol=2e-4, atol=1e-6)
    counts["max_logit_err"] = float(err.max()) if err.size else 0.0
    return ids_ref, counts


def check_routing_e2e(ids_gpu, w_gpu, x, norm_w, eps, k, xhat_gpu=None, router_w=None,
                      router_bias=None, logits=None, name="", max_exempt=None):
    """End-to-end routing of a forward against the oracle, and the x_hat the
    oracle's FFN check should use.

    x_hat: the GPU rounds x_hat to bf16 from fp32, the oracle from fp64, so
    about one element in 2e4 lands on the other side of a rounding midpoint
    (checked here: at most one bf16 step, in under 0.1% of the elements).
    Everything downstream that rounds or quantises (the router's top-k, the
    E4M3 codes of the FP8 paths) is discontinuous in x_hat, so for the tokens
    whose x_hat rows differ -- and only for those -- the oracle recomputes from
    the GPU's x_hat, as it does for near ties.

    Routing: with given logits, the oracle's top-k of those logits.  With a
    router, the oracle's fp64 logits (from its own x_hat, or the GPU's for the
    rows above): the set must match wherever the k / (k+1) gap is at least
    TAU, the order wherever adjacent selected logits differ by at least TAU.
    Returns (ids to use for the output check, weights, x_hat to use, counts)."""
    x64 = np.asarray(x, dtype=np.float64)
    xhat = O.rms_norm(x64, norm_w, eps)
    T = x64.shape[0]
    differ = np.zeros(T, dtype=bool)
    xhat_use = xhat
    if xhat_gpu is not None:
        xg = np.asarray(xhat_gpu, dtype=np.float64)
        ulp = np.ldexp(1.0, np.frexp(np.abs(xhat))[1] - 8)
        assert np.all(np.abs(xg - xhat) <= ulp + 1e-30), "x_hat differs by more than one bf16 step"
        assert np.mean(xg != xhat) < 1e-3, "x_hat differs too often"
        differ = np.any(xg != xhat, axis=1)
        if differ.any():
            xhat_use = xhat.copy()
            xhat_use[differ] = xg[differ]
    if logits is not None:
        l_ref = np.asarray(logits, dtype=np.float64)
        _, counts = compare_routing(ids_gpu, l_ref, k)
        counts["rerouted_by_xhat"] = 0
    else:
        bias = None if router_bias is None else np.asarray(router_bias, dtype=np.float64)
        l64 = O.router_logits(xhat, router_w, bias)
        l_ref = l64
        if differ.any():
            l_ref = l64.copy()
            l_ref[differ] = O.router_logits(xhat_use[differ], router_w, bias)
        _, counts = compare_routing(ids_gpu, l_ref, k)
        ids_def, _ = O.topk_renorm(l64, k)
        counts["rerouted_by_xhat"] = int((np.any(ids_def != np.asarray(ids_gpu), axis=1) & differ).sum())
    counts["xhat_rows_differ"] = int(differ.sum())
    w_use = topk_weights(l_ref, ids_gpu)
    np.testing.assert_allclose(w_gpu, w_use, rtol=2e-4, atol=1e-6)
    limit = max_exempt if max_exempt is not None else max(2, int(0.005 * T))
    exempt = counts["set_ties_routed_apart"] + counts["order_ties_routed_apart"] + counts["rerouted_by_xhat"]
    assert exempt <= limit, f"{name}: {exempt} tokens exempted from bit-exact routing (> {limit})"
    record(name, counts)
    return np.asarray(ids_gpu), w_use, xhat_use, counts


def o1_weights(inp):
    """Rescale a small workload's expert weights so that FC1 and the forward's
    outputs are of order one (std 1/sqrt(H) for W13, 2/sqrt(I) for W2): the
    tolerance then bounds errors relative to values near 1, not to 0.02."""
    H, I = inp["H"], inp["I"]
    inp["w13"] = (inp["w13"].float() * (H ** -0.5 / 0.02)).to(torch.bfloat16)
    inp["w2"] = (inp["w2"].float() * (2.0 * I ** -0.5 / 0.02)).to(torch.bfloat16)
    return inp


# ------------------------------------------------------------ sampling --

def covering_tokens(ids, E, k, tile=128, n_min=256, seed=0, T=None):
    """Tokens to recompute at full size: at least one row of every
    (expert, tile-row token tile) of the permuted order -- the tiles the
    prefill kernels compute -- then random tokens up to n_min."""
    ids = np.asarray(ids)
    T = ids.shape[0] if T is None else T
    offsets, row_src = O.permute(ids, E)
    rng = np.random.default_rng(seed)
    tok_of_row = np.asarray(row_src) // k
    tiles = []
    for e in range(E):
        for r0 in range(int(offsets[e]), int(offsets[e + 1]), tile):
            tiles.append((r0, min(r0 + tile, int(offsets[e + 1]))))
    pos = np.empty(T * k, dtype=np.int64)
    pos[np.asarray(row_src, dtype=np.int64)] = np.arange(T * k)
    covered = np.zeros(len(tiles), dtype=bool)
    starts = np.array([t[0] for t in tiles])
    chosen = set()
    for i in rng.permutation(len(tiles)):
        if covered[i]:
            continue
        r0, r1 = tiles[i]
        t = int(tok_of_row[rng.integers(r0, r1)])
        chosen.add(t)
        rows = pos[t * k:(t + 1) * k]
        covered[np.searchsorted(starts, rows, side="right") - 1] = True
    assert covered.all()
    rest = [t for t in rng.permutation(T) if t not in chosen]
    need = max(0, n_min - len(chosen))
    chosen.update(int(t) for t in rest[:need])
    return np.array(sorted(chosen), dtype=np.int64), len(tiles)


# ------------------------------------------------------------- records --

RECORDS: dict = {}


def record(name, counts):
    """Keep a workload's routing-exemption counts for the session summary
    (conftest prints them as one JSON line; MOE_PARITY_RECORD=path also
    writes them to a file)."""
    if not name:
        return
    RECORDS[name] = counts
    path = os.environ.get("MOE_PARITY_RECORD")
    if path:
        with open(path, "w") as f:
            json.dump(RECORDS, f, indent=1, sort_keys=True)


def forward_xhat(M, ws, T, H):
    """The x_hat a forward computed: the library keeps it at the start of the
    forward's workspace (its first region, T x H bf16)."""
    off = M._ws_ptr(ws) - ws.data_ptr()
    return ws[off:off + T * H * 2].view(torch.bfloat16).view(T, H)
