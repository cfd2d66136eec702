"""Helpers shared by the GPU parity tests: run the library on a workload and
compare with the oracle (routing bit-exact outside near ties, outputs within
the stated tolerance)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

TOL_BF16 = 2e-2
TOL_FP8 = 6e-2
# Near-tie band for routing.  The GPU rounds x_hat to bf16 from an fp32
# value, the oracle from an fp64 one; about one element in 2e4 lands on the
# other side of a rounding midpoint, which moves it by one bf16 step (up to
# ~2^-7 |x_hat|) and a logit by up to ~|x_hat| 2^-7 max|W_r| ~ 1e-3.  A token
# whose k-th and (k+1)-th fp64 logits (or two adjacent selected logits) are
# closer than the band may therefore select differently; elsewhere the ids
# must match exactly.
TIE_REL = 1e-3
# Weight tolerance that follows: dw = w(1-w) dl <= 0.25 * 1e-3.
W_ATOL = 3e-4


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def scaled_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(got - ref) / np.maximum(1.0, np.abs(ref))


def assert_close(got, ref, tol, what=""):
    err = scaled_err(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err.max() <= tol, f"{what}: max scaled error {err.max():.3e} > {tol} at {np.unravel_index(err.argmax(), err.shape)}"
    return err.max()


def near_tie_tokens(logits: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose top-(k+1) sorted logits have an adjacent gap below the band."""
    l = np.sort(logits, axis=1)[:, ::-1][:, :k + 1]
    band = TIE_REL * np.maximum(1.0, np.abs(l[:, :1]))
    gaps = l[:, :-1] - l[:, 1:]
    if l.shape[1] == k:  # k == E: only the order inside the selection matters
        return np.any(gaps < band, axis=1)
    return np.any(gaps < band, axis=1)


def check_routing(ids_gpu, w_gpu, logits64, k, tol_w=1e-3):
    """ids must equal the oracle's outside near ties; inside them the GPU's
    choice must be a valid top-k within the band.  Returns (oracle ids,
    weights used for the output check, number of near-tie tokens that differ)."""
    ids_ref, w_ref = O.topk_renorm(logits64, k)
    tie = near_tie_tokens(logits64, k)
    diff = np.any(ids_gpu != ids_ref, axis=1)
    bad = diff & ~tie
    assert not bad.any(), f"routing differs outside near ties for tokens {np.where(bad)[0][:10]}"
    ids_use = ids_ref.copy()
    w_use = w_ref.copy()
    for t in np.where(diff)[0]:
        sel = ids_gpu[t].astype(np.int64)
        assert len(set(sel.tolist())) == k
        l = logits64[t]
        kth = np.sort(l)[::-1][k - 1]
        assert np.all(l[sel] >= kth - TIE_REL * max(1.0, abs(l.max()))), "GPU pick outside the tie band"
        ids_use[t] = ids_gpu[t]
        z = np.exp(l[sel] - l.max())
        w_use[t] = z / z.sum()
    np.testing.assert_allclose(w_gpu, w_use, rtol=tol_w, atol=W_ATOL)
    return ids_ref, w_use, int(diff.sum())
