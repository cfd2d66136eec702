"""Host logic of the GPU parity checks, on the CPU: the routing tie bands
accept only what they should, and the sampled tokens reach every tile."""
import numpy as np
import pytest

import oracle as O
from tests.parity_util import (TAU, assert_close, compare_routing, covering_tokens,
                               row_scaled_err)


def _logits(rng, T, E, spread=1.0):
    return rng.standard_normal((T, E)) * spread


def test_routing_identical_passes_and_counts_ties():
    rng = np.random.default_rng(0)
    l = _logits(rng, 50, 16)
    l[3, 5] = l[3, np.argsort(-l[3])[3]] + 0.3 * TAU     # a k / k+1 near tie (k = 4)
    ids, _ = O.topk_renorm(l, 4)
    _, c = compare_routing(ids, l, 4)
    assert c["set_ties_routed_apart"] == 0 and c["order_ties_routed_apart"] == 0


def test_routing_set_swap_outside_band_fails_inside_passes():
    rng = np.random.default_rng(1)
    l = _logits(rng, 20, 12)
    k = 3
    ids, _ = O.topk_renorm(l, k)
    t = 7
    srt = np.argsort(-l[t], kind="stable")
    bad = ids.copy()
    bad[t, k - 1] = srt[k]                      # the (k+1)-th expert instead of the k-th
    gap = l[t, srt[k - 1]] - l[t, srt[k]]
    assert gap > TAU
    with pytest.raises(AssertionError, match="set differs"):
        compare_routing(bad, l, k)
    # move the two logits inside the band: now either choice is accepted
    l2 = l.copy()
    l2[t, srt[k]] = l2[t, srt[k - 1]] - 0.5 * TAU
    ids2, _ = O.topk_renorm(l2, k)
    alt = ids2.copy()
    pos = list(ids2[t]).index(srt[k - 1]) if srt[k - 1] in ids2[t] else k - 1
    alt[t, pos] = srt[k] if srt[k] not in ids2[t] else srt[k - 1]
    _, c = compare_routing(alt, l2, k)
    assert c["set_ties_routed_apart"] == 1


def test_routing_order_swap_outside_band_fails_inside_passes():
    rng = np.random.default_rng(2)
    l = _logits(rng, 10, 8)
    k = 4
    ids, _ = O.topk_renorm(l, k)
    bad = ids.copy()
    bad[2, [0, 1]] = bad[2, [1, 0]]
    with pytest.raises(AssertionError, match="order differs"):
        compare_routing(bad, l, k)
    l2 = l.copy()
    l2[2, ids[2, 1]] = l2[2, ids[2, 0]] - 0.2 * TAU
    _, c = compare_routing(bad, l2, k)
    assert c["order_ties_routed_apart"] == 1


def test_routing_pick_outside_band_fails_even_at_a_tie():
    rng = np.random.default_rng(3)
    l = _logits(rng, 5, 10)
    k = 2
    srt = np.argsort(-l[1], kind="stable")
    l[1, srt[2]] = l[1, srt[1]] - 0.1 * TAU     # the 2nd and 3rd tie
    ids, _ = O.topk_renorm(l, k)
    bad = ids.copy()
    bad[1, 1] = srt[5]                          # a pick far below the band
    with pytest.raises(AssertionError):
        compare_routing(bad, l, k)


@pytest.mark.parametrize("T,E,k", [(4096, 64, 8), (300, 4, 2), (1000, 256, 8)])
def test_covering_tokens_reach_every_tile(T, E, k):
    rng = np.random.default_rng(T)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[: T // 5, 0] = 0                        # one hot expert with many tiles
    toks, ntiles = covering_tokens(ids, E, k, tile=128, n_min=256, seed=0)
    offsets, row_src = O.permute(ids, E)
    pos = np.empty(T * k, dtype=np.int64)
    pos[row_src] = np.arange(T * k)
    rows = pos[(toks[:, None] * k + np.arange(k)).reshape(-1)]
    hit = set()
    for r in rows:
        e = int(np.searchsorted(offsets, r, side="right") - 1)
        hit.add((e, (int(r) - int(offsets[e])) // 128))
    want = {(e, i) for e in range(E) for i in range((int(offsets[e + 1]) - int(offsets[e]) + 127) // 128)}
    assert hit == want and len(want) == ntiles
    assert len(toks) >= min(T, 256) and len(np.unique(toks)) == len(toks)


def test_row_relative_tolerance_has_teeth_at_small_magnitudes():
    rng = np.random.default_rng(4)
    ref = rng.standard_normal((6, 64)) * 0.02
    got = ref.copy()
    got[2, 7] += 0.3 * np.sqrt(np.mean(ref[2] ** 2))   # 30% of the row's rms
    with pytest.raises(AssertionError, match="row-relative"):
        assert_close(got, ref, 2e-2)
    assert row_scaled_err(ref, ref).max() == 0
    assert_close(ref * (1 + 1e-3), ref, 2e-2)


def test_xhat_rows_that_differ_are_taken_from_the_gpu_and_bounded():
    from tests.parity_util import check_routing_e2e
    rng = np.random.default_rng(5)
    T, H, E, k = 40, 64, 8, 2
    x = O.bf16_round(rng.standard_normal((T, H)))
    nw = O.bf16_round(1 + 0.1 * rng.standard_normal(H))
    Wr = rng.standard_normal((H, E)) * 0.02
    xhat = O.rms_norm(x, nw, 1e-6)
    l = O.router_logits(xhat, Wr)
    ids, w = O.topk_renorm(l, k)
    xg = xhat.copy()
    # one element of token 3 one bf16 step away (a rounding decision taken the other way)
    step = np.ldexp(1.0, np.frexp(abs(xg[3, 5]))[1] - 8)
    xg[3, 5] += step
    ids_g, _ = O.topk_renorm(O.router_logits(xg, Wr), k)
    w_g = O.topk_renorm(O.router_logits(xg, Wr), k)[1]
    _, _, xuse, c = check_routing_e2e(ids_g, w_g, x, nw, 1e-6, k, xhat_gpu=xg, router_w=Wr)
    assert c["xhat_rows_differ"] == 1
    np.testing.assert_array_equal(xuse[3], xg[3])
    np.testing.assert_array_equal(np.delete(xuse, 3, axis=0), np.delete(xhat, 3, axis=0))
    # two steps away is not a rounding decision: rejected
    xbad = xg.copy()
    xbad[3, 5] += step
    with pytest.raises(AssertionError, match="more than one bf16 step"):
        check_routing_e2e(ids_g, w_g, x, nw, 1e-6, k, xhat_gpu=xbad, router_w=Wr)
