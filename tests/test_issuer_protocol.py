"""Host-side models of the stage hand-offs in the kernels with several MMA
issuer threads: the NVFP4 decode kernel (csrc/gemm_nvfp4.cu) and the
block-wise FP8 prefill tiles (csrc/gemm_fp8b.cu, `run_tiles` below).

K stages n = 0, 1, .. of a CTA flow through two rings: the TMA producer fills
stage slot n % S (barriers sfull / sempty), the converting warps turn it into
an A operand in TMEM slot n % A (afull / aempty), and MMA issuer n % ni
consumes both; its commit releases the two slots when the MMAs complete.
Every wait is an mbarrier parity wait, which cannot tell phase k from phase
k - 2 or k + 2.  The kernel relies on each issuer's own previous stage being
at most A stages back (the kernel keeps ni <= min(S, A)), so that no wait
sees a phase that is a whole phase behind or ahead.

The model runs the roles under random interleavings (the MMA completions as
separate, delayed events) and checks every wait that passes against the
ground truth.  With ni <= A no run goes wrong (the A-slot wait also covers a
short stage ring); with more issuers than A slots, some interleaving
consumes a stage whose operand is not there yet.
"""
import random

import pytest


class Barrier:
    """An mbarrier: `count` arrivals complete the current phase."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0  # number of completed phases

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def try_wait_parity(self, parity):
        # true when the phase with this parity has completed, as the hardware
        # sees it: the current (incomplete) phase has the other parity
        return (self.phase & 1) != parity


class Violation(Exception):
    pass


def run(n_stages, ring_s, ring_a, ni, seed, max_delay=6):
    rng = random.Random(seed)
    sfull = [Barrier(1) for _ in range(ring_s)]
    sempty = [Barrier(2) for _ in range(ring_s)]  # MMA commit + the converters
    afull = [Barrier(1) for _ in range(ring_a)]
    aempty = [Barrier(1) for _ in range(ring_a)]  # MMA commit
    loaded, converted, consumed = set(), set(), set()
    slot_s = [None] * ring_s  # stage whose data a stage slot holds
    slot_a = [None] * ring_a  # stage whose operand an A slot holds
    prod = [0]
    conv = [0]
    iss = [b for b in range(ni)]  # next stage of each issuer
    inflight = []  # (time left, stage) of issued MMAs

    def producer():
        n = prod[0]
        if n >= n_stages:
            return False
        s = n % ring_s
        if not sempty[s].try_wait_parity(((n // ring_s) & 1) ^ 1):
            return False
        old = slot_s[s]
        if old is not None and not (old in consumed and old in converted):
            raise Violation(f"producer overwrote stage {old} with {n}")
        slot_s[s] = n
        loaded.add(n)
        sfull[s].arrive()
        prod[0] += 1
        return True

    def converter():
        n = conv[0]
        if n >= n_stages:
            return False
        s, a = n % ring_s, n % ring_a
        if not (sfull[s].try_wait_parity((n // ring_s) & 1) and
                aempty[a].try_wait_parity(((n // ring_a) & 1) ^ 1)):
            return False
        if slot_s[s] != n:
            raise Violation(f"converter read stage slot {s} for {n}, holds {slot_s[s]}")
        old = slot_a[a]
        if old is not None and old not in consumed:
            raise Violation(f"converter overwrote A operand of stage {old} with {n}")
        slot_a[a] = n
        converted.add(n)
        afull[a].arrive()
        sempty[s].arrive()
        conv[0] += 1
        return True

    def issuer(b):
        n = iss[b]
        if n >= n_stages:
            return False
        s, a = n % ring_s, n % ring_a
        if not (sfull[s].try_wait_parity((n // ring_s) & 1) and
                afull[a].try_wait_parity((n // ring_a) & 1)):
            return False
        if slot_s[s] != n or n not in loaded:
            raise Violation(f"issuer {b} read stage slot {s} for {n}, holds {slot_s[s]}")
        if slot_a[a] != n or n not in converted:
            raise Violation(f"issuer {b} read A slot {a} for {n}, holds {slot_a[a]}")
        inflight.append([rng.randint(0, max_delay), n])
        iss[b] += ni
        return True

    def complete():
        ready = [m for m in inflight if m[0] <= 0]
        if not ready:
            for m in inflight:
                m[0] -= 1
            return bool(inflight)
        m = rng.choice(ready)
        inflight.remove(m)
        n = m[1]
        consumed.add(n)
        aempty[n % ring_a].arrive()
        sempty[n % ring_s].arrive()
        return True

    roles = [producer, converter, complete] + [lambda b=b: issuer(b) for b in range(ni)]
    while len(consumed) < n_stages:
        order = roles[:]
        rng.shuffle(order)
        if not any(r() for r in order):
            raise Violation(f"deadlock with {len(consumed)} of {n_stages} stages consumed")
    return True


@pytest.mark.parametrize("ring_s,ring_a,ni", [(8, 3, 1), (8, 3, 2), (8, 3, 3), (4, 3, 3), (3, 3, 3),
                                              (5, 3, 2), (2, 3, 2)])
def test_issuers_within_the_ring_bound_never_misread(ring_s, ring_a, ni):
    assert ni <= min(ring_s, ring_a)
    for seed in range(300):
        run(40, ring_s, ring_a, ni, seed)


@pytest.mark.parametrize("ring_s,ring_a,ni", [(8, 3, 4), (8, 3, 5), (3, 3, 4)])
def test_more_issuers_than_a_slots_misreads_somewhere(ring_s, ring_a, ni):
    # the kernel's static_assert (issuers <= A slots) exists because of this
    failures = 0
    for seed in range(300):
        try:
            run(40, ring_s, ring_a, ni, seed)
        except Violation:
            failures += 1
    assert failures > 0


def test_stage_ring_shorter_than_the_issuer_count_is_still_covered():
    # An issuer's stage-slot wait may pass a phase early here, but its A-slot
    # wait holds it until the converters, which run in order behind the
    # producer, have converted its stage; so only the A ring bounds ni (the
    # kernel also keeps ni <= stages, which costs nothing at decode sizes).
    for seed in range(300):
        run(40, 2, 3, 3, seed)


def test_class_order_sum_is_independent_of_the_first_bank():
    """The epilogue adds bank (first + c) mod ni for c = 0, 1, ..: the bank
    holding the unit's stages ks = c (mod ni).  Each class's partial sum is
    the same whatever bank holds it, so the fp32 total is too."""
    import numpy as np
    rng = np.random.default_rng(0)
    for ni in (1, 2, 3):
        for kst in (1, 2, 3, 5, 16):
            parts = rng.standard_normal((kst, 16)).astype(np.float32)
            totals = set()
            for n0 in range(6):
                banks = [np.zeros(16, np.float32) for _ in range(ni)]
                for ks in range(kst):
                    banks[(n0 + ks) % ni] += parts[ks]
                first, nclass = n0 % ni, min(kst, ni)
                v = banks[first].copy()
                for c in range(1, nclass):
                    v += banks[(first + c) % ni]
                totals.add(v.tobytes())
            assert len(totals) == 1


def run_tiles(n_groups, ring_s, ring_q, ni, seed, max_delay=6):
    """The block-wise FP8 prefill tiles: TMA stages (ring S, released by the
    MMA commit), one TMEM slot per K group (ring Q: the MMA commit fills it,
    the in-order epilogue drains it), K group g issued by thread g % ni."""
    rng = random.Random(seed)
    sfull = [Barrier(1) for _ in range(ring_s)]
    sempty = [Barrier(1) for _ in range(ring_s)]
    kfull = [Barrier(1) for _ in range(ring_q)]
    kempty = [Barrier(1) for _ in range(ring_q)]
    slot_s = [None] * ring_s
    slot_q = [None] * ring_q  # group whose product a TMEM slot holds
    done, drained = set(), set()
    prod, epi = [0], [0]
    iss = [b for b in range(ni)]
    inflight = []

    def producer():
        g = prod[0]
        if g >= n_groups:
            return False
        s = g % ring_s
        if not sempty[s].try_wait_parity(((g // ring_s) & 1) ^ 1):
            return False
        old = slot_s[s]
        if old is not None and old not in done:
            raise Violation(f"producer overwrote group {old} with {g}")
        slot_s[s] = g
        sfull[s].arrive()
        prod[0] += 1
        return True

    def issuer(b):
        g = iss[b]
        if g >= n_groups:
            return False
        s, q = g % ring_s, g % ring_q
        if not (sfull[s].try_wait_parity((g // ring_s) & 1) and
                kempty[q].try_wait_parity(((g // ring_q) & 1) ^ 1)):
            return False
        if slot_s[s] != g:
            raise Violation(f"issuer {b} read stage slot {s} for {g}, holds {slot_s[s]}")
        old = slot_q[q]
        if old is not None and old not in drained:
            raise Violation(f"issuer {b} overwrote the product of group {old} with {g}")
        slot_q[q] = g
        inflight.append([rng.randint(0, max_delay), g])
        iss[b] += ni
        return True

    def complete():
        ready = [m for m in inflight if m[0] <= 0]
        if not ready:
            for m in inflight:
                m[0] -= 1
            return bool(inflight)
        m = rng.choice(ready)
        inflight.remove(m)
        g = m[1]
        done.add(g)
        sempty[g % ring_s].arrive()
        kfull[g % ring_q].arrive()
        return True

    def epilogue():
        g = epi[0]
        if g >= n_groups:
            return False
        q = g % ring_q
        if not kfull[q].try_wait_parity((g // ring_q) & 1):
            return False
        if slot_q[q] != g or g not in done:
            raise Violation(f"epilogue read slot {q} for {g}, holds {slot_q[q]}")
        drained.add(g)
        kempty[q].arrive()
        epi[0] += 1
        return True

    roles = [producer, complete, epilogue] + [lambda b=b: issuer(b) for b in range(ni)]
    while len(drained) < n_groups:
        order = roles[:]
        rng.shuffle(order)
        if not any(r() for r in order):
            raise Violation(f"deadlock with {len(drained)} of {n_groups} groups drained")
    return True


@pytest.mark.parametrize("ring_s,ring_q,ni", [(6, 4, 2), (6, 4, 1), (6, 4, 3), (5, 3, 2), (4, 4, 4),
                                              (2, 2, 2)])
def test_tile_issuers_within_the_slot_count_never_misread(ring_s, ring_q, ni):
    # the kernel runs six stages, four slots and two issuers; it keeps both
    # rings even, which is enough, though ni <= both ring lengths already is
    for seed in range(300):
        run_tiles(48, ring_s, ring_q, ni, seed)


@pytest.mark.parametrize("ring_s,ring_q,ni", [(6, 2, 3), (6, 4, 5)])
def test_tile_issuers_beyond_the_slot_count_misread_somewhere(ring_s, ring_q, ni):
    failures = 0
    for seed in range(300):
        try:
            run_tiles(48, ring_s, ring_q, ni, seed)
        except Violation:
            failures += 1
    assert failures > 0
