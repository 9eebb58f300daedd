"""A model of the E4M3 attention kernel's reference-max hand-over, checked on
the CPU.

In the kernel two softmax warps share each TMEM lane quarter: the warp of
parity 0 takes key blocks 0, 2, 4, ..., the warp of parity 1 blocks 1, 3, 5, ...
The reference max is sequential over blocks, so at block b a warp first waits
on a 64-thread named barrier for its partner's arrival from block b-1 (bar.sync,
b >= 1), reads the max the partner left in shared-memory slot (b-1) & 1, then
writes its own into slot b & 1 and arrives on its own barrier (bar.arrive)
when a block b+1 exists.  A warp whose wait for S(b) timed out, or whose
partner handed on NaN, hands on NaN and leaves the loop; a warp whose PV wait
timed out carries on to its next block and gives up there.  All eight softmax
warps then meet at a barrier that ANDs their status: the epilogue runs only if
every warp finished.

What must hold on every schedule and every pattern of give-ups:
  * no deadlock: every bar.sync is matched by an arrival;
  * a named barrier never holds two pending arrivals from one warp (a second
    bar.arrive before the partner's bar.sync would complete the barrier's
    current generation without the partner);
  * a shared-memory slot is never overwritten before the partner read it;
  * a clean run (no give-ups) leaves no pending arrival and both warps finish;
  * if any wait gave up, the epilogue is skipped.
"""
import itertools
import random

import pytest


class Deadlock(Exception):
    pass


def _warp(par, nb, fail_s, fail_pv, st):
    """One softmax warp as a generator: yields "wait" while its bar.sync has no
    arrival to consume, "step" after every other action."""
    ok = True
    for b in range(par, nb, 2):
        wok = ok and b not in fail_s                       # the wait for S(b)
        partner_nan = False
        if b >= 1:
            while not st["arrivals"][par ^ 1]:
                yield "wait"
            st["arrivals"][par ^ 1].pop()
            slot = (b - 1) & 1
            assert st["unread"][slot], ("read of a slot nobody wrote", par, b)
            st["unread"][slot] = False
            partner_nan = st["value"][slot]
            yield "step"
        valid = wok and not partner_nan
        if b + 1 < nb:
            assert not st["arrivals"][par], ("second pending arrival", par, b)
            assert not st["unread"][b & 1], ("slot overwritten before it was read", par, b)
            st["value"][b & 1] = not valid                 # NaN marks a give-up
            st["unread"][b & 1] = True
            st["arrivals"][par].append(True)
            yield "step"
        if not valid:
            ok = False
            break
        if b in fail_pv:                                   # the PV or rescale wait timed out
            ok = False
        yield "step"
    st["ok"][par] = ok


def run_protocol(nb, fail_s, fail_pv, rng, warp=_warp):
    st = {"arrivals": {0: [], 1: []}, "unread": [False, False], "value": [False, False], "ok": [None, None]}
    gens = {p: warp(p, nb, fail_s, fail_pv, st) for p in (0, 1)}
    waiting = set()
    while gens:
        p = rng.choice(sorted(gens))
        try:
            r = next(gens[p])
        except StopIteration:
            del gens[p]
            waiting.discard(p)
            continue
        if r == "wait":
            waiting.add(p)
            if waiting == set(gens):
                raise Deadlock((nb, sorted(fail_s), sorted(fail_pv)))
        else:
            waiting.clear()
    return st


def _check(nb, fail_s, fail_pv, rng):
    st = run_protocol(nb, fail_s, fail_pv, rng)
    epilogue = all(st["ok"])                               # the AND over the softmax warps
    if not fail_s and not fail_pv:
        assert epilogue, nb
        assert not st["arrivals"][0] and not st["arrivals"][1], ("leftover arrival on a clean run", nb)
    else:
        assert not epilogue, (nb, fail_s, fail_pv)


@pytest.mark.parametrize("nb", range(1, 7))
def test_every_give_up_pattern_small(nb):
    rng = random.Random(nb)
    blocks = range(nb)
    subsets = [set(c) for r in range(nb + 1) for c in itertools.combinations(blocks, r)]
    for fail_s in subsets:
        for fail_pv in subsets:
            for _ in range(3):
                _check(nb, fail_s, fail_pv, rng)


def test_random_give_ups_up_to_44_blocks():
    rng = random.Random(7)
    for nb in range(1, 45):
        for trial in range(600):
            rate = 0.0 if trial < 20 else 0.02                # clean runs under 20 schedules first
            fail_s = {b for b in range(nb) if rng.random() < rate}
            fail_pv = {b for b in range(nb) if rng.random() < rate}
            _check(nb, fail_s, fail_pv, rng)


def test_the_model_catches_a_broken_protocol():
    """Variants of the protocol with one rule dropped must fail the checks: a
    check that nothing can trip would prove nothing."""
    def arrive_always(par, nb, fail_s, fail_pv, st):
        # publishes even when no block b+1 exists
        for b in range(par, nb, 2):
            if b >= 1:
                while not st["arrivals"][par ^ 1]:
                    yield "wait"
                st["arrivals"][par ^ 1].pop()
            assert not st["arrivals"][par], ("second pending arrival", par, b)
            st["arrivals"][par].append(True)
            yield "step"
        st["ok"][par] = True

    def leave_silently(par, nb, fail_s, fail_pv, st):
        # gives up without handing NaN on
        for b in range(par, nb, 2):
            if b >= 1:
                while not st["arrivals"][par ^ 1]:
                    yield "wait"
                st["arrivals"][par ^ 1].pop()
            if b in fail_s:
                st["ok"][par] = False
                return
            if b + 1 < nb:
                st["arrivals"][par].append(True)
            yield "step"
        st["ok"][par] = True

    rng = random.Random(1)
    st = run_protocol(3, set(), set(), rng, warp=arrive_always)
    assert st["arrivals"][0] or st["arrivals"][1]          # the clean-run check fails
    with pytest.raises(Deadlock):
        run_protocol(4, {1}, set(), rng, warp=leave_silently)
