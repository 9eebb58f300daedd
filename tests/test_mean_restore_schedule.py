"""A model of the attention kernels' mean-restore schedule (the 8-bit and the
4-bit kernel share it), checked on the CPU for every block count up to 600.

Per query row the kernel keeps each key block's row sum in a ring of kRsSlots
shared-memory slots (block j in slot j % kRsSlots): the thread of the block's
parity writes it at block j + 2, once PV(j) is done.  After PV(b), for every b
with flush_after(b), one MMA adds the terms of blocks b - kMeanJ - kMeanLag ..
b - kMeanLag - 1, staged by the thread of block b; the blocks after the last
such range (the tail) are added in the epilogue by one more MMA group, two
when the tail is longer than kMeanJ.  What must hold:
  * the MMA ranges and the epilogue's tail cover every block exactly once;
  * every row sum an MMA stages is visible to the staging thread: its own
    parity's sums were written by itself earlier, the partner's before a
    reference-max hand-over that thread has already received;
  * no slot is overwritten while its entry is still to be read (by a later MMA
    or the epilogue);
  * the epilogue's tail fits the two operand groups it is staged into.
The constants and the flush rule are read from the kernel source, so the model
follows the kernel.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_attention_video_smooth_gb300", "csrc")


def _const(text, name):
    m = re.search(rf"constexpr\s+(?:int|uint32_t)\s+{name}\s*=\s*(\d+)\s*;", text)
    assert m, name
    return int(m.group(1))


@pytest.fixture(scope="module", params=["vca_attention.cu", "vca_attention_fp4.cu"])
def K(request):
    """The schedule as the shared header defines it, checked to be the one each
    kernel (8-bit and 4-bit) follows."""
    common = open(os.path.join(CSRC, "vca_attention_common.cuh")).read()
    kern = open(os.path.join(CSRC, request.param)).read()
    # the rules the model restates, as the kernels write them
    assert "return b >= kMeanJ + kMeanLag && (b % kMeanJ) == kMeanLag;" in common
    assert "const int bf = nb - 1 >= kMeanJ + kMeanLag ? kMeanLag + kMeanJ * ((nb - 1 - kMeanLag) / kMeanJ) : -1;" in kern
    assert "const int tail0 = bf >= 0 ? bf - kMeanLag : 0;" in kern
    assert "const int b0 = b - kMeanJ - kMeanLag;" in kern
    assert "stage_means(row, sRS, sRSM, m_new, b0," in kern
    assert "if (flush_after(j))" in kern and "if (ok && flush_after(b))" in kern
    assert "ok = restore_tail_means(par, row, warp == 2 && lane == 0, sRS, sRSM, mf, tail0, nb - tail0," in kern
    assert "const int n0 = rs_cnt < kMeanJ ? rs_cnt : kMeanJ, n1 = rs_cnt - n0;" in common
    return {"J": _const(common, "kMeanJ"), "L": _const(common, "kMeanLag"), "S": _const(common, "kRsSlots"),
            "blk": 128, "d": 128, "tile_bytes": 128 * 128}


def flush_after(K, b):
    return b >= K["J"] + K["L"] and b % K["J"] == K["L"]


def schedule(K, nb):
    """(flushes: list of (b, first block, last block)), tail0 of the epilogue."""
    J, L = K["J"], K["L"]
    flushes = [(b, b - J - L, b - L - 1) for b in range(nb) if flush_after(K, b)]
    bf = L + J * ((nb - 1 - L) // J) if nb - 1 >= J + L else -1
    tail0 = bf - L if bf >= 0 else 0
    return flushes, tail0


@pytest.mark.parametrize("chunk", range(6))
def test_every_block_is_restored_exactly_once(K, chunk):
    for nb in range(1 + 100 * chunk, 101 + 100 * chunk):
        flushes, tail0 = schedule(K, nb)
        covered = [j for _, lo, hi in flushes for j in range(lo, hi + 1)] + list(range(tail0, nb))
        assert sorted(covered) == list(range(nb)), nb
        for b, lo, hi in flushes:
            assert hi - lo + 1 == K["J"] and lo >= 0 and b < nb
        # the last range ends where the tail starts
        if flushes:
            assert flushes[-1][2] + 1 == tail0


def test_staged_sums_are_visible_to_the_staging_thread(K):
    """Block j's sum is written by the thread of parity j % 2 at its block
    j + 2; a thread receives its partner's hand-over of block p at its own
    block p + 1, and the partner wrote everything of its blocks <= p - 2 before
    that hand-over (the sum of block j is written at block j + 2, after that
    block's own hand-over)."""
    for nb in range(1, 400):
        flushes, _ = schedule(K, nb)
        for b, lo, hi in flushes:
            for j in range(lo, hi + 1):
                if j % 2 == b % 2:
                    assert j + 2 <= b - 2, (nb, b, j)          # written by this thread at an earlier block
                else:
                    # written by the partner at block j + 2, before its hand-over at
                    # block j + 4, which this thread took at block j + 5 <= b
                    assert j + 5 <= b, (nb, b, j)


def test_no_ring_slot_is_overwritten_before_it_is_read(K):
    S = K["S"]
    for nb in range(1, 400):
        flushes, tail0 = schedule(K, nb)
        read_at = {}                                        # block j -> the block whose staging reads it
        for b, lo, hi in flushes:
            for j in range(lo, hi + 1):
                read_at[j] = b
        for j in range(tail0, nb):
            read_at[j] = nb + 1                             # the epilogue, after every block
        for j in range(nb):
            later = j + S                                   # the next entry in the same slot
            if later >= nb:
                continue
            # that entry is written by the thread of parity j % 2 at its block
            # later + 2 (or in the epilogue, later still); the read of j must
            # come first.  A read by the same thread needs an earlier block; a
            # read by the partner at its block r is ordered before the write only
            # through the partner's hand-over at block r + 2, which the writer
            # takes at block r + 3.
            r = read_at[j]
            assert r <= nb - 1, (nb, j)                     # tail entries never have a later one
            if r % 2 == j % 2:
                assert r < later + 2, (nb, j, r)
            else:
                assert r + 3 <= later + 2, (nb, j, r)


def test_epilogue_tail_fits_its_staging(K):
    worst = 0
    for nb in range(1, 600):
        _, tail0 = schedule(K, nb)
        worst = max(worst, nb - tail0)
        # the tail starts a means group (its first kMeanJ blocks share one
        # group buffer, the rest the next one) and both its groups are the
        # last two loaded, so neither buffer has been refilled
        assert tail0 % K["J"] == 0, nb
        assert (nb - 1) // K["J"] - tail0 // K["J"] <= 1, nb
    # the tail is staged as at most two operand groups of kMeanJ blocks
    assert worst <= 2 * K["J"], worst
    assert worst <= K["S"]
    assert worst == K["J"] + K["L"]
