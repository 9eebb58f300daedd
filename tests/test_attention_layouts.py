"""The attention kernels' TMEM column plans and shared-memory layouts, read
from their sources and checked on the CPU.

Both kernels hold S0, S1, the accumulator O, two row-sum slots E0/E1, two P
buffers and Q in the 512 TMEM columns of one CTA (the 4-bit kernel also the
scale factors of its block-scaled MMAs).  The 8-bit kernel's PV MMA of an even
block writes N = 144 columns [E0 | O] and of an odd block [O | E1], so those
pairs must be contiguous; nothing may overlap.  Shared-memory tiles read by the tensor core
with the 128-byte swizzle start on 1024-byte boundaries, mbarriers on 8-byte
ones, and the whole layout fits the 227 KB a CTA may use.
"""
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bit_attention_video_smooth_gb300",
                    "csrc")


def constants(*files):
    """Namespace-level integer constexprs of the files, evaluated in order."""
    env = {}
    for f in files:
        text = open(os.path.join(CSRC, f)).read()
        for m in re.finditer(r"^constexpr\s+(?:int|uint32_t)\s+([^;]*);", text, flags=re.M):
            for part in m.group(1).split(","):
                name, _, expr = part.partition("=")
                expr = re.sub(r"//.*", "", expr).replace("/", "//").strip()
                expr = re.sub(r"\b(\d+)u\b", r"\1", expr)   # unsigned literals
                try:
                    env[name.strip()] = int(eval(expr, {"__builtins__": {}}, dict(env)))
                except (NameError, SyntaxError):
                    pass
    return env


def _disjoint(ranges, total):
    spans = sorted(ranges.values())
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0, ranges
    assert spans[0][0] >= 0 and spans[-1][1] <= total, ranges


@pytest.fixture(scope="module")
def e4m3():
    return constants("vca_device.cuh", "vca_attention_common.cuh", "vca_attention.cu")


@pytest.fixture(scope="module")
def nvfp4():
    return constants("vca_device.cuh", "vca_attention_common.cuh", "vca_attention_fp4.cu")


def test_e4m3_tmem_plan(e4m3):
    c = e4m3
    cols = {"S0": (0, 128), "S1": (128, 256), "E0": (c["kTmemE0"], c["kTmemE0"] + 16),
            "O": (c["kTmemO"], c["kTmemO"] + 128), "E1": (c["kTmemE1"], c["kTmemE1"] + 16),
            "P0": (c["kTmemP0"], c["kTmemP0"] + 32), "P1": (c["kTmemP0"] + 32, c["kTmemP0"] + 64),
            "Q": (c["kTmemQ"], c["kTmemQ"] + 32)}
    _disjoint(cols, c["kTmemCols"])
    assert c["kTmemCols"] == 512
    assert c["kTmemE0"] + 16 == c["kTmemO"] and c["kTmemO"] + 128 == c["kTmemE1"]     # [E0 | O], [O | E1]


def test_e4m3_shared_memory_layout(e4m3):
    c = e4m3
    assert c["kThreads"] == 384 and c["kTileBytes"] == 16384
    for s in range(c["kKStages"]):
        assert (c["kOffK"] + s * c["kTileBytes"]) % 1024 == 0
    for s in range(c["kVStages"]):
        stage = c["kOffV"] + s * c["kVStageBytes"]
        assert stage % 1024 == 0 and (stage + c["kOnesBytes"]) % 1024 == 0      # [ones ; V] and [V ; ones]
    assert c["kOffMA"] % 1024 == 0 and c["kOffMB"] % 1024 == 0
    assert c["kOffBar"] % 8 == 0
    assert c["kSmemBytes"] <= 232448
    # the regions follow one another without overlap
    order = ["kOffK", "kOffV", "kOffMA", "kOffMB", "kOffMean", "kOffRS", "kOffRSM", "kOffSV", "kOffMX", "kOffL",
             "kOffBar", "kOffMisc"]
    offs = [c[k] for k in order]
    assert offs == sorted(offs)
    # the means of two 16-block groups: bulk-copy destinations (16-byte aligned)
    assert c["kOffMean"] % 16 == 0 and c["kOffRS"] - c["kOffMean"] == 2 * c["kMeanGroupBytes"]
    assert c["kMeanGroupBytes"] == c["kMeanJ"] * 128 * 2
    assert c["kOffRSM"] - c["kOffRS"] == c["kRsSlots"] * 128 * 4
    # one mbarrier each: q_full, K and V full/empty rings, s_full, s_free, p_full, pv_done, drain (two each),
    # the epilogue's tail MMAs
    assert c["kNumBars"] == 1 + 2 * c["kKStages"] + 2 * c["kVStages"] + 2 * 5 + 1


def test_nvfp4_tmem_plan(nvfp4):
    """The 4-bit kernel's columns: two P buffers as E2M1 codes (128 keys at
    eight per column), their scales (per parity two MMAs x four lane-quarter
    columns), two V-scale buffers (per parity two MMAs x four columns, filled
    in every lane quarter) and the ones rows' scale column, none overlapping S,
    O or the row-sum slots (Q is QK's A operand from shared memory here)."""
    c = nvfp4
    cols = {"S0": (0, 128), "S1": (128, 256), "O": (c["kTmemO"], c["kTmemO"] + 128),
            "E0": (c["kTmemE0"], c["kTmemE0"] + 16), "E1": (c["kTmemE0"] + 16, c["kTmemE0"] + 32),
            "P0": (c["kTmemP0"], c["kTmemP0"] + 128 // 8), "P1": (c["kTmemP0"] + 16, c["kTmemP0"] + 32),
            "SFA0": (c["kTmemSFA0"], c["kTmemSFA0"] + 2 * 4), "SFA1": (c["kTmemSFA0"] + 8, c["kTmemSFA0"] + 16),
            "SFB0": (c["kTmemSFB"], c["kTmemSFB"] + 2 * 4), "SFB1": (c["kTmemSFB"] + 8, c["kTmemSFB"] + 16),
            "SF1": (c["kTmemSF1"], c["kTmemSF1"] + 1)}
    _disjoint(cols, c["kTmemCols"])
    # the row-sum MMA writes N = 16 columns into a slot of 16
    assert c["kOnesRows"] == 16
    # mbarriers for Q, the K ring, the V ring (landed, laid out, released),
    # S / P / PV per parity, the two issuers' drains and the epilogue's tail MMAs
    assert c["kNumBars"] == 1 + 2 * c["kKStages"] + 3 * c["kVStages"] + 2 * 5 + 1


def test_nvfp4_shared_memory_layout(nvfp4):
    c = nvfp4
    assert c["kThreads"] == 384
    # a V stage: the block's codes as TMA writes them with the 64-byte swizzle
    # (128 channel rows of 64 bytes, 512-byte atoms), its raw scales and the two
    # 32-row x 16-byte matrices the PV issuer copies into TMEM
    assert c["kVStageBytes"] == 128 * 64 + 1024 + 2 * 512
    for s in range(c["kVStages"]):
        st = c["kOffV"] + s * c["kVStageBytes"]
        assert st % 1024 == 0                                                  # swizzle atoms
        assert (st + c["kCodeBytes"]) % 16 == 0                                # bulk-copy destination
        assert (st + c["kCodeBytes"] + c["kSfBytes"]) % 16 == 0                # scale-copy source
    assert c["kOffOnes"] % 1024 == 0 and c["kOnesBytes"] == 16 * 128
    assert c["kOffMA"] % 1024 == 0 and c["kOffMB"] % 1024 == 0
    assert c["kOffBar"] % 8 == 0 and c["kSmemBytes"] <= 232448
    assert c["kOffQ"] % 1024 == 0 and c["kOffV"] >= c["kOffQ"] + 128 * 128   # the swizzled Q tile
    order = ["kOffK", "kOffQ", "kOffV", "kOffOnes", "kOffMA", "kOffMB", "kOffMean", "kOffRS", "kOffRSM", "kOffSV",
             "kOffMX", "kOffL", "kOffLg", "kOffBar", "kOffMisc"]
    offs = [c[k] for k in order]
    assert offs == sorted(offs)
    # the V loads run ahead by all stages but the one being laid out
    assert c["kVAhead"] == c["kVStages"] - 1


def test_the_evaluator_reads_the_sources(e4m3, nvfp4):
    """Guard against a silent parse failure: the constants the checks use exist
    and have the values the kernels' comments state."""
    assert e4m3["kBlk"] == 128 and e4m3["kD"] == 128 and e4m3["kMeanJ"] == 16 and e4m3["kRsSlots"] == 32
    assert e4m3["kOnesBytes"] == 2048 and e4m3["kVStageBytes"] == 2048 + 16384 + 2048
    assert nvfp4["kCodeBytes"] == 8192 and nvfp4["kSfBytes"] == 1024 and nvfp4["kOnesBytes"] == 2048
