"""The C-ABI library loads on a machine without a GPU, exports every entry point
declared in include/vca.h, and rejects bad arguments synchronously (before any
CUDA call) with the documented status codes."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_attention_video_smooth_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    src = open(os.path.join(ROOT, "include", "vca.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vca_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "vca_group" in names and "vca_prep_quant" in names and "vca_attention" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_lists_every_export():
    from bit_attention_video_smooth_gb300 import vca
    assert sorted(vca.EXPORTS) == _declared()


def test_status_strings_and_version(lib):
    lib.vca_status_string.restype = ctypes.c_char_p
    assert lib.vca_status_string(0) == b"ok"
    assert lib.vca_status_string(4) == b"device wait timed out"
    assert lib.vca_status_string(99) == b"unknown status"
    assert lib.vca_version() >= 100


def test_workspace_sizes(lib):
    lib.vca_workspace_bytes.restype = ctypes.c_size_t
    ws = lib.vca_workspace_bytes
    assert ws(0, 1, 40, 70656, 128, 64, 0) > 0
    assert ws(1, 1, 40, 70656, 128, 1, 0) > 0
    assert ws(0, 1, 2, 1000, 128, 8, 0) == 0        # N not a multiple of 128
    assert ws(0, 1, 2, 1024, 64, 8, 0) == 0         # d != 128
    assert ws(0, 1, 2, 1024, 128, 0, 0) == 0        # k < 1
    assert ws(0, 1, 2, 1024, 128, 129, 0) == 0      # k above the supported maximum
    assert ws(2, 1, 2, 1024, 128, 8, 0) == 0        # attention needs no workspace
    assert ws(0, 1, 65535, 128, 128, 8, 0) > 0      # B*H at the grid limit
    assert ws(0, 256, 256, 128, 128, 8, 0) == 0     # B*H = 65,536: one past it
    assert ws(0, 1, 16, 1 << 27, 128, 8, 0) == 0    # B*H*N = 2^31 tokens
    assert ws(0, 0, 2, 1024, 128, 8, 0) == 0        # empty batch
    assert ws(1, 1, 2, 0, 128, 8, 0) == 0           # empty sequence
    # K smoothing adds the block sums (512 B a block) and the mean (512 B a head)
    assert ws(3, 1, 2, 1024, 128, 1, 0) == ws(1, 1, 2, 1024, 128, 1, 0) + 2 * 8 * 512 + 2 * 512


def test_invalid_arguments_rejected_without_cuda(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)                                  # aligned, never dereferenced
    lib.vca_attention.argtypes = [P] * 8 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, P, P, P]
    # null output pointer
    assert lib.vca_attention(*([fake] * 8), 1, 2, 1024, 128, 0.0, 1, 0, None, None, None) == 1
    # ragged N
    assert lib.vca_attention(*([fake] * 8), 1, 2, 1000, 128, 0.0, 1, 0, fake, None, None) == 1
    # misaligned pointer
    assert lib.vca_attention(P(0x10001), *([fake] * 7), 1, 2, 1024, 128, 0.0, 1, 0, fake, None, None) == 1
    # B*H beyond the grid limit, and an empty sequence
    assert lib.vca_attention(*([fake] * 8), 256, 256, 1024, 128, 0.0, 1, 0, fake, None, None) == 1
    assert lib.vca_attention(*([fake] * 8), 1, 2, 0, 128, 0.0, 1, 0, fake, None, None) == 1
    # ExpCast has no NVFP4 counterpart
    assert lib.vca_attention(*([fake] * 8), 1, 2, 1024, 128, 0.0, 1, 1, fake, None, None) == 2
    # K smoothing wants its larger workspace: the plain prep's size is rejected before any launch
    lib.vca_workspace_bytes.restype = ctypes.c_size_t
    lib.vca_prep_quant_ex.argtypes = [P] * 4 + [ctypes.c_int] * 5 + [ctypes.c_uint32] + [P] * 9 + \
        [ctypes.c_size_t, P]
    plain_ws = lib.vca_workspace_bytes(1, 1, 2, 1024, 128, 1, 0)
    assert lib.vca_prep_quant_ex(*([fake] * 4), 1, 2, 1024, 128, 0, 2, *([fake] * 9), plain_ws, None) == 5
    lib.vca_group.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              ctypes.c_int, P, P, P, P, P, ctypes.c_size_t, P, P]
    assert lib.vca_group(fake, 1, 2, 1024, 128, 8, 0, fake, fake, None, None, fake, 1 << 30, None, None) == 1  # iters
    assert lib.vca_group(fake, 1, 2, 1024, 128, 200, 4, fake, fake, None, None, fake, 1 << 30, None, None) == 1  # k
    assert lib.vca_group(fake, 1, 2, 1024, 128, 8, 4, fake, fake, None, None, None, 0, None, None) == 5    # no ws
    assert lib.vca_group(fake, 1, 2, 1024, 128, 8, 4, fake, fake, None, None, fake, 16, None, None) == 5   # too small
    assert lib.vca_group(fake, 1, 2, 1024, 128, 8, 4, fake, fake, None, None, fake, 1 << 30, P(0x10002),
                         None) == 1                                                                       # status
    lib.vca_selftest_timeout.argtypes = [P, ctypes.c_uint64, P]
    assert lib.vca_selftest_timeout(fake, 10, None) == 1
    # prep option flags: VCA_PREP_QK_HADAMARD (bit 0) and VCA_PREP_K_SMOOTH (bit 1) are defined
    lib.vca_prep_quant_ex.argtypes = [P, P, P, P] + [ctypes.c_int] * 5 + [ctypes.c_uint32] + [P] * 8 + \
        [P, ctypes.c_size_t, P]
    assert lib.vca_prep_quant_ex(*([fake] * 4), 1, 2, 1024, 128, 0, 4, *([fake] * 8), fake, 1 << 30, None) == 1
    assert lib.vca_prep_quant_ex(*([fake] * 4), 1, 2, 1000, 128, 0, 1, *([fake] * 8), fake, 1 << 30, None) == 1
    assert lib.vca_prep_quant_ex(*([fake] * 4), 1, 2, 1024, 128, 0, 1, *([fake] * 8), None, 0, None) == 5


def test_oracle_and_library_share_no_code():
    # the oracle is plain C compiled by gcc; the library is CUDA compiled by nvcc;
    # neither includes the other's files
    orc = open(os.path.join(ROOT, "oracle", "vca_oracle.c")).read()
    assert "#include \"" not in orc
    csrc = os.path.join(ROOT, "bit_attention_video_smooth_gb300", "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert "oracle" not in text.lower(), f
    binding = open(os.path.join(ROOT, "bit_attention_video_smooth_gb300", "vca.py")).read()
    assert "import oracle" not in binding and "from oracle" not in binding


def test_header_compiles_as_c_and_links(lib, tmp_path):
    """A plain C99 program includes include/vca.h, links libvca.so and makes
    the calls that need no GPU (tests/c/abi_consumer.c)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from bit_attention_video_smooth_gb300 import build
    libdir = os.path.dirname(build.build())
    exe = str(tmp_path / "abi_consumer")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_consumer.c"), "-L", libdir, "-lvca",
                    f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok  ") == 10
