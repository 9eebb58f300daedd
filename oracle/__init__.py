"""CPU oracle for the VC-Attention hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it, and shares no code with it.

The arithmetic lives in ``vca_oracle.c`` (plain C, fp64 where the method does
not fix a precision, compiled with ``-ffp-contract=off``).  This module compiles
it with gcc on first use and wraps it for numpy arrays.  Each function cites the
passage of the method it follows; see the C file for the readings taken where
the pages are silent.

Parity pins for every function are in ``tests/test_oracle_*.py`` (the QK
Hadamard option of ``prep`` and ``fwht_f32`` in ``test_oracle_hadamard.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vca_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liborc.so")
_lock = threading.Lock()
_lib = None

P_EXPCAST, P_EXP, P_NVFP4, P_EXACT = 0, 1, 2, 3
V_E4M3, V_NVFP4 = 0, 1
BLK = 128


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liborc.so`` (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
            sig = {
                "orc_threads": (ctypes.c_int, []),
                "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
                "orc_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "orc_e2m1_encode": (ctypes.c_uint8, [ctypes.c_double]),
                "orc_bf16_round": (ctypes.c_uint16, [ctypes.c_double]),
                "orc_e4m3_encode_f32": (None, [P, i64, P]),
                "orc_e4m3_encode_bits": (None, [ctypes.c_uint32, i64, P]),
                "orc_e2m1_encode_f32": (None, [P, i64, P]),
                "orc_expcast_codes": (None, [P, P, P, i64, P]),
                "orc_exp_codes": (None, [P, P, P, i64, P]),
                "orc_stable_sort": (None, [P, i32, i32, i32, P, P]),
                "orc_kmeans": (None, [P, i32, i32, i32, i32, i32, P, P, P]),
                "orc_kmeans_sse": (ctypes.c_double, [P, i32, i32, P, P]),
                "orc_prep": (i32, [P, P, P, P, i32, i32, i32, i32,
                                   P, P, P, P, P, P, P, P]),
                "orc_prep_ex": (i32, [P, P, P, P, i32, i32, i32, i32, ctypes.c_uint,
                                      P, P, P, P, P, P, P, P]),
                "orc_fwht_f32": (None, [P, i32]),
                "orc_k_channel_mean": (None, [P, P, i32, i32, P]),
                "orc_attention": (i32, [P, P, P, P, P, P, P, P, i32, i32, i32, f32, f32, i32, i32,
                                        P, i32, P, P]),
                "orc_attention_exact": (i32, [P, P, P, i32, i32, i32, f32, P, i32, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    """Threads the oracle's parallel loops use in this process."""
    return int(_load().orc_threads())


# ---------------------------------------------------------------------------
# Formats (OCP 8-bit float and microscaling specifications)
# ---------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 byte (fp64); 0x7F/0xFF decode to NaN."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(x)) for x in c.ravel()]).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even E4M3 with saturation to +-448 (fp32 inputs)."""
    lib = _load()
    a = _c(x, np.float32)
    out = np.empty(a.shape, np.uint8)
    lib.orc_e4m3_encode_f32(_p(a), a.size, _p(out))
    return out


def e4m3_encode_bits(start: int, count: int) -> np.ndarray:
    """E4M3 encodings of the fp32 bit patterns start .. start+count-1."""
    lib = _load()
    out = np.empty(count, np.uint8)
    lib.orc_e4m3_encode_bits(ctypes.c_uint32(start), count, _p(out))
    return out


def e2m1_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e2m1_decode(int(x)) for x in c.ravel()]).reshape(c.shape)


def e2m1_encode(x) -> np.ndarray:
    """Round-to-nearest-even E2M1 (4-bit code in the low nibble), saturating at 6."""
    lib = _load()
    a = _c(x, np.float32)
    out = np.empty(a.shape, np.uint8)
    lib.orc_e2m1_encode_f32(_p(a), a.size, _p(out))
    return out


def bf16_round(x: float) -> int:
    return int(_load().orc_bf16_round(float(x)))


# ---------------------------------------------------------------------------
# ExpCast-FP8 (paper page "method"; news page "ExpCast-FP8")
# ---------------------------------------------------------------------------
def expcast_codes(s_raw, c, m) -> np.ndarray:
    """E4M3 byte of p = 2^(s_raw*c - m) written by one fp32 FMA:
    code = rne(fma(s_raw, 8c, 56 + beta - 8m)), beta = -0.35; codes below 8
    flush to 0, codes above 126 clip to 126."""
    lib = _load()
    s = _c(s_raw, np.float32)
    cc = _c(np.broadcast_to(c, s.shape), np.float32)
    mm = _c(np.broadcast_to(m, s.shape), np.float32)
    out = np.empty(s.shape, np.uint8)
    lib.orc_expcast_codes(_p(s), _p(cc), _p(mm), s.size, _p(out))
    return out


def exp_codes(s_raw, c, m) -> np.ndarray:
    """The conventional path: p = 2^(fma(s_raw, c, -m)), then E4M3 RNE."""
    lib = _load()
    s = _c(s_raw, np.float32)
    cc = _c(np.broadcast_to(c, s.shape), np.float32)
    mm = _c(np.broadcast_to(m, s.shape), np.float32)
    out = np.empty(s.shape, np.uint8)
    lib.orc_exp_codes(_p(s), _p(cc), _p(mm), s.size, _p(out))
    return out


# ---------------------------------------------------------------------------
# V-Smooth group: k-means + stable permutation (paper page "method")
# ---------------------------------------------------------------------------
def kmeans(V: np.ndarray, k: int, iters: int):
    """Lloyd k-means per (b,h) on bf16 V [BH, N, d] (uint16 bit patterns).

    Returns (labels int32 [BH,N], counts int32 [BH,k], centroids fp32 [BH,k,d]).
    """
    lib = _load()
    v = _c(V, np.uint16)
    BH, N, d = v.shape
    labels = np.empty((BH, N), np.int32)
    counts = np.empty((BH, k), np.int32)
    cent = np.empty((BH, k, d), np.float32)
    lib.orc_kmeans(_p(v), BH, N, d, k, iters, _p(labels), _p(counts), _p(cent))
    return labels, counts, cent


def stable_sort(labels: np.ndarray, k: int):
    """perm[i] = token placed in slot i, ordered by (label, original index)."""
    lib = _load()
    lab = _c(labels, np.int32)
    BH, N = lab.shape
    perm = np.empty((BH, N), np.int32)
    counts = np.empty((BH, k), np.int32)
    lib.orc_stable_sort(_p(lab), BH, N, k, _p(perm), _p(counts))
    return perm, counts


def kmeans_sse(V: np.ndarray, labels: np.ndarray, centroids: np.ndarray) -> float:
    lib = _load()
    v = _c(V, np.uint16)
    N, d = v.shape
    return float(lib.orc_kmeans_sse(_p(v), N, d, _p(_c(labels, np.int32)), _p(_c(centroids, np.float32))))


def group(V: np.ndarray, k: int, iters: int):
    """Full group step: (labels, perm, counts, centroids)."""
    labels, counts, cent = kmeans(V, k, iters)
    perm, counts2 = stable_sort(labels, k)
    assert np.array_equal(counts, counts2)
    return labels, perm, counts, cent


# ---------------------------------------------------------------------------
# Fused prep (paper page "method"; news page "V-Smooth" bullet "Demean")
# ---------------------------------------------------------------------------
PREP_QK_HADAMARD = 1
PREP_K_SMOOTH = 2


def k_channel_mean(K, perm) -> np.ndarray:
    """The channel mean of K over the sequence of each (b,h) that K smoothing
    subtracts (fp32, a fixed summation order: a halving tree per permuted
    128-token block, the block sums in block order, divided by N)."""
    lib = _load()
    k = _c(K, np.uint16)
    pm = _c(perm, np.int32)
    BH, N, d = k.shape
    out = np.empty((BH, d), np.float32)
    for bh in range(BH):
        row = np.empty(d, np.float32)
        lib.orc_k_channel_mean(_p(np.ascontiguousarray(k[bh])), _p(np.ascontiguousarray(pm[bh])), N, d, _p(row))
        out[bh] = row
    return out


def fwht_f32(x) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform of the last axis (a power of two)
    as fp32 butterflies, bit 0 first (the rounding the device reproduces)."""
    lib = _load()
    a = np.array(x, dtype=np.float32, copy=True)
    d = a.shape[-1]
    flat = a.reshape(-1, d)
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        lib.orc_fwht_f32(_p(row), d)
        flat[r] = row
    return flat.reshape(a.shape)


def prep(Q, K, V, perm, vmode: int = V_E4M3, qk_hadamard: bool = False, k_smooth: bool = False) -> dict:
    """Gather, block means, residual and Q/K quantisation for bf16 [BH,N,d].
    qk_hadamard: rotate Q and K rows by fwht_f32 before the FP8 quantisation;
    the key scales then carry the factor 1/d.  k_smooth: subtract the keys'
    channel mean (k_channel_mean) before that."""
    lib = _load()
    q, k, v = (_c(a, np.uint16) for a in (Q, K, V))
    pm = _c(perm, np.int32)
    BH, N, d = q.shape
    nb = N // BLK
    out = {
        "q8": np.empty((BH, N, d), np.uint8), "sq": np.empty((BH, nb), np.float32),
        "k8": np.empty((BH, N, d), np.uint8), "sk": np.empty((BH, nb), np.float32),
        "v_mean": np.empty((BH, nb, d), np.uint16),
    }
    if vmode == V_E4M3:
        out["v_res"] = np.empty((BH, nb, d, BLK), np.uint8)
        out["v_sf"] = None
        out["v_scale"] = np.empty((BH, d), np.float32)
    else:
        out["v_res"] = np.empty((BH, nb, d, BLK // 2), np.uint8)
        out["v_sf"] = np.empty((BH, nb, d, BLK // 16), np.uint8)
        out["v_scale"] = np.empty((BH,), np.float32)
    flags = (PREP_QK_HADAMARD if qk_hadamard else 0) | (PREP_K_SMOOTH if k_smooth else 0)
    rc = lib.orc_prep_ex(_p(q), _p(k), _p(v), _p(pm), BH, N, d, vmode, flags,
                         _p(out["q8"]), _p(out["sq"]), _p(out["k8"]), _p(out["sk"]),
                         _p(out["v_res"]), _p(out["v_sf"]), _p(out["v_scale"]), _p(out["v_mean"]))
    if rc:
        raise ValueError("oracle prep: N must be a multiple of 128 (and d a power of two with qk_hadamard)")
    return out


# ---------------------------------------------------------------------------
# Attention (paper page "method": online softmax, ExpCast, mean restore)
# ---------------------------------------------------------------------------
TAU = 8.0   # lazy-rescale threshold of the kernel (log2 units)


def attention(prepped: dict, mode: int, softmax_scale: float = 0.0, rows=None,
              return_l: bool = False, tau: float = TAU):
    """Schedule-emulating attention on prepared operands.

    mode: P_EXPCAST, P_EXP, P_NVFP4 or P_EXACT (P unquantised; a pin mode).
    The residual format (E4M3 or NVFP4) follows ``prepped`` (NVFP4 when it
    holds ``v_sf``).  tau: the reference max moves to a block's max only when
    that exceeds it by more than tau (FlashAttention-4's lazy rescale; 0 gives
    the plain running max).  rows: optional int array of query rows computed for every
    (b,h).  Returns bf16 O [BH, nrows, d] (uint16), optionally l.
    """
    lib = _load()
    q8 = prepped["q8"]
    BH, N, d = q8.shape
    r = None if rows is None else _c(rows, np.int32)
    nrows = N if r is None else r.size
    O = np.empty((BH, nrows, d), np.uint16)
    l = np.empty((BH, nrows), np.float64) if return_l else None
    rc = lib.orc_attention(_p(q8), _p(prepped["sq"]), _p(prepped["k8"]), _p(prepped["sk"]),
                           _p(prepped["v_res"]), _p(prepped.get("v_sf")), _p(prepped["v_scale"]),
                           _p(prepped["v_mean"]), BH, N, d, float(softmax_scale), float(tau), mode,
                           V_E4M3 if prepped.get("v_sf") is None else V_NVFP4,
                           _p(r), nrows, _p(O), _p(l))
    if rc:
        raise ValueError("oracle attention: N must be a multiple of 128")
    return (O, l) if return_l else O


def attention_exact(Q, K, V, softmax_scale: float = 0.0, rows=None) -> np.ndarray:
    """Exact fp64 softmax(Q K^T * scale) V on bf16 inputs; fp64 [BH, nrows, d]."""
    lib = _load()
    q, k, v = (_c(a, np.uint16) for a in (Q, K, V))
    BH, N, d = q.shape
    r = None if rows is None else _c(rows, np.int32)
    nrows = N if r is None else r.size
    O = np.empty((BH, nrows, d), np.float64)
    lib.orc_attention_exact(_p(q), _p(k), _p(v), BH, N, d, float(softmax_scale), _p(r), nrows, _p(O))
    return O


def bf16_to_f32(a) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 (exact)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
