"""Thin ctypes binding of ``libvca.so`` (the C ABI in ``include/vca.h``).

The functions keep the C entry points' names and only marshal arguments:
PyTorch tensors provide device memory and the current CUDA stream; every step
of the computation runs in the library's CUDA kernels.  If the library has not
been built (``__graft_entry__.build()`` or ``python
bit_attention_video_smooth_gb300/build.py``) importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvca.so")

VCA_OK, VCA_ERR_INVALID_ARG, VCA_ERR_UNSUPPORTED, VCA_ERR_CUDA, VCA_ERR_TIMEOUT, VCA_ERR_WORKSPACE = range(6)
VCA_V_E4M3, VCA_V_NVFP4 = 0, 1
VCA_OP_GROUP, VCA_OP_PREP, VCA_OP_ATTENTION, VCA_OP_PREP_KSMOOTH = 0, 1, 2, 3

# Entry points declared in include/vca.h (the ABI test checks they are exported).
EXPORTS = ("vca_status_string", "vca_version", "vca_workspace_bytes", "vca_group", "vca_prep_quant",
           "vca_attention", "vca_expcast_codes", "vca_e4m3_encode_bits", "vca_selftest_timeout",
           "vca_set_wait_limit_ns", "vca_prep_quant_noalloc", "vca_prep_quant_ex")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libvca.so is not built ({LIB_PATH}); run __graft_entry__.build() -- "
                      "there is no fallback implementation")

_lib = ctypes.CDLL(LIB_PATH)
_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "vca_status_string": (ctypes.c_char_p, [_I]),
    "vca_version": (_I, []),
    "vca_workspace_bytes": (_SZ, [_I] * 7),
    "vca_group": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "vca_prep_quant": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "vca_attention": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P]),
    "vca_expcast_codes": (_I, [_P, _P, _P, _I64, _P, _P]),
    "vca_e4m3_encode_bits": (_I, [ctypes.c_uint32, _I64, _P, _P]),
    "vca_selftest_timeout": (_I, [_P, ctypes.c_uint64, _P]),
    "vca_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "vca_prep_quant_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "vca_prep_quant_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_uint32, _P, _P, _P, _P, _P, _P, _P, _P,
                               _P, _SZ, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class VCAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {vca_status_string(status)} ({status})")


def vca_status_string(status: int) -> str:
    return _lib.vca_status_string(int(status)).decode()


def vca_version() -> int:
    return int(_lib.vca_version())


def vca_workspace_bytes(op: int, B: int, H: int, N: int, d: int = 128, k: int = 1, vmode: int = 0) -> int:
    return int(_lib.vca_workspace_bytes(op, B, H, N, d, k, vmode))


def vca_set_wait_limit_ns(limit_ns: int) -> None:
    _lib.vca_set_wait_limit_ns(int(limit_ns))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _buffers(where: str, need) -> torch.device:
    """The library sees plain pointers and cannot check what they point to, so
    the binding does: every (name, tensor, bytes) entry with a tensor must be
    contiguous and hold at least `bytes` bytes, and all of them must sit on one
    CUDA device, which is returned.  Sizes are checked first, so a call with
    host tensors of the right sizes fails only on the device check."""
    need = [(n, t, b) for n, t, b in need if t is not None]
    for name, t, nbytes in need:
        if not t.is_contiguous():
            raise ValueError(f"{where}: {name} must be contiguous")
        have = t.numel() * t.element_size()
        if have < nbytes:
            raise ValueError(f"{where}: {name} holds {have} bytes, {nbytes} needed")
    for name, t, _ in need:
        if not t.is_cuda:
            raise ValueError(f"{where}: {name} is not a CUDA tensor")
    devs = {t.device for _, t, _ in need}
    if len(devs) != 1:
        raise ValueError(f"{where}: tensors on several devices {sorted(str(d) for d in devs)}")
    return devs.pop()


def _stream(stream=None, device=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != VCA_OK:
        raise VCAError(status, where)


def _u16(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------
def vca_group(V: torch.Tensor, k: int, iters: int, labels: torch.Tensor, perm: torch.Tensor,
              counts: Optional[torch.Tensor], centroids: Optional[torch.Tensor], ws: torch.Tensor,
              dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    B, H, N, d = V.shape
    tok = B * H * N
    dev = _buffers("vca_group", [("V", V, 2 * tok * d), ("labels", labels, 4 * tok), ("perm", perm, 4 * tok),
                                 ("counts", counts, 4 * B * H * k), ("centroids", centroids, 4 * B * H * k * d),
                                 ("ws", ws, 0), ("dev_status", dev_status, 4)])
    with torch.cuda.device(dev):
        st = _lib.vca_group(_ptr(_u16(V)), B, H, N, d, k, iters, _ptr(labels), _ptr(perm), _ptr(counts),
                            _ptr(centroids), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
                            _stream(stream, dev))
    _check(st, "vca_group")


def vca_prep_quant(Q, K, V, perm, vmode: int, q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean, ws,
                   stream=None) -> None:
    B, H, N, d = Q.shape
    dev = _prep_buffers("vca_prep_quant", B, H, N, d, vmode, Q, K, V, perm, q8, sq, k8, sk, v_res, v_sf, v_scale,
                        v_mean, ws=ws)
    with torch.cuda.device(dev):
        st = _lib.vca_prep_quant(_ptr(_u16(Q)), _ptr(_u16(K)), _ptr(_u16(V)), _ptr(perm), B, H, N, d, vmode,
                                 _ptr(q8), _ptr(sq), _ptr(k8), _ptr(sk), _ptr(v_res), _ptr(v_sf), _ptr(v_scale),
                                 _ptr(_u16(v_mean)), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream, dev))
    _check(st, "vca_prep_quant")


VCA_PREP_QK_HADAMARD = 1
VCA_PREP_K_SMOOTH = 2


def _prep_buffers(where, B, H, N, d, vmode, Q, K, V, perm, q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean,
                  O=None, ws=None, dev_status=None):
    """Byte counts of the prep's inputs and outputs (the attention's operands)
    at this size and V format, checked against the tensors given."""
    BH, tok, nb = B * H, B * H * N, N // 128
    fp4 = vmode == VCA_V_NVFP4
    return _buffers(where, [
        ("Q", Q, 2 * tok * d), ("K", K, 2 * tok * d), ("V", V, 2 * tok * d), ("perm", perm, 4 * tok),
        ("q8", q8, tok * d), ("sq", sq, 4 * BH * nb), ("k8", k8, tok * d), ("sk", sk, 4 * BH * nb),
        ("v_res", v_res, tok * d // 2 if fp4 else tok * d), ("v_sf", v_sf, tok * d // 16 if fp4 else 0),
        ("v_scale", v_scale, 4 * BH if fp4 else 4 * BH * d), ("v_mean", v_mean, 2 * BH * nb * d),
        ("O", O, 2 * tok * d), ("ws", ws, 0), ("dev_status", dev_status, 4)])


def vca_prep_quant_ex(Q, K, V, perm, vmode: int, flags: int, q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean, ws,
                      stream=None) -> None:
    B, H, N, d = Q.shape
    dev = _prep_buffers("vca_prep_quant_ex", B, H, N, d, vmode, Q, K, V, perm, q8, sq, k8, sk, v_res, v_sf,
                        v_scale, v_mean, ws=ws)
    with torch.cuda.device(dev):
        st = _lib.vca_prep_quant_ex(_ptr(_u16(Q)), _ptr(_u16(K)), _ptr(_u16(V)), _ptr(perm), B, H, N, d, vmode,
                                    flags, _ptr(q8), _ptr(sq), _ptr(k8), _ptr(sk), _ptr(v_res), _ptr(v_sf),
                                    _ptr(v_scale), _ptr(_u16(v_mean)), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream, dev))
    _check(st, "vca_prep_quant_ex")


def vca_prep_quant_noalloc(Q, K, V, perm, vmode: int, q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean,
                           stream=None) -> None:
    """vca_prep_quant without a workspace argument: the scratch is a buffer built
    into the library (for callers that cannot provide device scratch memory).
    Calls that overlap on the GPU share that buffer and must be ordered."""
    B, H, N, d = Q.shape
    dev = _prep_buffers("vca_prep_quant_noalloc", B, H, N, d, vmode, Q, K, V, perm, q8, sq, k8, sk, v_res, v_sf,
                        v_scale, v_mean)
    with torch.cuda.device(dev):
        st = _lib.vca_prep_quant_noalloc(_ptr(_u16(Q)), _ptr(_u16(K)), _ptr(_u16(V)), _ptr(perm), B, H, N, d,
                                         vmode, _ptr(q8), _ptr(sq), _ptr(k8), _ptr(sk), _ptr(v_res), _ptr(v_sf),
                                         _ptr(v_scale), _ptr(_u16(v_mean)), _stream(stream, dev))
    _check(st, "vca_prep_quant_noalloc")


def vca_attention(q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean, B: int, H: int, N: int, d: int,
                  softmax_scale: float, expcast: int, vmode: int, O, dev_status=None, stream=None) -> None:
    dev = _prep_buffers("vca_attention", B, H, N, d, vmode, None, None, None, None, q8, sq, k8, sk, v_res, v_sf,
                        v_scale, v_mean, O=O, dev_status=dev_status)
    with torch.cuda.device(dev):
        st = _lib.vca_attention(_ptr(q8), _ptr(sq), _ptr(k8), _ptr(sk), _ptr(v_res), _ptr(v_sf), _ptr(v_scale),
                                _ptr(_u16(v_mean)), B, H, N, d, float(softmax_scale), int(expcast), int(vmode),
                                _ptr(_u16(O)), _ptr(dev_status), _stream(stream, dev))
    _check(st, "vca_attention")


def vca_expcast_codes(s_raw, c, m, out, stream=None) -> None:
    n = s_raw.numel()
    dev = _buffers("vca_expcast_codes", [("s_raw", s_raw, 4 * n), ("c", c, 4 * n), ("m", m, 4 * n), ("out", out, n)])
    with torch.cuda.device(dev):
        _check(_lib.vca_expcast_codes(_ptr(s_raw), _ptr(c), _ptr(m), n, _ptr(out), _stream(stream, dev)),
               "vca_expcast_codes")


def vca_e4m3_encode_bits(start: int, n: int, out, stream=None) -> None:
    dev = _buffers("vca_e4m3_encode_bits", [("out", out, n)])
    with torch.cuda.device(dev):
        _check(_lib.vca_e4m3_encode_bits(ctypes.c_uint32(start), n, _ptr(out), _stream(stream, dev)),
               "vca_e4m3_encode_bits")


def vca_selftest_timeout(dev_status, limit_ns: int, stream=None) -> None:
    dev = _buffers("vca_selftest_timeout", [("dev_status", dev_status, 4)])
    with torch.cuda.device(dev):
        _check(_lib.vca_selftest_timeout(_ptr(dev_status), ctypes.c_uint64(limit_ns), _stream(stream, dev)),
               "vca_selftest_timeout")


# ---------------------------------------------------------------------------
# Buffer sets and the whole path (allocation through PyTorch)
# ---------------------------------------------------------------------------
@dataclass
class Grouped:
    labels: torch.Tensor
    perm: torch.Tensor
    counts: torch.Tensor
    centroids: torch.Tensor
    ws: torch.Tensor


@dataclass
class Prepared:
    q8: torch.Tensor
    sq: torch.Tensor
    k8: torch.Tensor
    sk: torch.Tensor
    v_res: torch.Tensor
    v_sf: Optional[torch.Tensor]
    v_scale: torch.Tensor
    v_mean: torch.Tensor
    ws: torch.Tensor
    vmode: int


def alloc_group(B, H, N, k, device="cuda") -> Grouped:
    BH = B * H
    ws = torch.empty(max(16, vca_workspace_bytes(VCA_OP_GROUP, B, H, N, 128, k, 0)), dtype=torch.uint8, device=device)
    return Grouped(torch.empty((BH, N), dtype=torch.int32, device=device),
                   torch.empty((BH, N), dtype=torch.int32, device=device),
                   torch.empty((BH, k), dtype=torch.int32, device=device),
                   torch.empty((BH, k, 128), dtype=torch.float32, device=device), ws)


def alloc_prep(B, H, N, vmode=VCA_V_E4M3, device="cuda", k_smooth: bool = False) -> Prepared:
    BH, nb, d = B * H, N // 128, 128
    op = VCA_OP_PREP_KSMOOTH if k_smooth else VCA_OP_PREP
    ws = torch.empty(max(16, vca_workspace_bytes(op, B, H, N, d, 1, vmode)), dtype=torch.uint8, device=device)
    if vmode == VCA_V_E4M3:
        v_res = torch.empty((BH, nb, d, 128), dtype=torch.uint8, device=device)
        v_sf = None
        v_scale = torch.empty((BH, d), dtype=torch.float32, device=device)
    else:
        v_res = torch.empty((BH, nb, d, 64), dtype=torch.uint8, device=device)
        v_sf = torch.empty((BH, nb, d, 8), dtype=torch.uint8, device=device)
        v_scale = torch.empty((BH,), dtype=torch.float32, device=device)
    return Prepared(torch.empty((BH, N, d), dtype=torch.uint8, device=device),
                    torch.empty((BH, nb), dtype=torch.float32, device=device),
                    torch.empty((BH, N, d), dtype=torch.uint8, device=device),
                    torch.empty((BH, nb), dtype=torch.float32, device=device),
                    v_res, v_sf, v_scale,
                    torch.empty((BH, nb, d), dtype=torch.bfloat16, device=device), ws, vmode)


def group(V: torch.Tensor, k: int, iters: int, out: Optional[Grouped] = None,
          dev_status: Optional[torch.Tensor] = None) -> Grouped:
    B, H, N, _ = V.shape
    g = out or alloc_group(B, H, N, k, V.device)
    vca_group(V, k, iters, g.labels, g.perm, g.counts, g.centroids, g.ws, dev_status)
    return g


def prep_quant(Q, K, V, perm, vmode=VCA_V_E4M3, out: Optional[Prepared] = None,
               qk_hadamard: bool = False, k_smooth: bool = False) -> Prepared:
    B, H, N, _ = Q.shape
    p = out or alloc_prep(B, H, N, vmode, Q.device, k_smooth=k_smooth)
    flags = (VCA_PREP_QK_HADAMARD if qk_hadamard else 0) | (VCA_PREP_K_SMOOTH if k_smooth else 0)
    vca_prep_quant_ex(Q, K, V, perm, vmode, flags, p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale, p.v_mean,
                      p.ws)
    return p


def attention(p: Prepared, B: int, H: int, N: int, expcast: bool = True, softmax_scale: float = 0.0,
              out: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    O = out if out is not None else torch.empty((B, H, N, 128), dtype=torch.bfloat16, device=p.q8.device)
    vca_attention(p.q8, p.sq, p.k8, p.sk, p.v_res, p.v_sf, p.v_scale, p.v_mean, B, H, N, 128,
                  softmax_scale, int(expcast), p.vmode, O, dev_status)
    return O


def vc_attention(Q, K, V, k: int = 64, iters: int = 8, expcast: bool = True, vmode: int = VCA_V_E4M3,
                 softmax_scale: float = 0.0):
    """The whole hot path: group -> prep -> attention.  Returns (O, grouped, prepared)."""
    B, H, N, _ = Q.shape
    g = group(V, k, iters)
    p = prep_quant(Q, K, V, g.perm, vmode)
    O = attention(p, B, H, N, expcast=expcast, softmax_scale=softmax_scale)
    return O, g, p
