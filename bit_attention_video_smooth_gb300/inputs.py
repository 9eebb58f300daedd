"""Seeded synthetic inputs for the VC-Attention hot path.

This module only draws random numbers: it holds none of the method's arithmetic
and is the one piece of code shared by the CUDA path's tests and the CPU oracle.
It stands in for the video-DiT activations the method was measured on
(Wan2.2-14B self-attention: 5 s of 720p video, about 70K flattened tokens, 40
heads of width 128), which are not available here.

Recipe (every value drawn from a ``torch.Generator`` seeded with ``seed``, on
the requested device):
  * Q, K, V ~ N(0, 1), rounded to bf16 (round-to-nearest-even), layout
    [B, H, N, d] contiguous.
  * Q and K: per (batch, head) an independent set of ``qk_channels`` channels is
    multiplied by ``qk_mult`` (channel outliers; signs kept).
  * V: per (batch, head) a set of ``v_channels`` channels is drawn; a fraction
    ``v_frac`` of the tokens (drawn per head) is multiplied by ``v_mult`` on
    those channels (token outliers whose channels change from head to head).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int = 128
    k: int = 64
    iters: int = 8
    vmode: str = "e4m3"      # "e4m3" or "nvfp4"
    expcast: bool = True
    qk_channels: int = 4
    qk_mult: float = 8.0
    v_frac: float = 0.02
    v_mult: float = 16.0
    v_channels: int = 8
    sweep: tuple = field(default=())

    @property
    def BH(self) -> int:
        return self.B * self.H

    @property
    def flops(self) -> float:
        """4 B H N^2 d: the two contractions QK^T and PV."""
        return 4.0 * self.B * self.H * self.N * self.N * self.d


# The five workloads: tiny (oracle-sized), the Wan2.2-14B-shaped video
# self-attention with ExpCast, the same without ExpCast, the 4-bit V path, and
# the sequence-length sweep.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 1024, k=8, iters=10, qk_mult=10.0, v_frac=0.01, v_mult=20.0),
    "wan": Workload("wan", 1, 40, 70656, k=64, iters=8),
    "wan_exp": Workload("wan_exp", 1, 40, 70656, k=64, iters=8, expcast=False),
    "nvfp4": Workload("nvfp4", 2, 24, 32768, k=32, iters=8, vmode="nvfp4", expcast=False),
    "sweep": Workload("sweep", 1, 40, 70656, k=64, iters=8,
                      sweep=(4096, 16384, 32768, 70656, 131072)),
}


def with_n(w: Workload, N: int, H: int | None = None, B: int | None = None) -> Workload:
    """The same recipe at another sequence length (and optionally head count)."""
    from dataclasses import replace
    return replace(w, N=N, H=w.H if H is None else H, B=w.B if B is None else B,
                   name=f"{w.name}_N{N}")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_qkv(w: Workload, seed: int = 0, device="cpu"):
    """Q, K, V bf16 [B, H, N, d] following the recipe above."""
    g = _gen(seed, device)
    B, H, N, d = w.B, w.H, w.N, w.d
    out = []
    for which in ("q", "k", "v"):
        x = torch.randn((B, H, N, d), generator=g, device=device, dtype=torch.float32)
        x = x.view(B * H, N, d)
        if which in ("q", "k"):
            # per-head channel outliers
            sel = torch.rand((B * H, d), generator=g, device=device).argsort(dim=1)[:, : w.qk_channels]
            mult = torch.ones((B * H, d), device=device)
            mult.scatter_(1, sel, w.qk_mult)
            x.mul_(mult[:, None, :])
        else:
            n_out = max(1, int(round(w.v_frac * N)))
            ch = torch.rand((B * H, d), generator=g, device=device).argsort(dim=1)[:, : w.v_channels]
            tok = torch.rand((B * H, N), generator=g, device=device).argsort(dim=1)[:, :n_out]
            chmask = torch.zeros((B * H, d), device=device, dtype=torch.bool)
            chmask.scatter_(1, ch, True)
            tokmask = torch.zeros((B * H, N), device=device, dtype=torch.bool)
            tokmask.scatter_(1, tok, True)
            m = tokmask[:, :, None] & chmask[:, None, :]
            x = torch.where(m, x * w.v_mult, x)
        out.append(x.view(B, H, N, d).to(torch.bfloat16).contiguous())
    return tuple(out)


def make_separated_v(BH: int, N: int, d: int, k: int, seed: int = 0, device="cpu",
                     spread: float = 8.0, noise: float = 0.05) -> torch.Tensor:
    """bf16 V [BH, N, d] made of k well-separated clusters.

    Token j belongs to a cluster drawn at random, except that the tokens at the
    k strided positions floor((c + 1/2) N / k) are placed in cluster c, so every
    cluster holds one of those positions.  Cluster centres ~ N(0, spread^2),
    per-token noise ~ N(0, noise^2).
    """
    g = _gen(seed, device)
    centres = torch.randn((BH, k, d), generator=g, device=device) * spread
    lab = torch.randint(0, k, (BH, N), generator=g, device=device)
    pos = (torch.arange(k, device=device) * 2 + 1) * N // (2 * k)
    lab[:, pos] = torch.arange(k, device=device)
    x = torch.gather(centres, 1, lab[:, :, None].expand(BH, N, d))
    x = x + noise * torch.randn((BH, N, d), generator=g, device=device)
    return x.to(torch.bfloat16).contiguous()


def random_perm(BH: int, N: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """A seeded permutation of 0..N-1 per (b,h), int32 [BH, N]."""
    g = _gen(seed, device)
    return torch.rand((BH, N), generator=g, device=device).argsort(dim=1).to(torch.int32).contiguous()


def sample_rows(N: int, n: int, seed: int = 0) -> torch.Tensor:
    """min(n, N) distinct query rows in [0, N), n >= 4, that always include the
    first and last 128-row blocks' first and last rows; the others are drawn
    from the remaining rows.  int32, sorted."""
    g = _gen(seed, "cpu")
    fixed = torch.unique(torch.tensor([0, 127, N - 128, N - 1], dtype=torch.int64))
    free = torch.ones(N, dtype=torch.bool)
    free[fixed] = False
    others = torch.nonzero(free).flatten()
    rest = others[torch.randperm(others.numel(), generator=g)[: max(0, n - fixed.numel())]]
    return torch.sort(torch.cat([fixed, rest])).values.to(torch.int32)


def to_u16(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the oracle)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
