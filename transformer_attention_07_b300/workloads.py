"""Seeded synthetic inputs for the differential-attention forward and backward.

This module only draws numbers: it holds none of the method's arithmetic, so
the tests, the benchmark and the oracle-side checks can all take their inputs
from it.  Shapes and value distributions follow the long-context language-
model workloads the Differential Transformer pages discuss (4K-128K tokens,
llmbytes.dev "The Mathematical Flaw in Standard Softmax Attention" and
"Multi-Needle Retrieval at 64K Context"); no dataset is involved.

Draw order is Q1, K1, Q2, K2, V, gamma, from one ``torch.Generator`` seeded
per workload, in fp32, then rounded to bf16 (nearest even).  The upstream
gradient of the backward pass (``make_dy``) is N(0, 1) from its own seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill" or "decode"
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dv: int
    causal: bool
    lam: float
    lam_init: float
    eps: float
    gamma: str           # "ones" or "uniform" (U(0.5, 1.5) per channel)
    qk_std: float        # standard deviation of the Q/K draws
    structure: str       # "plain" or "cancellation"
    seed: int

    @property
    def pairs(self) -> int:
        """Unmasked (query, key) pairs."""
        per = self.Nq * self.Nk
        if self.causal:  # query i sees i + (Nk - Nq) + 1 keys (Nq <= Nk)
            per = self.Nq * (self.Nq + 1) // 2 + self.Nq * (self.Nk - self.Nq)
        return self.B * self.H * per

    @property
    def flops(self) -> int:
        """Algorithmic flops: 2 QK^T (2d each) + 2 PV (2dv each) per pair."""
        return 4 * (self.d + self.dv) * self.pairs

    @property
    def bwd_flops(self) -> int:
        """Algorithmic flops of the backward pass per pair: S1, S2 recomputed
        (2d each), dP = do V^T (2dv), dV (2dv), dK1, dK2 (2d each), dQ1, dQ2
        (2d each)."""
        return (12 * self.d + 4 * self.dv) * self.pairs

    @property
    def kv_bytes(self) -> int:
        """Algorithmic bytes of a decode step: K1, K2, V read once, q in, out."""
        return self.B * self.H * (self.Nk * (2 * self.d + self.dv) + 2 * self.d + self.dv) * 2


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_noncausal", "prefill", 1, 2, 128, 128, 32, 64, False, 0.8, 0.8, 1e-5, "ones", 1.0,
                 "plain", 1000),
        Workload("causal_2k", "prefill", 4, 8, 2048, 2048, 64, 128, True, 0.5, 0.8, 1e-5, "uniform", 1.0,
                 "plain", 1001),
        Workload("cancel_8k", "prefill", 2, 16, 8192, 8192, 64, 128, True, 0.9, 0.8, 1e-5, "ones", 1.0,
                 "cancellation", 1002),
        Workload("long_64k", "prefill", 1, 16, 65536, 65536, 64, 128, True, 0.7, 0.8, 1e-5, "ones",
                 1.0 / math.sqrt(2.0), "plain", 1003),
        Workload("long_128k", "prefill", 1, 8, 131072, 131072, 64, 128, True, 0.7, 0.8, 1e-5, "ones",
                 1.0 / math.sqrt(2.0), "plain", 1005),
        Workload("decode_32k", "decode", 32, 32, 1, 32768, 64, 128, False, 0.6, 0.8, 1e-5, "ones", 1.0,
                 "plain", 1004),
        # Smaller cases of the same distributions, for multi-pass profiler
        # captures: inputs still larger than L2, a few GB on the device at most.
        Workload("long_16k", "prefill", 1, 16, 16384, 16384, 64, 128, True, 0.7, 0.8, 1e-5, "ones",
                 1.0 / math.sqrt(2.0), "plain", 1006),
        Workload("decode_32k_b4", "decode", 4, 32, 1, 32768, 64, 128, False, 0.6, 0.8, 1e-5, "ones", 1.0,
                 "plain", 1007),
    ]
}

NEEDLE_BLOCK = 256


def _randn(shape, gen, device, std=1.0):
    """fp32 N(0, std^2) draws, produced one leading slice at a time so that very
    large tensors never exist in fp32 all at once; returns bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for b in range(shape[0]):
        x = torch.randn(shape[1:], generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[b].copy_(x)
    return out


def make_inputs(w: Workload, device="cuda", seed: int | None = None, Nq: int | None = None,
                Nk: int | None = None, B: int | None = None, H: int | None = None):
    """Inputs of workload ``w`` (optionally with other sizes), as a dict of
    bf16 tensors q1, k1, q2, k2, v and fp32 ``gamma`` (None for all ones)."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    Nq = w.Nq if Nq is None else Nq
    Nk = w.Nk if Nk is None else Nk
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    if w.structure == "cancellation":
        q1 = torch.randn((B, H, Nq, w.d), generator=gen, device=device) * w.qk_std
        k1 = torch.randn((B, H, Nk, w.d), generator=gen, device=device) * w.qk_std
        q2 = q1 + 0.1 * torch.randn((B, H, Nq, w.d), generator=gen, device=device)
        k2 = k1 + 0.1 * torch.randn((B, H, Nk, w.d), generator=gen, device=device)
        plant_needles(q1, k1, w.d)
        q1, k1, q2, k2 = (t.to(torch.bfloat16) for t in (q1, k1, q2, k2))
    else:
        q1 = _randn((B, H, Nq, w.d), gen, device, w.qk_std)
        k1 = _randn((B, H, Nk, w.d), gen, device, w.qk_std)
        q2 = _randn((B, H, Nq, w.d), gen, device, w.qk_std)
        k2 = _randn((B, H, Nk, w.d), gen, device, w.qk_std)
    v = _randn((B, H, Nk, w.dv), gen, device)
    gamma = None
    if w.gamma == "uniform":
        gamma = torch.rand((H * w.dv,), generator=gen, device=device, dtype=torch.float32) + 0.5
    return {"q1": q1, "k1": k1, "q2": q2, "k2": k2, "v": v, "gamma": gamma}


def standard_inputs(B: int, H: int, N: int, d: int = 128, dv: int = 128, seed: int = 2000, device="cuda"):
    """q, k, v (bf16, N(0,1)) for the single-map baseline of width d = dv =
    128: one differential head's [q1; q2] and v at equal parameters."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return {"q": _randn((B, H, N, d), gen, device), "k": _randn((B, H, N, d), gen, device),
            "v": _randn((B, H, N, dv), gen, device)}


# DiffAttn against the single-map baseline at the sequence lengths the pages
# quote a throughput overhead for (2K and 4K), with the same token count.
COMPARE_SHAPES = ((8, 16, 2048), (4, 16, 4096))


def plant_needles(q1: torch.Tensor, k1: torch.Tensor, d: int) -> None:
    """In place: the first key of every 256-token block of K1 becomes
    4*sqrt(d) times the unit direction of that block's mean Q1 row, a key
    every query of the block scores about 4x a typical logit on (K2 is drawn
    from K1 before this, so it keeps the original key: a needle in map 1
    only)."""
    B, H, N, _ = q1.shape
    nb = N // NEEDLE_BLOCK
    if nb == 0:
        return
    blocks = q1[:, :, : nb * NEEDLE_BLOCK].reshape(B, H, nb, NEEDLE_BLOCK, d).mean(dim=3)
    u = blocks / blocks.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    k1[:, :, 0: nb * NEEDLE_BLOCK: NEEDLE_BLOCK] = 4.0 * math.sqrt(d) * u


def needle_rows(N: int) -> list[int]:
    return list(range(0, N - N % NEEDLE_BLOCK, NEEDLE_BLOCK))


def sample_rows(N: int, seed: int, n_random: int = 384, edge: int = 64) -> list[int]:
    """Query rows checked against the oracle on large problems: the first and
    last ``edge`` rows plus ``n_random`` seeded random rows (sorted, unique)."""
    rows = set(range(min(edge, N))) | set(range(max(0, N - edge), N))
    g = torch.Generator().manual_seed(seed)
    if N > 2 * edge:
        rows |= set(torch.randint(edge, N - edge, (n_random,), generator=g).tolist())
    return sorted(rows)


def make_dy(w: Workload, device="cuda", seed=None):
    """Upstream gradient dL/dy for the backward pass: N(0, 1), bf16, [B,H,Nq,dv]."""
    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 500)
    dy = torch.empty((w.B, w.H, w.Nq, w.dv), dtype=torch.bfloat16, device=device)
    for b in range(w.B):
        for h in range(w.H):
            dy[b, h].copy_(torch.randn((w.Nq, w.dv), generator=g, device=device))
    return dy
