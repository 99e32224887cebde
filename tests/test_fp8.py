"""GPU parity of the fp8 (e4m3) Q/K prefill against the fp64 oracle.

Inputs are drawn in fp32, quantised per (tensor, head) with the scale
amax / 448 (448 is the largest finite e4m3 value), and the oracle receives the
dequantised values (the e4m3 value times its scale, exact in fp64).  So the
comparison measures the kernel, not the quantisation.  Tolerances are those of
the bf16 path: 1e-2 max-abs on the pre-norm output, 3e-2 on the normalised
output.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

TOL_PRE, TOL_OUT = 1e-2, 3e-2
E4M3_MAX = 448.0


def quantise(x):
    """Per-head e4m3 quantisation of [B,H,N,d]: returns (x8, scale[H], x_deq fp64 CPU)."""
    amax = x.abs().amax(dim=(0, 2, 3)).clamp_min(1e-6)
    scale = (amax / E4M3_MAX).float()
    x8 = (x / scale[None, :, None, None]).to(torch.float8_e4m3fn)
    deq = x8.cpu().double() * scale.cpu().double()[None, :, None, None]
    return x8, scale, deq


def problem(B, H, Nq, Nk, d, dv, seed, qk_std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    rn = lambda *s: torch.randn(s, generator=g, device="cuda")
    q1, k1, q2, k2 = rn(B, H, Nq, d) * qk_std, rn(B, H, Nk, d) * qk_std, rn(B, H, Nq, d) * qk_std, rn(B, H, Nk, d) * qk_std
    v = rn(B, H, Nk, dv).to(torch.bfloat16)
    gamma = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    qs = [quantise(t) for t in (q1, k1, q2, k2)]
    scale = torch.stack([s for _, s, _ in qs]).contiguous().view(-1)
    return qs, scale, v, gamma


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,causal", [
    (1, 2, 300, 333, 64, 128, True),
    (2, 2, 256, 256, 64, 128, False),
    (1, 2, 128, 128, 32, 64, False),
    (1, 3, 200, 200, 32, 64, True),
])
def test_fp8_matches_oracle(B, H, Nq, Nk, d, dv, causal):
    qs, scale, v, gamma = problem(B, H, Nq, Nk, d, dv, seed=Nq + d)
    pre = torch.empty((B, H, Nq, dv), dtype=torch.float32, device="cuda")
    out = da.fwd_fp8(qs[0][0], qs[1][0], qs[2][0], qs[3][0], v, scale, 0.6, 0.8, causal=causal, gamma=gamma,
                     o_prenorm=pre)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    o_ref, y_ref = oracle.diffattn_fwd(qs[0][2], qs[1][2], qs[2][2], qs[3][2], v.cpu().double(), 0.6, 0.8,
                                       causal=causal, gamma=gamma.double().cpu())
    assert np.abs(pre.cpu().numpy() - o_ref).max() <= TOL_PRE
    assert np.abs(out.float().cpu().numpy() - y_ref).max() <= TOL_OUT


def test_fp8_equals_bf16_path_on_representable_inputs():
    """With unit scales, e4m3 values are exactly representable in bf16: the 8-bit
    and the 16-bit tensor-core products of the same numbers agree to fp32
    accumulation order."""
    B, H, N, d, dv = 1, 2, 384, 64, 128
    g = torch.Generator(device="cuda").manual_seed(5)
    mk8 = lambda n: (torch.randn((B, H, n, d), generator=g, device="cuda") * 0.5).to(torch.float8_e4m3fn)
    q1, k1, q2, k2 = mk8(N), mk8(N), mk8(N), mk8(N)
    v = torch.randn((B, H, N, dv), generator=g, device="cuda").to(torch.bfloat16)
    ones = torch.ones(4 * H, device="cuda")
    p8 = torch.empty((B, H, N, dv), device="cuda")
    p16 = torch.empty_like(p8)
    da.fwd_fp8(q1, k1, q2, k2, v, ones, 0.5, 0.8, causal=True, o_prenorm=p8)
    b = lambda t: t.to(torch.bfloat16)
    da.fwd(b(q1), b(k1), b(q2), b(k2), v, 0.5, 0.8, causal=True, o_prenorm=p16)
    torch.cuda.synchronize()
    assert (p8 - p16).abs().max().item() <= 1e-3


def test_fp8_long_sampled_rows():
    """B1 H4 N8192 causal with Q/K ~ N(0, 1/2): sampled rows against the oracle."""
    B, H, N, d, dv = 1, 4, 8192, 64, 128
    qs, scale, v, gamma = problem(B, H, N, N, d, dv, seed=81, qk_std=2 ** -0.5)
    pre = torch.empty((B, H, N, dv), dtype=torch.float32, device="cuda")
    out = da.fwd_fp8(qs[0][0], qs[1][0], qs[2][0], qs[3][0], v, scale, 0.7, 0.8, causal=True, o_prenorm=pre)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(32), np.random.default_rng(1).choice(N, 64, replace=False), np.arange(N - 32, N)])
    o_ref, y_ref = oracle.diffattn_fwd(qs[0][2], qs[1][2], qs[2][2], qs[3][2], v.cpu().double(), 0.7, 0.8,
                                       causal=True, rows=rows)
    assert np.abs(pre[:, :, rows].cpu().numpy() - o_ref).max() <= TOL_PRE
    assert np.abs(out[:, :, rows].float().cpu().numpy() - y_ref).max() <= TOL_OUT


def test_fp8_benchmarked_configuration_sampled_rows():
    """The configuration bench.py times for the fp8 row: the long_64k workload
    (causal, B1 H16 N65536) quantised exactly as the bench does (per-head
    amax / 448), sampled rows against the oracle on the dequantised values."""
    from transformer_attention_07_b300.workloads import WORKLOADS, make_inputs, sample_rows
    w = WORKLOADS["long_64k"]
    inp = make_inputs(w, device="cuda")
    qs = [quantise(inp[n].float()) for n in ("q1", "k1", "q2", "k2")]
    scale = torch.stack([s for _, s, _ in qs]).contiguous().view(-1)
    pre = torch.empty((w.B, w.H, w.Nq, w.dv), dtype=torch.float32, device="cuda")
    out = da.fwd_fp8(qs[0][0], qs[1][0], qs[2][0], qs[3][0], inp["v"], scale, w.lam, w.lam_init, causal=w.causal,
                     gamma=inp["gamma"], eps=w.eps, o_prenorm=pre)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    rows = np.asarray(sample_rows(w.Nq, w.seed, n_random=32, edge=16))
    g = inp["gamma"]
    o_ref, y_ref = oracle.diffattn_fwd(qs[0][2], qs[1][2], qs[2][2], qs[3][2], inp["v"].cpu().double(), w.lam,
                                       w.lam_init, causal=w.causal, eps=w.eps,
                                       gamma=None if g is None else g.double().cpu(), rows=rows)
    assert np.abs(pre[:, :, rows].cpu().numpy() - o_ref).max() <= TOL_PRE
    assert np.abs(out[:, :, rows].float().cpu().numpy() - y_ref).max() <= TOL_OUT
