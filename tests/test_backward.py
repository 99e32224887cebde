"""GPU parity of the training forward outputs and the backward pass against
the fp64 oracle (whose gradients are pinned by finite differences and torch
autograd in test_oracle_bwd.py).

Tolerances.  Every gradient is stored in bf16 (relative rounding 2^-9), and
the tile kernels multiply bf16 operands: the rounded do, the probabilities
and dS rounded to bf16 before each tensor-core product, with fp32
accumulation.  Each such rounding is a relative error of at most 2^-9 per
term; over sums of many terms they partly cancel.  The checks are therefore
relative to the size of each gradient tensor: the Frobenius-norm relative
error must stay below 1e-2 and the largest element error below 3e-2 of the
tensor's largest magnitude (plus an absolute 1e-5 per element, for
gradients that vanish exactly).  dlambda is a sum of one term per row that
can cancel to far below its terms (with one key per row the normalisation
makes y independent of lambda and dlambda is 0); its bound, derived from the
forward's rounding, and the check that the bound still rejects a flipped,
dropped or misweighted term are in dlambda_bound.py.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da
from dlambda_bound import assert_dlambda

pytestmark = pytest.mark.gpu

FRO_TOL, MAX_TOL = 1e-2, 3e-2


def inputs(B, H, Nq, Nk, seed, d=64, dv=128, qk_scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s, sc=1.0: (torch.randn(s, generator=g, device="cuda") * sc).to(torch.bfloat16)
    q1, k1 = mk(B, H, Nq, d, sc=qk_scale), mk(B, H, Nk, d, sc=qk_scale)
    q2, k2 = mk(B, H, Nq, d, sc=qk_scale), mk(B, H, Nk, d, sc=qk_scale)
    v = mk(B, H, Nk, dv)
    dy = mk(B, H, Nq, dv)
    gamma = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    return q1, k1, q2, k2, v, dy, gamma


def rel_check(name, got, ref, floor=1e-5):
    """Errors relative to the gradient's own size; `floor` is an absolute
    allowance per element for gradients that vanish exactly (a row whose
    only visible key is itself has dq = 0; the kernels return rounding noise
    around 1e-8 there)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = got - ref
    fro_ok = np.linalg.norm(err) <= FRO_TOL * np.linalg.norm(ref) + floor * np.sqrt(err.size)
    mx_ok = np.abs(err).max() <= MAX_TOL * np.abs(ref).max() + floor
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(err).max() / max(np.abs(ref).max(), 1e-30)
    assert fro_ok and mx_ok, f"{name}: frobenius rel {fro:.3e}, max rel {mx:.3e}"


def run(q1, k1, q2, k2, v, dy, gamma, lam, lam_init, causal):
    out, saved = da.fwd_train(q1, k1, q2, k2, v, lam, lam_init, causal=causal, gamma=gamma)
    grads = da.bwd(q1, k1, q2, k2, v, dy, saved, lam, lam_init, causal=causal, gamma=gamma)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    return out, saved, grads


def cpu(*ts):
    return [t.cpu() for t in ts]


@pytest.mark.parametrize("B,H,Nq,Nk,causal,lam,d,dv", [
    (2, 2, 256, 256, True, 0.5, 64, 128),
    (1, 2, 200, 333, True, 0.8, 64, 128),
    (1, 2, 200, 333, False, -0.3, 64, 128),
    (2, 1, 130, 70, False, 0.0, 64, 128),
    (1, 1, 1, 1, True, 0.6, 64, 128),
    (2, 2, 256, 256, True, 0.5, 32, 64),
    (1, 2, 200, 333, True, 0.8, 32, 64),
    (2, 1, 130, 70, False, -0.3, 32, 64),
])
def test_backward_matches_oracle(B, H, Nq, Nk, causal, lam, d, dv):
    q1, k1, q2, k2, v, dy, gamma = inputs(B, H, Nq, Nk, seed=Nq + Nk + int(causal) + d, d=d, dv=dv)
    _, _, g = run(q1, k1, q2, k2, v, dy, gamma, lam, 0.8, causal)
    ref = oracle.diffattn_bwd(*cpu(q1, k1, q2, k2, v, dy), lam, 0.8, causal=causal, gamma=gamma.double().cpu())
    for n in ("dq1", "dk1", "dq2", "dk2", "dv"):
        rel_check(n, g[n].float().cpu().numpy(), ref[n])
    assert_dlambda(g["dlambda"].item(), ref["dlambda"], ref["dlambda_rss"])
    rel_check("dgamma", g["dgamma"].cpu().numpy(), ref["dgamma"])


def test_training_outputs_match_the_definition():
    """o2 = A2 V = o_pre(lambda=0) - o_pre(lambda=1) from the oracle; lse_r,i
    recovered from the oracle's probabilities: a_r,ij = exp(s_r,ij - lse_r,i)."""
    B, H, N = 1, 2, 150
    q1, k1, q2, k2, v, dy, gamma = inputs(B, H, N, N, seed=4)
    out, saved = da.fwd_train(q1, k1, q2, k2, v, 0.5, 0.8, causal=True, gamma=gamma)
    torch.cuda.synchronize()
    c = cpu(q1, k1, q2, k2, v)
    o0, _ = oracle.diffattn_fwd(*c, 0.0, 0.8, causal=True)
    o1, _ = oracle.diffattn_fwd(*c, 1.0, 0.8, causal=True)
    assert np.abs(saved["o2"].cpu().numpy() - (o0 - o1)).max() <= 1e-2
    o_ref, y_ref = oracle.diffattn_fwd(*c, 0.5, 0.8, causal=True, gamma=gamma.double().cpu())
    assert np.abs(saved["o_prenorm"].cpu().numpy() - o_ref).max() <= 1e-2
    assert np.abs(out.float().cpu().numpy() - y_ref).max() <= 3e-2
    a1, a2 = oracle.diffattn_maps(*c[:4], causal=True)
    lse = saved["lse"].double().cpu().numpy()
    for r, (q, k, a) in enumerate(((c[0], c[1], a1), (c[2], c[3], a2))):
        s = q.double().numpy() @ k.double().numpy().transpose(0, 1, 3, 2) / np.sqrt(64.0)
        # the largest probability of each row gives the best-conditioned estimate
        j = a.argmax(-1)
        s_j = np.take_along_axis(s, j[..., None], -1)[..., 0]
        a_j = np.take_along_axis(a, j[..., None], -1)[..., 0]
        # The forward's normaliser sums the bf16-rounded probabilities (the
        # values the P V product uses), each within a relative 2^-9 of the
        # exact one, so log l is within log(1 + 2^-9) < 2e-3 of the exact
        # log-sum-exp.
        assert np.abs(lse[r] - (s_j - np.log(a_j))).max() <= 2e-3


def test_backward_is_deterministic():
    q1, k1, q2, k2, v, dy, gamma = inputs(1, 4, 512, 512, seed=9)
    _, saved, g1 = run(q1, k1, q2, k2, v, dy, gamma, 0.7, 0.8, True)
    g1 = {k: t.clone() for k, t in g1.items()}
    g2 = da.bwd(q1, k1, q2, k2, v, dy, saved, 0.7, 0.8, causal=True, gamma=gamma)
    torch.cuda.synchronize()
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_backward_cancelling_maps():
    """Q2 = Q1, K2 = K1, lambda = 1: the pre-norm output is 0 for every input,
    so y does not depend on V, Q or K except through eps-regularised zeros:
    the oracle and the kernels must agree on dV = (A1 - A2)^T do = 0."""
    q1, k1, _, _, v, dy, gamma = inputs(1, 2, 192, 192, seed=12)
    _, _, g = run(q1, k1, q1, k1, v, dy, gamma, 1.0, 0.8, True)
    assert g["dv"].abs().max().item() == 0.0


def test_backward_2k_sampled():
    """B4 H8 N2048 causal (the 2K prefill shape): sampled query rows for dq and
    the last keys (seen only by the last queries) for dk, dv."""
    B, H, N = 4, 8, 2048
    q1, k1, q2, k2, v, dy, gamma = inputs(B, H, N, N, seed=2048)
    _, _, g = run(q1, k1, q2, k2, v, dy, gamma, 0.5, 0.8, True)
    rng = np.random.default_rng(0)
    rows = np.concatenate([np.arange(64), rng.choice(np.arange(64, N - 64), 64, replace=False), np.arange(N - 64, N)])
    keys = np.arange(N - 96, N)
    ref = oracle.diffattn_bwd(*cpu(q1, k1, q2, k2, v, dy), 0.5, 0.8, causal=True, gamma=gamma.double().cpu(),
                              rows=rows, keys=keys)
    for n in ("dq1", "dq2"):
        rel_check(n, g[n][:, :, rows].float().cpu().numpy(), ref[n])
    for n in ("dk1", "dk2", "dv"):
        rel_check(n, g[n][:, :, keys].float().cpu().numpy(), ref[n])


def test_backward_empty_queries_write_zero_key_gradients():
    q1, k1, q2, k2, v, dy, gamma = inputs(1, 2, 0, 64, seed=1)
    saved = {"o_prenorm": torch.empty((1, 2, 0, 128), device="cuda"), "o2": torch.empty((1, 2, 0, 128), device="cuda"),
             "lse": torch.empty((2, 1, 2, 0), device="cuda")}
    grads = {n: torch.full_like(t, 7.0) for n, t in (("dq1", q1), ("dk1", k1), ("dq2", q2), ("dk2", k2), ("dv", v))}
    grads["dlambda"] = torch.full((1,), 7.0, device="cuda")
    grads["dgamma"] = torch.full((256,), 7.0, device="cuda")
    da.bwd(q1, k1, q2, k2, v, dy, saved, 0.5, 0.8, causal=False, gamma=gamma, grads=grads)
    torch.cuda.synchronize()
    for n in ("dk1", "dk2", "dv", "dlambda", "dgamma"):
        assert grads[n].abs().max().item() == 0.0, n


def test_backward_64k_sampled():
    """The backward configuration bench.py times (causal 64K, B1 H16, the
    workload's own inputs and dy): dq on sampled rows (the first and last 16
    and 16 seeded rows), dk and dv on the last 64 keys, which only the last
    queries see (the oracle visits just those rows)."""
    from transformer_attention_07_b300.workloads import WORKLOADS, make_dy, make_inputs, sample_rows
    w = WORKLOADS["long_64k"]
    inp = make_inputs(w, device="cuda")
    dy = make_dy(w, device="cuda")
    q1, k1, q2, k2, v = (inp[n] for n in ("q1", "k1", "q2", "k2", "v"))
    gamma = inp["gamma"]
    out, saved = da.fwd_train(q1, k1, q2, k2, v, w.lam, w.lam_init, causal=w.causal, gamma=gamma, eps=w.eps)
    g = da.bwd(q1, k1, q2, k2, v, dy, saved, w.lam, w.lam_init, causal=w.causal, gamma=gamma, eps=w.eps)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    rows = np.asarray(sample_rows(w.Nq, w.seed, n_random=16, edge=16))
    keys = np.arange(w.Nk - 64, w.Nk)
    ref = oracle.diffattn_bwd(*cpu(q1, k1, q2, k2, v, dy), w.lam, w.lam_init, causal=w.causal,
                              gamma=None if gamma is None else gamma.double().cpu(), eps=w.eps, rows=rows, keys=keys)
    for n in ("dq1", "dq2"):
        rel_check(n, g[n][:, :, rows].float().cpu().numpy(), ref[n])
    for n in ("dk1", "dk2", "dv"):
        rel_check(n, g[n][:, :, keys].float().cpu().numpy(), ref[n])
