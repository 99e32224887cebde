"""Pins for the oracle's backward pass (CPU only).

The oracle's gradients are checked against two things outside it:

* central finite differences of the oracle's own forward pass (a check of
  the derivative, not of a retyped formula: a dropped term, a wrong sign, a
  swapped operand or a wrong index in the chain rule changes the result), for
  every element of every input, and for lambda and the GroupNorm gain;
* torch autograd through library routines (``scaled_dot_product_attention``
  for each map and ``group_norm``), in float64.

Plus the row/key subsetting of the oracle against its own full result.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def problem(B, H, Nq, Nk, d, dv, seed):
    rng = np.random.default_rng(seed)
    q1, q2 = rng.standard_normal((B, H, Nq, d)), rng.standard_normal((B, H, Nq, d))
    k1, k2 = rng.standard_normal((B, H, Nk, d)), rng.standard_normal((B, H, Nk, d))
    v = rng.standard_normal((B, H, Nk, dv))
    dy = rng.standard_normal((B, H, Nq, dv))
    gamma = rng.random(H * dv) + 0.5
    return {"q1": q1, "k1": k1, "q2": q2, "k2": k2, "v": v}, dy, gamma


def loss(t, dy, lam, lam_init, causal, gamma):
    _, y = oracle.diffattn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], lam, lam_init, causal=causal,
                               gamma=gamma, threads=1)
    return float((y * dy).sum())


@pytest.mark.parametrize("causal,Nq,Nk", [(False, 5, 6), (True, 6, 6), (True, 4, 7)])
def test_gradients_match_finite_differences(causal, Nq, Nk):
    B, H, d, dv = 1, 2, 4, 6
    t, dy, gamma = problem(B, H, Nq, Nk, d, dv, seed=Nq * 10 + Nk + causal)
    lam, lam_init, h = 0.6, 0.8, 1e-5
    g = oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, lam, lam_init, causal=causal,
                            gamma=gamma, threads=1)
    for name in ("q1", "k1", "q2", "k2", "v"):
        num = np.zeros_like(t[name])
        for idx in np.ndindex(t[name].shape):
            orig = t[name][idx]
            t[name][idx] = orig + h
            lp = loss(t, dy, lam, lam_init, causal, gamma)
            t[name][idx] = orig - h
            lm = loss(t, dy, lam, lam_init, causal, gamma)
            t[name][idx] = orig
            num[idx] = (lp - lm) / (2 * h)
        assert np.abs(g["d" + name] - num).max() < 1e-7 * max(1.0, np.abs(num).max()), name
    num_lam = (loss(t, dy, lam + h, lam_init, causal, gamma) - loss(t, dy, lam - h, lam_init, causal, gamma)) / (2 * h)
    assert abs(g["dlambda"] - num_lam) < 1e-7 * max(1.0, abs(num_lam))
    num_g = np.zeros_like(gamma)
    for c in range(gamma.size):
        gp, gm = gamma.copy(), gamma.copy()
        gp[c] += h
        gm[c] -= h
        num_g[c] = (loss(t, dy, lam, lam_init, causal, gp) - loss(t, dy, lam, lam_init, causal, gm)) / (2 * h)
    assert np.abs(g["dgamma"] - num_g).max() < 1e-7 * max(1.0, np.abs(num_g).max())


def torch_forward(q1, k1, q2, k2, v, lam, lam_init, causal, gamma, eps):
    """The forward pass assembled from library routines (float64)."""
    B, H, Nq, _ = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    mask = None
    if causal:   # key j visible to query i iff j <= i + Nk - Nq
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        mask = j <= i + (Nk - Nq)
    a1v = F.scaled_dot_product_attention(q1, k1, v, attn_mask=mask)
    a2v = F.scaled_dot_product_attention(q2, k2, v, attn_mask=mask)
    o = a1v - lam * a2v
    x = o.permute(0, 2, 1, 3).reshape(B * Nq, H * dv)
    y = F.group_norm(x, H, weight=gamma, bias=None, eps=eps) * (1 - lam_init)
    return y.reshape(B, Nq, H, dv).permute(0, 2, 1, 3)


@pytest.mark.parametrize("causal,Nq,Nk", [(False, 37, 41), (True, 37, 41), (True, 33, 33)])
def test_gradients_match_torch_autograd(causal, Nq, Nk):
    B, H, d, dv = 2, 3, 8, 16
    t, dy, gamma = problem(B, H, Nq, Nk, d, dv, seed=7 + Nq + causal)
    lam, lam_init, eps = -0.3 if causal else 0.9, 0.7, 1e-5
    tt = {k: torch.tensor(x, requires_grad=True) for k, x in t.items()}
    tlam = torch.tensor(lam, dtype=torch.float64, requires_grad=True)
    tg = torch.tensor(gamma, requires_grad=True)
    y = torch_forward(tt["q1"], tt["k1"], tt["q2"], tt["k2"], tt["v"], tlam, lam_init, causal, tg, eps)
    (y * torch.tensor(dy)).sum().backward()
    g = oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, lam, lam_init, causal=causal,
                            gamma=gamma, eps=eps)
    for name in ("q1", "k1", "q2", "k2", "v"):
        ref = tt[name].grad.numpy()
        assert np.abs(g["d" + name] - ref).max() < 1e-10 * max(1.0, np.abs(ref).max()), name
    assert abs(g["dlambda"] - tlam.grad.item()) < 1e-10 * max(1.0, abs(tlam.grad.item()))
    assert np.abs(g["dgamma"] - tg.grad.numpy()).max() < 1e-10 * max(1.0, np.abs(tg.grad.numpy()).max())


def test_row_and_key_subsets_equal_the_full_result():
    B, H, Nq, Nk, d, dv = 2, 2, 29, 35, 8, 16
    t, dy, gamma = problem(B, H, Nq, Nk, d, dv, seed=3)
    args = (t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, 0.5, 0.8)
    full = oracle.diffattn_bwd(*args, causal=True, gamma=gamma)
    rows, keys = [0, 7, 28], [1, 30, 34]
    sub = oracle.diffattn_bwd(*args, causal=True, gamma=gamma, rows=rows, keys=keys)
    for n in ("dq1", "dq2"):
        np.testing.assert_allclose(sub[n], full[n][:, :, rows], rtol=0, atol=1e-13)
    for n in ("dk1", "dk2", "dv"):
        np.testing.assert_allclose(sub[n], full[n][:, :, keys], rtol=0, atol=1e-13)
    assert "dlambda" not in sub and "dgamma" not in sub


def test_dlambda_rss_is_the_root_sum_square_of_row_terms():
    """dlambda sums one term per row; computing each row alone (a one-row
    problem per query, through the full oracle) gives the terms."""
    t, dy, gamma = problem(1, 1, 6, 6, 4, 8, seed=11)
    full = oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, 0.7, 0.8, gamma=gamma)
    terms = []
    for i in range(6):
        dyi = np.zeros_like(dy)
        dyi[:, :, i] = dy[:, :, i]
        terms.append(oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dyi, 0.7, 0.8,
                                         gamma=gamma)["dlambda"])
    assert abs(sum(terms) - full["dlambda"]) < 1e-12
    assert abs(np.sqrt(np.sum(np.square(terms))) - full["dlambda_rss"]) < 1e-12


def test_gradients_vanish_when_lambda_init_is_one():
    """With lambda_init = 1 the output scale (1 - lambda_init) is 0, so y = 0 for
    every input and every gradient is exactly 0."""
    t, dy, gamma = problem(1, 2, 9, 9, 4, 8, seed=5)
    g = oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, 0.4, 1.0, causal=True, gamma=gamma)
    for n in ("dq1", "dq2", "dk1", "dk2", "dv", "dgamma"):
        assert np.abs(g[n]).max() == 0.0, n
    assert g["dlambda"] == 0.0


def test_single_key_closed_form():
    """With one key every softmax row is exactly 1, so o = (1 - lambda) v0 for
    every query: the scores get no gradient (dq = dk = 0 exactly) and
    dv0 = (1 - lambda) sum_i do_i, where do is the gradient of the GroupNorm
    output alone (torch autograd through group_norm, a library routine)."""
    B, H, Nq, d, dv = 1, 2, 5, 4, 8
    t, dy, gamma = problem(B, H, Nq, 1, d, dv, seed=13)
    lam, lam_init, eps = 0.35, 0.8, 1e-5
    g = oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, lam, lam_init, gamma=gamma, eps=eps)
    for n in ("dq1", "dq2", "dk1", "dk2"):
        assert np.abs(g[n]).max() == 0.0, n
    o = torch.tensor(np.broadcast_to((1 - lam) * t["v"], (B, H, Nq, dv)).copy(), requires_grad=True)
    x = o.permute(0, 2, 1, 3).reshape(B * Nq, H * dv)
    y = F.group_norm(x, H, weight=torch.tensor(gamma), bias=None, eps=eps) * (1 - lam_init)
    (y.reshape(B, Nq, H, dv).permute(0, 2, 1, 3) * torch.tensor(dy)).sum().backward()
    dv_ref = (1 - lam) * o.grad.numpy().sum(axis=2, keepdims=True)
    assert np.abs(g["dv"] - dv_ref).max() < 1e-12 * max(1.0, np.abs(dv_ref).max())


def test_bwd_rejects_bad_arguments():
    t, dy, _ = problem(1, 1, 4, 4, 4, 8, seed=1)
    with pytest.raises(ValueError):
        oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy[:, :, :3], 0.5, 0.8)
    with pytest.raises(ValueError):
        oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, 0.5, 0.8, rows=[4])


@pytest.mark.parametrize("B,H,Nq,Nk,causal,lam", [
    (2, 2, 64, 64, True, 0.5), (1, 2, 40, 70, False, -0.3), (2, 1, 30, 20, False, 0.0), (1, 3, 50, 90, True, 0.8)])
def test_dlambda_bound_rejects_plausible_kernel_mistakes(B, H, Nq, Nk, causal, lam):
    """The GPU tests accept dlambda within 1e-2 |dlambda| + 3.2e-3 rss (rss =
    root-sum-square of the per-row terms; tests/dlambda_bound.py derives it
    from the forward's bf16 rounding).  On oracle gradients of problems like
    the GPU tests' (no GPU needed), that bound must reject what a kernel
    mistake would produce: the lambda term's sign flipped (-dlambda), the
    term dropped (0), or the terms of half the rows left out."""
    from dlambda_bound import assert_rejects_plausible_bugs, bound
    t, dy, gamma = problem(B, H, Nq, Nk, 64, 128, seed=B * 1000 + Nq + Nk)
    g = oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy, lam, 0.8, causal=causal, gamma=gamma)
    ref, rss = g["dlambda"], g["dlambda_rss"]
    assert_rejects_plausible_bugs(ref, rss)
    b = bound(ref, rss)
    for wrong in (-ref, 0.0):
        assert abs(wrong - ref) > b
    # Every second row's term dropped (a kernel summing only part of the
    # rows): the oracle's dlambda of the loss restricted to the other rows.
    dy_half = dy.copy()
    dy_half[:, :, 1::2] = 0.0
    part = oracle.diffattn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], dy_half, lam, 0.8, causal=causal,
                               gamma=gamma)["dlambda"]
    assert abs(part - ref) > b
