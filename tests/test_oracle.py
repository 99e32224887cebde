"""Pins for the fp64 oracle: each test ties it to something other than itself.

The pins are chosen so that a plausible slip anywhere in the oracle fails at
least one of them:

* wrong logit scale, transposed operand or an off-by-one causal mask — the
  lambda = 0 case must equal torch's scaled_dot_product_attention (fp64);
* a dropped or sign-flipped lambda term, lambda_init used in the subtraction,
  or a nested second softmax on the second map — the hand-worked golden
  fixtures, the two-key sigmoid closed form and the scalar brute force;
* GroupNorm over the wrong axis, unbiased variance or eps outside the root —
  torch's group_norm (fp64) on the pre-norm output;
* normalisation slips — row sums of A1 - lambda A2, constant keys, the
  identical-maps zero, affinity in lambda and the shift/permutation
  invariances.

Citations: DiffAttn formula, iloveeagents.com Q&A "Mathematical Formula";
standard attention, the same page's "Detail" and llmbytes.dev "The
Mathematical Flaw in Standard Softmax Attention"; steps 1-4 of llmbytes.dev
"How Differential Attention Cancels Common-Mode Noise".
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_inputs(rng, B, H, Nq, Nk, d, dv, dtype=np.float64, scale=1.0):
    q1 = rng.standard_normal((B, H, Nq, d)) * scale
    k1 = rng.standard_normal((B, H, Nk, d)) * scale
    q2 = rng.standard_normal((B, H, Nq, d)) * scale
    k2 = rng.standard_normal((B, H, Nk, d)) * scale
    v = rng.standard_normal((B, H, Nk, dv))
    return [np.ascontiguousarray(t, dtype=dtype) for t in (q1, k1, q2, k2, v)]


def bottom_right_mask(Nq, Nk):
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    return j <= i + (Nk - Nq)


# ---------------------------------------------------------------- library pins

@pytest.mark.parametrize("causal,Nq,Nk", [(False, 7, 13), (True, 9, 9), (True, 5, 11), (False, 1, 33)])
def test_lambda_zero_is_standard_attention(causal, Nq, Nk):
    """lambda = 0 leaves softmax(Q1 K1^T / sqrt d) V (standard attention)."""
    rng = np.random.default_rng(1)
    B, H, d, dv = 2, 3, 8, 5
    q1, k1, q2, k2, v = rand_inputs(rng, B, H, Nq, Nk, d, dv, scale=1.5)
    o_pre, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.0, 0.8, causal=causal)
    tq, tk, tv = (torch.from_numpy(x) for x in (q1, k1, v))
    mask = torch.from_numpy(bottom_right_mask(Nq, Nk)) if causal else None
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    np.testing.assert_allclose(o_pre, ref.numpy(), rtol=0, atol=1e-12)


def test_lambda_zero_second_map_irrelevant_and_first_map_sdpa_scale():
    """The scale is 1/sqrt(d) with d the Q/K width, not dv: pinned via SDPA's
    default scale at d != dv and by the second map having no effect at lambda=0."""
    rng = np.random.default_rng(2)
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 2, 6, 6, 16, 3, scale=2.0)
    a, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.0, 0.8)
    b, _ = oracle.diffattn_fwd(q1, k1, q2 * 3.0, k2[:, :, ::-1].copy(), v, 0.0, 0.8)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_groupnorm_matches_torch_group_norm(causal):
    """Step 4: GroupNorm with one group per head over the head's dv channels,
    per token, then the (1 - lambda_init) scale — torch.nn.functional.group_norm
    in fp64 on the pre-norm output is the textbook routine."""
    rng = np.random.default_rng(3)
    B, H, N, d, dv = 2, 3, 10, 4, 6
    q1, k1, q2, k2, v = rand_inputs(rng, B, H, N, N, d, dv)
    gamma = rng.uniform(0.5, 1.5, H * dv)
    lam, lam_init, eps = 0.35, 0.8, 1e-3
    o_pre, y = oracle.diffattn_fwd(q1, k1, q2, k2, v, lam, lam_init, causal=causal, gamma=gamma, eps=eps)
    # [B,H,N,dv] -> tokens x (H*dv) channels, H groups
    x = torch.from_numpy(o_pre).permute(0, 2, 1, 3).reshape(B * N, H * dv)
    ref = torch.nn.functional.group_norm(x, H, weight=torch.from_numpy(gamma), eps=eps) * (1 - lam_init)
    ref = ref.reshape(B, N, H, dv).permute(0, 2, 1, 3).numpy()
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------- golden fixtures

def _val(s):
    return float(eval(s, {"__builtins__": {}}, {"log": math.log, "sqrt": math.sqrt}))


@pytest.mark.parametrize("name", ["hand_two_keys.json", "hand_causal_three_channels.json"])
def test_hand_worked_examples(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    sh = g["shape"]
    B, H, Nq, Nk, d, dv = (sh[k] for k in ("B", "H", "Nq", "Nk", "d", "dv"))

    def arr(key, shape):
        return np.array([[_val(x) for x in row] for row in g[key]], np.float64).reshape(shape)

    q1, q2 = arr("q1", (B, H, Nq, d)), arr("q2", (B, H, Nq, d))
    k1, k2 = arr("k1", (B, H, Nk, d)), arr("k2", (B, H, Nk, d))
    v = arr("v", (B, H, Nk, dv))
    gamma = np.array([_val(x) for x in g["gamma"]])
    o_pre, y = oracle.diffattn_fwd(q1, k1, q2, k2, v, _val(g["lambda"]), _val(g["lambda_init"]),
                                   causal=g["causal"], gamma=gamma, eps=_val(g["eps"]))
    np.testing.assert_allclose(o_pre, arr("o_pre", o_pre.shape), rtol=0, atol=1e-13)
    np.testing.assert_allclose(y, arr("y", y.shape), rtol=0, atol=1e-12)


# ------------------------------------------------------------- closed forms

def test_single_key_gives_one_minus_lambda_v0():
    rng = np.random.default_rng(4)
    q1, k1, q2, k2, v = rand_inputs(rng, 2, 2, 3, 1, 8, 4)
    for lam in (0.0, 0.5, 0.9, -0.3, 1.7):
        o_pre, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, lam, 0.8)
        np.testing.assert_allclose(o_pre, np.broadcast_to((1 - lam) * v, o_pre.shape), rtol=0, atol=1e-14)


def test_two_keys_sigmoid_closed_form():
    """With two keys, each map's first weight is sigmoid(s_0 - s_1)."""
    rng = np.random.default_rng(5)
    B, H, Nq, d, dv = 1, 2, 6, 5, 3
    q1, k1, q2, k2, v = rand_inputs(rng, B, H, Nq, 2, d, dv, scale=1.3)
    lam = 0.65
    o_pre, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, lam, 0.8)
    sig = lambda x: 1.0 / (1.0 + np.exp(-x))
    s1 = np.einsum("bhid,bhjd->bhij", q1, k1) / math.sqrt(d)
    s2 = np.einsum("bhid,bhjd->bhij", q2, k2) / math.sqrt(d)
    g1 = sig(s1[..., 0] - s1[..., 1])[..., None]
    g2 = sig(s2[..., 0] - s2[..., 1])[..., None]
    v0, v1 = v[:, :, 0:1, :], v[:, :, 1:2, :]
    expect = (g1 - lam * g2) * v0 + ((1 - g1) - lam * (1 - g2)) * v1
    np.testing.assert_allclose(o_pre, expect, rtol=0, atol=1e-13)


def _scalar_brute_force(q1, k1, q2, k2, v, lam, causal):
    """Independent scalar restatement: weight_j = 1 / sum_k exp(s_k - s_j)."""
    B, H, Nq, d = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    out = np.zeros((B, H, Nq, dv))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                keys = [j for j in range(Nk) if (not causal) or j <= i + Nk - Nq]
                s1 = {j: sum(q1[b, h, i, c] * k1[b, h, j, c] for c in range(d)) / math.sqrt(d) for j in keys}
                s2 = {j: sum(q2[b, h, i, c] * k2[b, h, j, c] for c in range(d)) / math.sqrt(d) for j in keys}
                for j in keys:
                    w1 = 1.0 / sum(math.exp(s1[k] - s1[j]) for k in keys)
                    w2 = 1.0 / sum(math.exp(s2[k] - s2[j]) for k in keys)
                    for c in range(dv):
                        out[b, h, i, c] += (w1 - lam * w2) * v[b, h, j, c]
    return out


@pytest.mark.parametrize("causal,Nq,Nk", [(False, 3, 1), (False, 2, 3), (False, 4, 4), (True, 4, 4), (True, 2, 4)])
def test_brute_force_tiny(causal, Nq, Nk):
    rng = np.random.default_rng(6 + Nk)
    q1, k1, q2, k2, v = rand_inputs(rng, 2, 2, Nq, Nk, 3, 4, scale=1.2)
    for lam in (0.0, 0.8, -0.4):
        o_pre, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, lam, 0.8, causal=causal)
        ref = _scalar_brute_force(q1, k1, q2, k2, v, lam, causal)
        np.testing.assert_allclose(o_pre, ref, rtol=0, atol=1e-13)


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_maps_rows_are_distributions_and_difference_sums_to_one_minus_lambda(causal):
    rng = np.random.default_rng(7)
    q1, k1, q2, k2, _ = rand_inputs(rng, 1, 2, 12, 12, 4, 1, scale=2.0)
    a1, a2 = oracle.diffattn_maps(q1, k1, q2, k2, causal=causal)
    for a in (a1, a2):
        assert (a >= 0).all()
        np.testing.assert_allclose(a.sum(-1), 1.0, rtol=0, atol=1e-14)
    if causal:
        assert (a1[..., ~bottom_right_mask(12, 12)] == 0).all()
        assert (a2[..., ~bottom_right_mask(12, 12)] == 0).all()
    for lam in (0.2, 0.8, 1.3):
        np.testing.assert_allclose((a1 - lam * a2).sum(-1), 1 - lam, rtol=0, atol=1e-14)


def test_maps_consistent_with_rows():
    """The materialised maps times V give the row output (same definition)."""
    rng = np.random.default_rng(8)
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 2, 9, 9, 4, 3)
    a1, a2 = oracle.diffattn_maps(q1, k1, q2, k2, causal=True)
    o_pre, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.7, 0.8, causal=True)
    np.testing.assert_allclose(o_pre, np.einsum("bhij,bhjc->bhic", a1 - 0.7 * a2, v), rtol=0, atol=1e-13)


def test_identical_maps_lambda_one_cancel_exactly():
    rng = np.random.default_rng(9)
    q1, k1, _, _, v = rand_inputs(rng, 1, 2, 8, 8, 4, 6)
    for causal in (False, True):
        o_pre, y = oracle.diffattn_fwd(q1, k1, q1, k1, v, 1.0, 0.8, causal=causal)
        assert np.abs(o_pre).max() == 0.0
        assert np.abs(y).max() == 0.0


@pytest.mark.parametrize("causal", [False, True])
def test_constant_keys_give_scaled_running_mean(causal):
    rng = np.random.default_rng(10)
    B, H, N, d, dv = 1, 2, 11, 4, 5
    q1, _, q2, _, v = rand_inputs(rng, B, H, N, N, d, dv)
    k1 = np.broadcast_to(rng.standard_normal((B, H, 1, d)), (B, H, N, d)).copy()
    k2 = np.broadcast_to(rng.standard_normal((B, H, 1, d)), (B, H, N, d)).copy()
    lam = 0.3
    o_pre, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, lam, 0.8, causal=causal)
    if causal:
        expect = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    else:
        expect = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    np.testing.assert_allclose(o_pre, (1 - lam) * expect, rtol=0, atol=1e-13)


def test_affine_in_lambda():
    rng = np.random.default_rng(11)
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 2, 7, 7, 4, 3)
    o0, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.0, 0.8, causal=True)
    o1, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 1.0, 0.8, causal=True)
    for lam in (0.37, 0.9, -1.2):
        ol, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, lam, 0.8, causal=True)
        np.testing.assert_allclose(ol, o0 - lam * (o0 - o1), rtol=0, atol=1e-13)


def test_logit_shift_invariance():
    """Adding one vector u to every key shifts a query's logits by q.u, which
    each softmax removes."""
    rng = np.random.default_rng(12)
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 2, 6, 6, 4, 3)
    u1, u2 = rng.standard_normal(4), rng.standard_normal(4)
    a, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.6, 0.8, causal=True)
    b, _ = oracle.diffattn_fwd(q1, k1 + u1, q2, k2 + u2, v, 0.6, 0.8, causal=True)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_permutation_equivariance_noncausal():
    rng = np.random.default_rng(13)
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 2, 5, 9, 4, 3)
    perm = rng.permutation(9)
    a, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.6, 0.8)
    b, _ = oracle.diffattn_fwd(q1, k1[:, :, perm].copy(), q2, k2[:, :, perm].copy(), v[:, :, perm].copy(), 0.6, 0.8)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_groupnorm_invariant_to_affine_v():
    """V -> aV + b: pre-norm becomes a O + b(1 - lambda); the normalised output
    is unchanged when the variance dominates eps."""
    rng = np.random.default_rng(14)
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 2, 6, 6, 4, 8)
    lam = 0.4
    o, y = oracle.diffattn_fwd(q1, k1, q2, k2, v, lam, 0.8, causal=True, eps=0.0)
    o2, y2 = oracle.diffattn_fwd(q1, k1, q2, k2, 3.0 * v + 2.5, lam, 0.8, causal=True, eps=0.0)
    np.testing.assert_allclose(o2, 3.0 * o + 2.5 * (1 - lam), rtol=0, atol=1e-12)
    np.testing.assert_allclose(y2, y, rtol=0, atol=1e-12)


def test_causal_first_row_sees_only_first_key():
    rng = np.random.default_rng(15)
    q1, k1, q2, k2, v = rand_inputs(rng, 2, 2, 10, 10, 4, 3)
    o, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.55, 0.8, causal=True)
    np.testing.assert_allclose(o[:, :, 0], 0.45 * v[:, :, 0], rtol=0, atol=1e-15)


def test_causal_bottom_right_alignment():
    """Nq < Nk: query i sees keys j <= i + Nk - Nq; later keys have no effect."""
    rng = np.random.default_rng(16)
    Nq, Nk = 3, 8
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 1, Nq, Nk, 4, 3)
    o, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.5, 0.8, causal=True)
    for i in range(Nq):
        last = i + Nk - Nq
        v_later = v.copy()
        v_later[:, :, last + 1:] += 100.0
        ol, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v_later, 0.5, 0.8, causal=True)
        np.testing.assert_array_equal(ol[:, :, i], o[:, :, i])
        v_last = v.copy()
        v_last[:, :, last] += 100.0
        om, _ = oracle.diffattn_fwd(q1, k1, q2, k2, v_last, 0.5, 0.8, causal=True)
        assert np.abs(om[:, :, i] - o[:, :, i]).max() > 1e-6


# ------------------------------------------------------------- interface

def test_row_subset_matches_full_run():
    rng = np.random.default_rng(17)
    q1, k1, q2, k2, v = rand_inputs(rng, 2, 2, 20, 20, 4, 3)
    full = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.6, 0.8, causal=True)
    rows = [19, 0, 7, 7]
    sub = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.6, 0.8, causal=True, rows=rows)
    for f, s in zip(full, sub):
        np.testing.assert_array_equal(s, f[:, :, rows])


def test_bf16_and_f32_inputs_are_widened_exactly():
    rng = np.random.default_rng(18)
    ts = [torch.from_numpy(x).to(torch.bfloat16) for x in rand_inputs(rng, 1, 2, 9, 9, 8, 4)]
    a = oracle.diffattn_fwd(*ts, 0.6, 0.8, causal=True)
    b = oracle.diffattn_fwd(*[t.to(torch.float32) for t in ts], 0.6, 0.8, causal=True)
    c = oracle.diffattn_fwd(*[t.to(torch.float64).numpy() for t in ts], 0.6, 0.8, causal=True)
    for x, y_, z in zip(a, b, c):
        np.testing.assert_array_equal(x, y_)
        np.testing.assert_array_equal(x, z)


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(19)
    q1, k1, q2, k2, v = rand_inputs(rng, 2, 3, 17, 17, 4, 5)
    a = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.6, 0.8, causal=True, threads=1)
    b = oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.6, 0.8, causal=True, threads=8)
    for x, y_ in zip(a, b):
        np.testing.assert_array_equal(x, y_)


def test_invalid_arguments_rejected():
    rng = np.random.default_rng(20)
    q1, k1, q2, k2, v = rand_inputs(rng, 1, 1, 5, 3, 4, 2)
    with pytest.raises(ValueError):  # causal with more queries than keys
        oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.5, 0.8, causal=True)
    with pytest.raises(ValueError):
        oracle.diffattn_fwd(q1, k1, q2, k2, v, 0.5, 0.8, rows=[5])
    with pytest.raises(TypeError):
        oracle.diffattn_fwd(q1.astype(np.float32), k1, q2, k2, v, 0.5, 0.8)
