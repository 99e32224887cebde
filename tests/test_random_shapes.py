"""Seeded random shapes for every path against the fp64 oracle: ragged
lengths (not multiples of any tile), both head widths, causal and not,
several lambdas.  Tolerances as in the dedicated tests (1e-2 pre-norm,
3e-2 normalised; gradients relative to their own size)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da
from dlambda_bound import assert_dlambda

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(20261203)
CASES = []
for _ in range(12):
    d, dv = [(64, 128), (32, 64)][RNG.integers(2)]
    causal = bool(RNG.integers(2))
    Nk = int(RNG.integers(1, 700))
    Nq = int(RNG.integers(1, Nk + 1)) if causal else int(RNG.integers(1, 700))
    CASES.append((int(RNG.integers(1, 3)), int(RNG.integers(1, 4)), Nq, Nk, d, dv, causal,
                  float(np.round(RNG.uniform(-0.5, 1.2), 3))))


def draw(B, H, Nq, Nk, d, dv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    return mk(B, H, Nq, d), mk(B, H, Nk, d), mk(B, H, Nq, d), mk(B, H, Nk, d), mk(B, H, Nk, dv), mk(B, H, Nq, dv)


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,causal,lam", CASES)
def test_prefill_and_backward_random(B, H, Nq, Nk, d, dv, causal, lam):
    q1, k1, q2, k2, v, dy = draw(B, H, Nq, Nk, d, dv, seed=Nq * 1000 + Nk)
    out, saved = da.fwd_train(q1, k1, q2, k2, v, lam, 0.8, causal=causal)
    grads = da.bwd(q1, k1, q2, k2, v, dy, saved, lam, 0.8, causal=causal)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    cpu = [t.cpu() for t in (q1, k1, q2, k2, v)]
    o_ref, y_ref = oracle.diffattn_fwd(*cpu, lam, 0.8, causal=causal)
    assert np.abs(saved["o_prenorm"].cpu().numpy() - o_ref).max() <= 1e-2
    assert np.abs(out.float().cpu().numpy() - y_ref).max() <= 3e-2
    ref = oracle.diffattn_bwd(*cpu, dy.cpu(), lam, 0.8, causal=causal)
    for n in ("dq1", "dk1", "dq2", "dk2", "dv"):
        got, want = grads[n].float().cpu().numpy().astype(np.float64), ref[n]
        err = got - want
        assert np.linalg.norm(err) <= 1e-2 * np.linalg.norm(want) + 1e-5 * np.sqrt(err.size), n
        assert np.abs(err).max() <= 3e-2 * np.abs(want).max() + 1e-5, n
    assert_dlambda(grads["dlambda"].item(), ref["dlambda"], ref["dlambda_rss"])


@pytest.mark.parametrize("B,H,_Nq,Nk,d,dv,_causal,lam", CASES)
def test_decode_random(B, H, _Nq, Nk, d, dv, _causal, lam):
    q1, k1, q2, k2, v, _ = draw(B, H, 1, Nk, d, dv, seed=Nk)
    for splits in (0, 1, 3):
        pre = torch.empty((B, H, 1, dv), device="cuda")
        out = da.decode(q1, k1, q2, k2, v, lam, 0.8, num_splits=splits, o_prenorm=pre)
        torch.cuda.synchronize()
        assert da.last_device_error() == 0
        o_ref, y_ref = oracle.diffattn_fwd(*[t.cpu() for t in (q1, k1, q2, k2, v)], lam, 0.8)
        assert np.abs(pre.cpu().numpy() - o_ref).max() <= 1e-2
        assert np.abs(out.float().cpu().numpy() - y_ref).max() <= 3e-2
