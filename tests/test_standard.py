"""GPU parity of the single-map baseline (standard softmax attention,
d = dv = 128) against the fp64 oracle: with lambda = 0 the oracle's pre-norm
output is exactly softmax(Q K^T / sqrt d) V (pinned against torch's
scaled_dot_product_attention in test_oracle.py)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

TOL = 1e-2


def run(B, H, Nq, Nk, causal, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = mk(B, H, Nq, 128), mk(B, H, Nk, 128), mk(B, H, Nk, 128)
    out32 = torch.full((B, H, Nq, 128), float("nan"), dtype=torch.float32, device="cuda")
    out = da.standard_fwd(q, k, v, causal=causal, out_f32=out32)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    o_ref, _ = oracle.diffattn_fwd(qc, kc, qc, kc, vc, 0.0, 0.0, causal=causal)
    e32 = np.abs(out32.cpu().numpy() - o_ref).max()
    e16 = np.abs(out.float().cpu().numpy() - o_ref).max()
    print(f"[parity] standard attention max-abs error: fp32 {e32:.3e}, bf16 {e16:.3e}")
    assert np.isfinite(e32) and e32 <= TOL
    assert np.isfinite(e16) and e16 <= TOL


@pytest.mark.parametrize("B,H,Nq,Nk,causal", [
    (1, 2, 300, 300, True),      # one CTA pair of query tiles, ragged, diagonal
    (2, 1, 200, 333, False),     # ragged queries and keys
    (1, 2, 130, 400, True),      # Nq < Nk: bottom-right alignment
    (1, 1, 600, 600, True),      # two CTAs, second tile of a pair partly past Nq
    (2, 2, 512, 512, True),      # whole tiles
    (1, 1, 1, 77, False),        # one query
])
def test_standard_attention_matches_oracle(B, H, Nq, Nk, causal):
    run(B, H, Nq, Nk, causal, seed=Nq + 3 * Nk)


def test_standard_attention_2k_sampled():
    """The 2K causal shape used for the DiffAttn comparison, sampled rows."""
    B, H, N = 2, 4, 2048
    g = torch.Generator(device="cuda").manual_seed(77)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = mk(B, H, N, 128), mk(B, H, N, 128), mk(B, H, N, 128)
    out32 = torch.empty((B, H, N, 128), dtype=torch.float32, device="cuda")
    da.standard_fwd(q, k, v, causal=True, out_f32=out32)
    torch.cuda.synchronize()
    rows = [0, 1, 127, 128, 255, 256, 1000, 2047]
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    o_ref, _ = oracle.diffattn_fwd(qc, kc, qc, kc, vc, 0.0, 0.0, causal=True, rows=rows)
    assert np.abs(out32.cpu().numpy()[:, :, rows] - o_ref).max() <= TOL


@pytest.mark.parametrize("shape", [(8, 16, 2048), (4, 16, 4096)])
def test_standard_attention_benchmarked_configurations(shape):
    """The single-map baseline exactly as bench.py times it (its own inputs,
    causal, B8 H16 N2048 and B4 H16 N4096): sampled rows of every head."""
    from transformer_attention_07_b300.workloads import COMPARE_SHAPES, sample_rows, standard_inputs
    assert shape in COMPARE_SHAPES
    B, H, N = shape
    si = standard_inputs(B, H, N, device="cuda")
    out32 = torch.empty((B, H, N, 128), dtype=torch.float32, device="cuda")
    da.standard_fwd(si["q"], si["k"], si["v"], causal=True, out_f32=out32)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    rows = sample_rows(N, 2000 + N, n_random=8, edge=4)
    qc, kc, vc = si["q"].cpu(), si["k"].cpu(), si["v"].cpu()
    o_ref, _ = oracle.diffattn_fwd(qc, kc, qc, kc, vc, 0.0, 0.0, causal=True, rows=rows)
    assert np.abs(out32.cpu().numpy()[:, :, rows] - o_ref).max() <= TOL
