"""GPU tests of sequence-sharded decode: the key cache split into ranges of
different lengths (as different GPUs would hold them), partial states
computed per range, stacked as an all-gather would stack them, and merged.
The ranges run one after another on one GPU; nothing waits on anything
across ranges."""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu


def cache(B, H, N, d, dv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    return mk(B, H, 1, d), mk(B, H, N, d), mk(B, H, 1, d), mk(B, H, N, d), mk(B, H, N, dv)


@pytest.mark.parametrize("d,dv,lengths,splits", [(64, 128, (1000, 2048, 777), 4), (32, 64, (96, 31, 500), 2),
                                                 (64, 128, (4096,), 8)])
def test_sharded_ranges_merge_to_the_full_decode(d, dv, lengths, splits):
    B, H, N = 3, 4, sum(lengths)
    q1, k1, q2, k2, v = cache(B, H, N, d, dv, seed=N)
    g = torch.Generator(device="cuda").manual_seed(1)
    gamma = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    parts, k0 = [], 0
    for n in lengths:
        sl = lambda t: t[:, :, k0:k0 + n].contiguous()
        parts.append(da.decode_partials(q1, sl(k1), q2, sl(k2), sl(v), splits))
        k0 += n
    pre = torch.empty((B, H, 1, dv), device="cuda")
    out = da.decode_merge(torch.stack(parts), B, H, 0.6, 0.8, gamma=gamma, o_prenorm=pre)
    ref_pre = torch.empty_like(pre)
    ref = da.decode(q1, k1, q2, k2, v, 0.6, 0.8, gamma=gamma, o_prenorm=ref_pre)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    # the same algebra over different range boundaries: fp32 rounding only
    assert (pre - ref_pre).abs().max().item() <= 1e-4
    o_ref, y_ref = oracle.diffattn_fwd(*[t.cpu() for t in (q1, k1, q2, k2, v)], 0.6, 0.8,
                                       gamma=gamma.double().cpu())
    assert np.abs(pre.cpu().numpy() - o_ref).max() <= 1e-2
    assert np.abs(out.float().cpu().numpy() - y_ref).max() <= 3e-2


def test_one_part_equals_decode_bit_for_bit():
    B, H, N = 2, 3, 3000
    q1, k1, q2, k2, v = cache(B, H, N, 64, 128, seed=5)
    part = da.decode_partials(q1, k1, q2, k2, v, 6)
    out = da.decode_merge(part, B, H, 0.6, 0.8)
    ref = da.decode(q1, k1, q2, k2, v, 0.6, 0.8, num_splits=6)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_range_shorter_than_its_splits():
    """A range with fewer keys than splits x 32 leaves empty splits (m = -inf,
    l = 0), which the merge skips."""
    B, H = 1, 2
    q1, k1, q2, k2, v = cache(B, H, 40 + 3000, 64, 128, seed=8)
    a = da.decode_partials(q1, k1[:, :, :40].contiguous(), q2, k2[:, :, :40].contiguous(),
                           v[:, :, :40].contiguous(), 4)
    b = da.decode_partials(q1, k1[:, :, 40:].contiguous(), q2, k2[:, :, 40:].contiguous(),
                           v[:, :, 40:].contiguous(), 4)
    torch.cuda.synchronize()
    assert torch.isinf(a[:, 2:, :, 0]).all() and (a[:, 2:, :, 1] == 0).all()
    pre = torch.empty((B, H, 1, 128), device="cuda")
    da.decode_merge(torch.stack([a, b]), B, H, 0.6, 0.8, o_prenorm=pre)
    o_ref, _ = oracle.diffattn_fwd(*[t.cpu() for t in (q1, k1, q2, k2, v)], 0.6, 0.8)
    torch.cuda.synchronize()
    assert np.abs(pre.cpu().numpy() - o_ref).max() <= 1e-2
