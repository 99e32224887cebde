"""GPU parity of the persistent grids (one CTA per SM walking the query tiles),
which the prefill and the single-map kernel use for key lengths up to 4096
when there are more query tiles than SMs (the prefill also up to 8192 keys
when its tile list is weight-major).

Every shape here has more tiles than the B300's SMs, so the call runs the
persistent form.  Two checks per shape:
  * each head's output equals, bit for bit, a call on that head alone (a few
    tiles, so the single-tile kernel): every tile is computed exactly once,
    by the same arithmetic, at the right (batch, head, rows);
  * sampled rows (first and last rows, tile boundaries) against the fp64
    oracle within the parity tolerances (1e-2 pre-norm, 3e-2 normalised).
The shapes cover ragged Nq < Nk, non-causal ragged keys, d = 32, and tile
counts that end in a partial round after rounds in both directions.  Under
causal masking the tile list is weight-major when every head's K and V fit
in 64 MB together (the first, third, fourth and sixth shapes; the sixth has
8192 keys) and (b, h)-major otherwise (the fifth, 335 MB).

The one-tile form under causal masking runs a 1-D grid in weight order
within groups of heads when at least four heads' K and V fit in 16 MB;
`test_grouped_one_tile_grid` checks it the same way, each head against a
call on that head alone (one head: the (b, h, tile) 3-D grid).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

TOL_PRE = 1e-2
TOL_OUT = 3e-2
def plan_form(B, H, Nq, Nk, d, dv, causal):
    """The launch form the prefill entry points take on this device."""
    return da.prefill_plan(B, H, Nq, Nk, d, dv, causal=causal, sms=sms())[0]


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def random_inputs(B, H, Nq, Nk, d, dv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    inp = {"q1": mk(B, H, Nq, d), "k1": mk(B, H, Nk, d), "q2": mk(B, H, Nq, d), "k2": mk(B, H, Nk, d),
           "v": mk(B, H, Nk, dv)}
    inp["gamma"] = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    return inp


def boundary_rows(Nq):
    rows = {0, 1, Nq - 1}
    for t in range(128, Nq, 128):
        rows.update({t - 1, t})
    return sorted(r for r in rows if 0 <= r < Nq)


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,causal,form", [
    (1, 80, 300, 1000, 64, 128, True, "persistent_weight"),    # Nq < Nk, ragged rows; 240 tiles
    (2, 50, 256, 777, 64, 128, False, "persistent"),           # non-causal, ragged keys; 200 tiles
    (3, 50, 640, 640, 64, 128, True, "persistent_weight"),     # 750 tiles: five rounds in alternating directions, then a partial one
    (1, 160, 200, 200, 32, 64, True, "persistent_weight"),     # d = 32, dv = 64; 320 tiles
    (4, 40, 640, 4096, 64, 128, True, "persistent"),           # 800 tiles, K/V 335 MB: the (b, h)-major list
    (1, 16, 2000, 8192, 64, 128, True, "persistent_weight"),   # 256 tiles, 8192 keys, K/V 64 MiB
])
def test_persistent_prefill(B, H, Nq, Nk, d, dv, causal, form):
    assert plan_form(B, H, Nq, Nk, d, dv, causal) == form
    lam, lam_init, eps = 0.6, 0.8, 1e-5
    inp = random_inputs(B, H, Nq, Nk, d, dv, seed=Nq * 7 + Nk + H)
    pre = torch.full((B, H, Nq, dv), float("nan"), dtype=torch.float32, device="cuda")
    out = da.fwd(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], lam, lam_init, causal=causal,
                 gamma=inp["gamma"], eps=eps, o_prenorm=pre)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0

    # Each head alone: the single-tile kernel, same arithmetic per tile.
    for b in range(B):
        for h in range(H):
            one = {k: inp[k][b:b + 1, h:h + 1].contiguous() for k in ("q1", "k1", "q2", "k2", "v")}
            pre1 = torch.empty((1, 1, Nq, dv), dtype=torch.float32, device="cuda")
            out1 = da.fwd(one["q1"], one["k1"], one["q2"], one["k2"], one["v"], lam, lam_init, causal=causal,
                          gamma=inp["gamma"][h * dv:(h + 1) * dv].contiguous(), eps=eps, o_prenorm=pre1)
            assert torch.equal(out1[0, 0], out[b, h]), (b, h)
            assert torch.equal(pre1[0, 0], pre[b, h]), (b, h)
    assert da.last_device_error() == 0

    rows = boundary_rows(Nq)
    cpu = [inp[k].cpu() for k in ("q1", "k1", "q2", "k2", "v")]
    o_ref, y_ref = oracle.diffattn_fwd(*cpu, lam, lam_init, causal=causal,
                                       gamma=inp["gamma"].double().cpu().numpy(), eps=eps, rows=rows)
    got_pre = pre.cpu().numpy()[:, :, rows]
    got_out = out.float().cpu().numpy()[:, :, rows]
    e_pre = np.abs(got_pre - o_ref).max()
    e_out = np.abs(got_out - y_ref).max()
    print(f"[parity] persistent prefill max-abs error: pre-norm {e_pre:.3e}, normalised {e_out:.3e}")
    assert np.isfinite(e_pre) and e_pre <= TOL_PRE
    assert np.isfinite(e_out) and e_out <= TOL_OUT


def test_persistent_single_map_kernel():
    B, H, N = 4, 40, 700            # 3 pairs of query tiles per head: 480 pairs
    assert B * H * math.ceil(N / 256) > sms()
    g = torch.Generator(device="cuda").manual_seed(4242)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = mk(B, H, N, 128), mk(B, H, N, 128), mk(B, H, N, 128)
    out32 = torch.full((B, H, N, 128), float("nan"), dtype=torch.float32, device="cuda")
    out = da.standard_fwd(q, k, v, causal=True, out_f32=out32)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    for b in range(B):
        for h in range(H):
            o1 = da.standard_fwd(q[b:b + 1, h:h + 1].contiguous(), k[b:b + 1, h:h + 1].contiguous(),
                                 v[b:b + 1, h:h + 1].contiguous(), causal=True)
            assert torch.equal(o1[0, 0], out[b, h]), (b, h)
    rows = boundary_rows(N)
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    o_ref, _ = oracle.diffattn_fwd(qc, kc, qc, kc, vc, 0.0, 0.0, causal=True, rows=rows)
    e32 = np.abs(out32.cpu().numpy()[:, :, rows] - o_ref).max()
    print(f"[parity] persistent single-map max-abs error: {e32:.3e}")
    assert np.isfinite(e32) and e32 <= 1e-2


@pytest.mark.parametrize("B,H,Nq,Nk", [
    (1, 12, 640, 5000),   # 60 tiles, 2.6 MB of K/V per head: groups of 6 heads
    (2, 5, 300, 6000),    # 30 tiles, 10 heads in groups of 5, ragged rows
])
def test_grouped_one_tile_grid(B, H, Nq, Nk):
    d, dv = 64, 128
    assert plan_form(B, H, Nq, Nk, d, dv, True) == "tile_grouped"
    lam, lam_init, eps = 0.6, 0.8, 1e-5
    inp = random_inputs(B, H, Nq, Nk, d, dv, seed=Nq + Nk + 5 * H)
    out = da.fwd(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], lam, lam_init, causal=True,
                 gamma=inp["gamma"], eps=eps)
    for b in range(B):
        for h in range(H):
            one = {k: inp[k][b:b + 1, h:h + 1].contiguous() for k in ("q1", "k1", "q2", "k2", "v")}
            out1 = da.fwd(one["q1"], one["k1"], one["q2"], one["k2"], one["v"], lam, lam_init, causal=True,
                          gamma=inp["gamma"][h * dv:(h + 1) * dv].contiguous(), eps=eps)
            assert torch.equal(out1[0, 0], out[b, h]), (b, h)
    g = torch.Generator(device="cuda").manual_seed(B * H + Nq)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = mk(B, H, Nq, 128), mk(B, H, Nk, 128), mk(B, H, Nk, 128)
    o = da.standard_fwd(q, k, v, causal=True)
    for b in range(B):
        for h in range(H):
            o1 = da.standard_fwd(q[b:b + 1, h:h + 1].contiguous(), k[b:b + 1, h:h + 1].contiguous(),
                                 v[b:b + 1, h:h + 1].contiguous(), causal=True)
            assert torch.equal(o1[0, 0], o[b, h]), (b, h)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
