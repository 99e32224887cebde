"""The decode entry point that allocates nothing (diffattn_decode_noalloc).

It is meant for callers that cannot allocate device memory where they call
the library: for instance an operator inside a serving framework that owns
all device memory through a pool planned ahead of time, or a plugin interface
that hands over only input and output pointers.  Instead of a caller-owned
workspace it keeps the decode's per-split partials in one static 8 MiB array
inside the library.

These tests call it through the C ABI, two calls in a row each time (the
scratch keeps the previous call's contents), and check:
  * bit for bit against the workspace entry point (diffattn_decode) when both
    run the same split count: the same kernels on the same partials layout;
  * against the fp64 oracle, on every head of the smaller problems and on
    sampled heads of a 300-head problem in automatic mode;
  * that the free device memory does not change across the calls;
  * that a problem too large for the scratch, even at one split, is refused
    without a launch.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

TOL_PRE = 1e-2
TOL_OUT = 3e-2
ERR_INVALID_ARG = 1
ERR_WORKSPACE = 4
SCRATCH_BYTES = 8 << 20


def noalloc_fn():
    f = da.load().diffattn_decode_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, vp, f32, i32, vp, vp, vp]
    f.restype = i32
    return f


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def random_cache(B, H, Nk, d, dv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    return {"q1": mk(B, H, 1, d), "k1": mk(B, H, Nk, d), "q2": mk(B, H, 1, d), "k2": mk(B, H, Nk, d),
            "v": mk(B, H, Nk, dv), "gamma": torch.rand(H * dv, generator=g, device="cuda") + 0.5}


def nan_outputs(inp):
    B, H = inp["q1"].shape[:2]
    dv = inp["v"].shape[3]
    return (torch.full((B, H, 1, dv), float("nan"), dtype=torch.bfloat16, device="cuda"),
            torch.full((B, H, 1, dv), float("nan"), dtype=torch.float32, device="cuda"))


def run_noalloc(inp, lam, lam_init, splits=0, q1=None, outputs=None):
    B, H, _, d = inp["q1"].shape
    Nk, dv = inp["k1"].shape[2], inp["v"].shape[3]
    out, pre = nan_outputs(inp) if outputs is None else outputs
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = noalloc_fn()(ptr(inp["q1"]) if q1 is None else q1, ptr(inp["k1"]), ptr(inp["q2"]), ptr(inp["k2"]),
                      ptr(inp["v"]), lam, lam_init, B, H, Nk, d, dv, ptr(inp["gamma"]), 1e-5, splits, ptr(out),
                      ptr(pre), stream)
    return rc, out, pre


def run_workspace(inp, lam, lam_init, splits=0):
    B, H, _, _ = inp["q1"].shape
    dv = inp["v"].shape[3]
    pre = torch.empty((B, H, 1, dv), dtype=torch.float32, device="cuda")
    out = da.decode(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], lam, lam_init, gamma=inp["gamma"],
                    eps=1e-5, num_splits=splits, o_prenorm=pre)
    return out, pre


def oracle_heads(inp, lam, lam_init, heads):
    """fp64 oracle on the given flat (b * H + h) heads: (o_pre, y), [n, 1, 1, dv]."""
    H = inp["q1"].shape[1]
    sel = {k: torch.stack([inp[k][i // H, i % H] for i in heads])[:, None].cpu()
           for k in ("q1", "k1", "q2", "k2", "v")}
    dv = inp["v"].shape[3]
    gam = inp["gamma"].double().cpu().numpy()
    out_pre, out_y = [], []
    # One call per head so that each head's own gain slice applies.
    for n, i in enumerate(heads):
        g = gam[(i % H) * dv:(i % H + 1) * dv]
        o, y = oracle.diffattn_fwd(*[sel[k][n:n + 1] for k in ("q1", "k1", "q2", "k2", "v")], lam, lam_init,
                                   causal=False, gamma=g, eps=1e-5)
        out_pre.append(o)
        out_y.append(y)
    return np.concatenate(out_pre), np.concatenate(out_y)


def flat(t, heads):
    H = t.shape[1]
    return torch.stack([t[i // H, i % H] for i in heads])[:, None].float().cpu().numpy()


def test_noalloc_equals_workspace_entry_point_bitwise_and_matches_oracle():
    cases = [((2, 3, 3000, 64, 128), 21, 0.6, 0), ((4, 8, 1000, 64, 128), 22, 0.3, 5),
             ((2, 2, 2500, 32, 64), 24, 0.5, 0)]
    for (B, H, Nk, d, dv), seed, lam, splits in cases:
        inp = random_cache(B, H, Nk, d, dv, seed)
        ref_out, ref_pre = run_workspace(inp, lam, 0.8, splits)
        outputs = [nan_outputs(inp) for _ in range(2)]
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for i in range(2):   # two calls in a row: the scratch holds the first call's partials
            rc, out, pre = run_noalloc(inp, lam, 0.8, splits, outputs=outputs[i])
            torch.cuda.synchronize()
            assert rc == 0, da.status_string(rc)
            assert da.last_device_error() == 0
            assert torch.equal(pre, ref_pre) and torch.equal(out, ref_out)
        assert torch.cuda.mem_get_info()[0] == free0
        heads = list(range(B * H))
        o_ref, y_ref = oracle_heads(inp, lam, 0.8, heads)
        assert np.abs(flat(pre, heads) - o_ref).max() <= TOL_PRE
        assert np.abs(flat(out, heads) - y_ref).max() <= TOL_OUT


def test_noalloc_automatic_split_count_fits_and_matches_the_workspace_entry_point():
    """B=1, H=300, Nk=16384 with num_splits = 0: the no-alloc call picks its
    key-range count with the workspace entry point's model, capped to what
    the scratch holds (26 ranges here).  The model's pick fits, so both entry
    points run the same count and must agree bit for bit.  (The cap itself is
    host arithmetic, checked without a GPU through diffattn_decode_auto_splits.)"""
    B, H, Nk, d, dv = 1, 300, 16384, 64, 128
    per_split = B * H * 2 * (dv + 4) * 4
    fit = SCRATCH_BYTES // per_split
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    auto = da.decode_auto_splits(B, H, Nk, d, dv, sms)
    assert auto == da.decode_auto_splits(B, H, Nk, d, dv, sms, min(fit, 32))
    inp = random_cache(B, H, Nk, d, dv, 25)
    ref_out, ref_pre = run_workspace(inp, 0.6, 0.8, 0)
    outputs = [nan_outputs(inp) for _ in range(2)]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    outs = []
    for i in range(2):
        rc, out, pre = run_noalloc(inp, 0.6, 0.8, 0, outputs=outputs[i])
        torch.cuda.synchronize()
        assert rc == 0, da.status_string(rc)
        assert da.last_device_error() == 0
        outs.append((out, pre))
    assert torch.cuda.mem_get_info()[0] == free0
    for out, pre in outs:
        assert torch.equal(out, ref_out) and torch.equal(pre, ref_pre)
    out, pre = outs[1]
    heads = torch.randperm(B * H, generator=torch.Generator().manual_seed(26))[:32].tolist()
    o_ref, y_ref = oracle_heads(inp, 0.6, 0.8, heads)
    assert np.abs(flat(pre, heads) - o_ref).max() <= TOL_PRE
    assert np.abs(flat(out, heads) - y_ref).max() <= TOL_OUT


def test_noalloc_refuses_problems_larger_than_its_scratch():
    B, H, Nk, d, dv, splits = 16, 32, 64, 64, 128, 64
    assert B * H * splits * 2 * (dv + 4) * 4 > SCRATCH_BYTES
    inp = random_cache(B, H, Nk, d, dv, 23)
    rc, out, pre = run_noalloc(inp, 0.5, 0.8, splits)
    torch.cuda.synchronize()
    assert rc == ERR_WORKSPACE
    assert torch.isnan(pre).all()          # nothing was launched
    # the largest split count that fits still runs
    fit = SCRATCH_BYTES // (B * H * 2 * (dv + 4) * 4)
    rc, out, pre = run_noalloc(inp, 0.5, 0.8, int(fit))
    torch.cuda.synchronize()
    assert rc == 0 and torch.isfinite(pre).all()
    # more heads than one split each can hold: refused in automatic mode too
    B, H, Nk = 64, 128, 32
    assert B * H * 2 * (dv + 4) * 4 > SCRATCH_BYTES
    big = random_cache(B, H, Nk, d, dv, 27)
    rc, out, pre = run_noalloc(big, 0.5, 0.8, 0)
    torch.cuda.synchronize()
    assert rc == ERR_WORKSPACE and torch.isnan(pre).all()
    # an invalid argument is reported as such, not as a scratch problem
    rc, out, pre = run_noalloc(inp, 0.5, 0.8, 0, q1=ctypes.c_void_p(0))
    assert rc == ERR_INVALID_ARG and torch.isnan(pre).all()
