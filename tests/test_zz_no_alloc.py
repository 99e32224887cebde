"""The decode entry point that allocates nothing (diffattn_decode_noalloc).

It is meant for callers that cannot allocate device memory where they call
the library: for instance an operator inside a serving framework that owns
all device memory through a pool planned ahead of time, or a plugin interface
that hands over only input and output pointers.  Instead of a caller-owned
workspace it keeps the decode's per-split partials in one static 8 MiB array
inside the library.

These tests call it through the C ABI and check it against the workspace
entry point (diffattn_decode) on two calls in a row (the scratch keeps the
previous call's contents), and check that a problem too large for the
scratch is refused without a launch.
"""
import ctypes

import numpy as np
import pytest
import torch

import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

TOL_PRE = 1e-2
TOL_OUT = 3e-2
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


def run_noalloc(inp, lam, lam_init, splits=0):
    B, H, _, d = inp["q1"].shape
    Nk, dv = inp["k1"].shape[2], inp["v"].shape[3]
    out = torch.full((B, H, 1, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    pre = torch.full((B, H, 1, dv), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = noalloc_fn()(ptr(inp["q1"]), ptr(inp["k1"]), ptr(inp["q2"]), ptr(inp["k2"]), ptr(inp["v"]), lam, lam_init,
                      B, H, Nk, d, dv, ptr(inp["gamma"]), 1e-5, splits, ptr(out), ptr(pre), stream)
    return rc, out, pre


def run_workspace(inp, lam, lam_init, splits=0):
    B, H, _, _ = inp["q1"].shape
    dv = inp["v"].shape[3]
    pre = torch.empty((B, H, 1, dv), dtype=torch.float32, device="cuda")
    out = da.decode(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], lam, lam_init, gamma=inp["gamma"],
                    eps=1e-5, num_splits=splits, o_prenorm=pre)
    return out, pre


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    cases = [((2, 3, 3000, 64, 128), 21, 0.6, 0), ((4, 8, 1000, 64, 128), 22, 0.3, 5)]
    for (B, H, Nk, d, dv), seed, lam, splits in cases:
        inp = random_cache(B, H, Nk, d, dv, seed)
        ref_out, ref_pre = run_workspace(inp, lam, 0.8, splits)
        rc, out, pre = run_noalloc(inp, lam, 0.8, splits)
        torch.cuda.synchronize()
        assert rc == 0, da.status_string(rc)
        assert da.last_device_error() == 0
        e_pre = (pre - ref_pre).abs().max().item()
        e_out = (out.float() - ref_out.float()).abs().max().item()
        assert np.isfinite(e_pre) and e_pre <= TOL_PRE
        assert np.isfinite(e_out) and e_out <= TOL_OUT


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
