"""The bounded-wait failure path on the GPU, made to run without a fault: a
diagnostic kernel waits for an mbarrier phase that nothing completes.  The
wait must end by itself, record its site code in the device error word, leave
the context usable, and the word must be cleared by reading it."""
import time

import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

SITE_SELFTEST = 0x601


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    assert da.last_device_error() == 0
    t0 = time.monotonic()
    da.selftest_wait_timeout()
    code = da.last_device_error()           # synchronises: the kernel has exited
    elapsed = time.monotonic() - t0
    assert code == SITE_SELFTEST
    assert 1.0 < elapsed < 30.0             # the 2 s device-side limit, not a hang
    assert da.last_device_error() == 0      # reading cleared the word
    # A normal call afterwards runs and matches the oracle.
    g = torch.Generator(device="cuda").manual_seed(1)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    q1, k1, q2, k2, v = mk(1, 2, 130, 64), mk(1, 2, 130, 64), mk(1, 2, 130, 64), mk(1, 2, 130, 64), mk(1, 2, 130, 128)
    pre = torch.empty((1, 2, 130, 128), dtype=torch.float32, device="cuda")
    da.fwd(q1, k1, q2, k2, v, 0.5, 0.8, causal=True, o_prenorm=pre)
    assert da.last_device_error() == 0
    o_ref, _ = oracle.diffattn_fwd(q1.cpu(), k1.cpu(), q2.cpu(), k2.cpu(), v.cpu(), 0.5, 0.8, causal=True)
    assert np.abs(pre.cpu().numpy() - o_ref).max() <= 1e-2
