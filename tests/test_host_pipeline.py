"""GPU tests of the host-buffer prefill (diffattn_fwd_host): chunks of heads
copied in, computed and copied out on their own streams.  Each head runs the
same kernel as the device-resident call, so the output must be identical to
diffattn_fwd's bit for bit, whatever the chunking, and whether the host
memory is page-locked or not."""
import pytest
import torch

import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu


def inputs(B, H, Nq, Nk, d, dv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda n, w: torch.randn((B, H, n, w), generator=g, device="cuda").to(torch.bfloat16)
    dev = {"q1": mk(Nq, d), "k1": mk(Nk, d), "q2": mk(Nq, d), "k2": mk(Nk, d), "v": mk(Nk, dv)}
    gamma = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    return dev, gamma


@pytest.mark.parametrize("chunk", [0, 1, 2, 3, 5])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_call_equals_device_call(chunk, pinned):
    B, H, N = 2, 3, 300
    dev, gamma = inputs(B, H, N, N, 64, 128, seed=chunk)
    ref = da.fwd(dev["q1"], dev["k1"], dev["q2"], dev["k2"], dev["v"], 0.6, 0.8, causal=True, gamma=gamma)
    host = {k: (t.cpu().pin_memory() if pinned else t.cpu()) for k, t in dev.items()}
    out = da.fwd_host(host["q1"], host["k1"], host["q2"], host["k2"], host["v"], 0.6, 0.8, causal=True, gamma=gamma,
                      heads_per_chunk=chunk)
    torch.cuda.current_stream().synchronize()
    assert da.last_device_error() == 0
    assert torch.equal(out, ref.cpu())


def test_host_call_small_heads_noncausal():
    B, H, Nq, Nk = 1, 4, 128, 200
    dev, _ = inputs(B, H, Nq, Nk, 32, 64, seed=9)
    ref = da.fwd(dev["q1"], dev["k1"], dev["q2"], dev["k2"], dev["v"], 0.8, 0.8)
    host = {k: t.cpu().pin_memory() for k, t in dev.items()}
    out = da.fwd_host(host["q1"], host["k1"], host["q2"], host["k2"], host["v"], 0.8, 0.8, heads_per_chunk=3)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out, ref.cpu())


def test_host_call_orders_after_earlier_stream_work():
    """Inputs written by the caller's stream just before the call (the copies
    run on the library's own streams and must wait for that work)."""
    B, H, N = 1, 2, 256
    dev, gamma = inputs(B, H, N, N, 64, 128, seed=3)
    host = {k: torch.zeros_like(t, device="cpu").pin_memory() for k, t in dev.items()}
    s = torch.cuda.current_stream()
    torch.cuda._sleep(50_000_000)                  # keep the stream busy
    for k in host:
        host[k].copy_(dev[k], non_blocking=True)   # device -> pinned host on the caller's stream
    out = da.fwd_host(host["q1"], host["k1"], host["q2"], host["k2"], host["v"], 0.6, 0.8, causal=True, gamma=gamma)
    s.synchronize()
    ref = da.fwd(dev["q1"], dev["k1"], dev["q2"], dev["k2"], dev["v"], 0.6, 0.8, causal=True, gamma=gamma)
    assert torch.equal(out, ref.cpu())


def test_host_call_in_the_benchmarked_configuration():
    """The e2e leg of bench.py: long_64k (causal, B1 H16 N65536) from pinned host
    buffers with the default chunking equals the device-resident call."""
    from transformer_attention_07_b300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS["long_64k"]
    inp = make_inputs(w, device="cuda")
    names = ("q1", "k1", "q2", "k2", "v")
    ref = da.fwd(*(inp[k] for k in names), w.lam, w.lam_init, causal=w.causal, gamma=inp["gamma"], eps=w.eps)
    host = {k: inp[k].cpu().pin_memory() for k in names}
    out = da.fwd_host(*(host[k] for k in names), w.lam, w.lam_init, causal=w.causal, gamma=inp["gamma"], eps=w.eps)
    torch.cuda.current_stream().synchronize()
    assert da.last_device_error() == 0
    assert torch.equal(out, ref.cpu())
