"""The device-pointer entry points only enqueue kernels on the given stream:
they allocate nothing and never synchronise, so a whole step (prefill,
decode, training forward + backward) can be captured once in a CUDA graph and
replayed.  Replays must reproduce the eager results bit for bit (the same
kernels on the same data)."""
import pytest
import torch

import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu


def test_graph_replay_equals_eager():
    g = torch.Generator(device="cuda").manual_seed(0)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    B, H, N, Nk = 1, 4, 640, 4096
    q1, k1, q2, k2, v, dy = mk(B, H, N, 64), mk(B, H, N, 64), mk(B, H, N, 64), mk(B, H, N, 64), mk(B, H, N, 128), \
        mk(B, H, N, 128)
    dq1, dk1, dq2, dk2, dvv = mk(8, 4, 1, 64), mk(8, 4, Nk, 64), mk(8, 4, 1, 64), mk(8, 4, Nk, 64), mk(8, 4, Nk, 128)
    # every buffer the captured calls use is allocated up front
    out = torch.empty((B, H, N, 128), dtype=torch.bfloat16, device="cuda")
    dout = torch.empty((8, 4, 1, 128), dtype=torch.bfloat16, device="cuda")
    dws = torch.empty(da.decode_workspace_bytes(8, 4, Nk, 128, 8), dtype=torch.uint8, device="cuda")
    tout = torch.empty_like(out)
    saved = {"o_prenorm": torch.empty((B, H, N, 128), device="cuda"), "o2": torch.empty((B, H, N, 128), device="cuda"),
             "lse": torch.empty((2, B, H, N), device="cuda")}
    grads = {"dq1": torch.empty_like(q1), "dk1": torch.empty_like(k1), "dq2": torch.empty_like(q2),
             "dk2": torch.empty_like(k2), "dv": torch.empty_like(v), "dlambda": torch.empty(1, device="cuda"),
             "dgamma": torch.empty(H * 128, device="cuda")}
    bws = torch.empty(da.bwd_workspace_bytes(B, H, N, 128), dtype=torch.uint8, device="cuda")
    from transformer_attention_07_b300 import load, _ptr, _stream

    def step(stream):
        da.fwd(q1, k1, q2, k2, v, 0.6, 0.8, causal=True, out=out, stream=stream)
        da.decode(dq1, dk1, dq2, dk2, dvv, 0.6, 0.8, num_splits=8, workspace=dws, out=dout, stream=stream)
        rc = load().diffattn_fwd_train(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), 0.6, 0.8, 1, B, H, N, N, 64,
                                       128, None, 1e-5, _ptr(tout), _ptr(saved["o_prenorm"]), _ptr(saved["o2"]),
                                       _ptr(saved["lse"]), _stream(stream))
        assert rc == 0
        da.bwd(q1, k1, q2, k2, v, dy, saved, 0.6, 0.8, causal=True, workspace=bws, grads=grads, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)                      # eager, on the side stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, dout, tout)] + [grads[k].clone() for k in sorted(grads)]
    for t in (out, dout, tout, *grads.values()):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    replayed = [out, dout, tout] + [grads[k] for k in sorted(grads)]
    for a, b in zip(eager, replayed):
        assert torch.equal(a, b)
