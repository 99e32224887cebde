"""The two multi-GPU layouts end to end, as two processes (gloo, world size
2) sharing the one GPU of the test machine.  The ranks' kernels never wait
on each other: every exchange is a host-side all-gather between launches.

* Sequence-sharded decode: each rank holds half of the key cache (unequal
  halves), runs the split kernel on its range (decode_partials), the partial
  softmax states are all-gathered and every rank merges them
  (decode_merge).  The result must match the single-process decode of the
  whole cache to fp32 rounding, and the fp64 oracle.
* Head-partitioned prefill: each rank computes its share of the B*H heads
  and the slices are all-gathered; every head is computed by the same
  kernel on the same inputs as in one call, so the gathered output must
  equal the single-process output bit for bit.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(B, H, Nq, Nk, d, dv, seed):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    inp = {"q1": mk(B, H, Nq, d), "k1": mk(B, H, Nk, d), "q2": mk(B, H, Nq, d), "k2": mk(B, H, Nk, d),
           "v": mk(B, H, Nk, dv)}
    inp["gamma"] = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    return inp


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    import transformer_attention_07_b300 as da
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = {"rank": rank}
        # --- sequence-sharded decode: rank 0 holds keys [0, 3000), rank 1 [3000, 7000)
        B, H, Nk, d, dv = 2, 4, 7000, 64, 128
        inp = _inputs(B, H, 1, Nk, d, dv, seed=77)
        cut = [0, 3000, Nk][rank:rank + 2]
        shard = {k: inp[k][:, :, cut[0]:cut[1]].contiguous() for k in ("k1", "k2", "v")}
        out = da.decode_sharded(inp["q1"], shard["k1"], inp["q2"], shard["k2"], shard["v"], 0.6, 0.8, num_splits=4,
                                gamma=inp["gamma"])
        pre_single = torch.empty((B, H, 1, dv), dtype=torch.float32, device="cuda")
        out_single = da.decode(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], 0.6, 0.8, gamma=inp["gamma"],
                               o_prenorm=pre_single)
        # the merged pre-norm output of the sharded path
        part = da.decode_partials(inp["q1"], shard["k1"], inp["q2"], shard["k2"], shard["v"], 4)
        pre_sharded = torch.empty_like(pre_single)
        da.decode_merge(da.gather_partials(part), B, H, 0.6, 0.8, gamma=inp["gamma"], o_prenorm=pre_sharded)
        torch.cuda.synchronize()
        res["device_error"] = da.last_device_error()
        res["dec_vs_single_pre"] = (pre_sharded - pre_single).abs().max().item()
        res["dec_vs_single_out"] = (out.float() - out_single.float()).abs().max().item()
        cpu = [inp[k].cpu() for k in ("q1", "k1", "q2", "k2", "v")]
        o_ref, y_ref = oracle.diffattn_fwd(*cpu, 0.6, 0.8, gamma=inp["gamma"].double().cpu().numpy())
        res["dec_vs_oracle_pre"] = float(np.abs(pre_sharded.cpu().numpy() - o_ref).max())
        res["dec_vs_oracle_out"] = float(np.abs(out.float().cpu().numpy() - y_ref).max())
        # --- head-partitioned prefill: 3 x 5 = 15 heads, causal, ragged length
        B, H, N = 3, 5, 700
        pin = _inputs(B, H, N, N, d, dv, seed=78)
        full = da.fwd_sharded(pin["q1"], pin["k1"], pin["q2"], pin["k2"], pin["v"], 0.5, 0.8, causal=True,
                              gamma=pin["gamma"], gather=True)
        single = da.fwd(pin["q1"], pin["k1"], pin["q2"], pin["k2"], pin["v"], 0.5, 0.8, causal=True,
                        gamma=pin["gamma"])
        torch.cuda.synchronize()
        res["prefill_equal"] = bool(torch.equal(full, single))
        res["device_error"] |= da.last_device_error()
        q.put(res)
    except Exception as e:  # report, then let the parent fail the test
        q.put({"rank": rank, "error": repr(e)})
    finally:
        dist.destroy_process_group()


def test_two_processes_sharded_decode_and_head_partitioned_prefill():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=600) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in results:
        assert "error" not in r, r
        assert r["device_error"] == 0
        assert r["dec_vs_single_pre"] < 1e-5, r
        assert r["dec_vs_single_out"] <= 2 ** -7, r   # one bf16 ulp at |y| < 2
        assert r["dec_vs_oracle_pre"] <= 1e-2 and r["dec_vs_oracle_out"] <= 3e-2, r
        assert r["prefill_equal"], r
