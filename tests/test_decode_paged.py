"""GPU tests of the paged, variable-length split-KV decode.

* A contiguous cache cut into shuffled pages gives bit-for-bit the result of
  the contiguous decode (same keys, same chunking, same split count).
* Variable sequence lengths against the fp64 oracle, which sees each
  sequence's keys gathered back into order (input preparation only).
* Out-of-range table entries and lengths are clamped on the device and
  reported through the device error word, never dereferenced.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

TOL_PRE, TOL_OUT = 1e-2, 3e-2


def make_paged(B, H, max_len, d, dv, page_size, seed, extra_pages=3):
    """Random contiguous caches [B,H,max_len,*], and the same data in shuffled
    pages plus a few unused pages."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    k1, k2, v = mk(B, H, max_len, d), mk(B, H, max_len, d), mk(B, H, max_len, dv)
    q1, q2 = mk(B, H, 1, d), mk(B, H, 1, d)
    max_pages = max_len // page_size
    num_pages = B * max_pages + extra_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed))[: B * max_pages]
    table = perm.view(B, max_pages).to(torch.int32)
    pages = {}
    for name, t, w in (("k1", k1, d), ("k2", k2, d), ("v", v, dv)):
        pg = mk(num_pages, H, page_size, w)   # unused pages hold noise
        src = t.view(B, H, max_pages, page_size, w).permute(0, 2, 1, 3, 4).reshape(B * max_pages, H, page_size, w)
        pg[perm.to("cuda")] = src
        pages[name] = pg.contiguous()
    return {"q1": q1, "q2": q2, "k1": k1, "k2": k2, "v": v, "pages": pages, "table": table.cuda(),
            "max_pages": max_pages, "page_size": page_size}


def paged_decode(c, seq_lens, lam=0.6, splits=0, gamma=None):
    B, H = c["q1"].shape[:2]
    dv = c["v"].shape[3]
    pre = torch.full((B, H, 1, dv), float("nan"), dtype=torch.float32, device="cuda")
    out = da.decode_paged(c["q1"], c["q2"], c["pages"]["k1"], c["pages"]["k2"], c["pages"]["v"], c["table"],
                          torch.tensor(seq_lens, dtype=torch.int32, device="cuda"), lam, 0.8, gamma=gamma,
                          num_splits=splits, o_prenorm=pre)
    torch.cuda.synchronize()
    return out, pre


@pytest.mark.parametrize("page_size,splits", [(64, 0), (32, 7), (256, 3), (128, 1)])
def test_paged_equals_contiguous(page_size, splits):
    c = make_paged(3, 4, 2048, 64, 128, page_size, seed=page_size + splits)
    out_p, pre_p = paged_decode(c, [2048] * 3, splits=splits)
    assert da.last_device_error() == 0
    pre_c = torch.empty_like(pre_p)
    out_c = da.decode(c["q1"], c["k1"], c["q2"], c["k2"], c["v"], 0.6, 0.8, num_splits=splits, o_prenorm=pre_c)
    torch.cuda.synchronize()
    if splits:
        assert torch.equal(pre_p, pre_c) and torch.equal(out_p, out_c)
    else:
        assert (pre_p - pre_c).abs().max().item() < 1e-5


@pytest.mark.parametrize("d,dv,page_size", [(64, 128, 64), (32, 64, 32)])
def test_variable_lengths_match_oracle(d, dv, page_size):
    B, H, max_len = 5, 3, 1024
    c = make_paged(B, H, max_len, d, dv, page_size, seed=11 + d)
    lens = [1, 31, 32, 700, 1024]
    g = torch.Generator(device="cuda").manual_seed(3)
    gamma = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    out, pre = paged_decode(c, lens, gamma=gamma)
    assert da.last_device_error() == 0
    for b, n in enumerate(lens):
        sl = lambda t: t[b:b + 1, :, :n].cpu()
        o_ref, y_ref = oracle.diffattn_fwd(c["q1"][b:b + 1].cpu(), sl(c["k1"]), c["q2"][b:b + 1].cpu(), sl(c["k2"]),
                                           sl(c["v"]), 0.6, 0.8, gamma=gamma.double().cpu().numpy())
        assert np.abs(pre[b:b + 1].cpu().numpy() - o_ref).max() <= TOL_PRE
        assert np.abs(out[b:b + 1].float().cpu().numpy() - y_ref).max() <= TOL_OUT


def test_bad_table_entries_and_lengths_are_reported_not_read():
    c = make_paged(2, 2, 256, 64, 128, 64, seed=5)
    num_pages = c["pages"]["k1"].shape[0]
    c["table"][1, 2] = num_pages + 7             # out of range: clamped to page 0, reported
    paged_decode(c, [256, 256])
    assert da.last_device_error() == 0x301
    c["table"][1, 2] = 0
    paged_decode(c, [256, 0])                    # empty sequence: clamped to one key, reported
    assert da.last_device_error() == 0x302
    out, pre = paged_decode(c, [256, 100])
    assert da.last_device_error() == 0 and torch.isfinite(pre).all()


def test_paged_decode_32k_pages_of_64():
    """Full decode size (B=32, H=32, 32768 keys) in pages of 64: sampled heads
    against the oracle."""
    B, H, N = 32, 32, 32768
    c = make_paged(B, H, N, 64, 128, 64, seed=21, extra_pages=0)
    lens = [N - 997 * b for b in range(B)]
    out, pre = paged_decode(c, lens)
    assert da.last_device_error() == 0
    gen = torch.Generator().manual_seed(9)
    for idx in torch.randperm(B * H, generator=gen)[:6].tolist():
        b, h = divmod(idx, H)
        n = lens[b]
        sl = lambda t: t[b:b + 1, h:h + 1, :n].cpu()
        o_ref, _ = oracle.diffattn_fwd(c["q1"][b:b + 1, h:h + 1].cpu(), sl(c["k1"]), c["q2"][b:b + 1, h:h + 1].cpu(),
                                       sl(c["k2"]), sl(c["v"]), 0.6, 0.8)
        assert np.abs(pre[b, h].cpu().numpy() - o_ref[0, 0]).max() <= TOL_PRE
