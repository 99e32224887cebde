"""Out-of-bounds write checks without a sanitizer: every output buffer sits
inside a larger allocation whose margins hold a canary pattern (all-ones
bits: a NaN in every float format).  After each call on ragged shapes (tails
of partial 128-row tiles, keys not a multiple of the tile), the margins must
be untouched and the outputs must hold no canary."""
import pytest
import torch

import transformer_attention_07_b300 as da

pytestmark = pytest.mark.gpu

PAD = 4096   # elements before and after each output (keeps 16-byte alignment)


class Canaried:
    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        raw = torch.empty(n + 2 * PAD, dtype=dtype, device="cuda")
        raw.view(torch.int8 if dtype.itemsize == 1 else {2: torch.int16, 4: torch.int32}[dtype.itemsize]).fill_(-1)
        self.bufs.append((raw, n))
        return raw[PAD:PAD + n].view(shape)

    def check(self):
        torch.cuda.synchronize()
        assert da.last_device_error() == 0
        for raw, n in self.bufs:
            bits = raw.view({2: torch.int16, 4: torch.int32, 1: torch.int8}[raw.element_size()])
            assert bool((bits[:PAD] == -1).all()), "write before the output"
            assert bool((bits[PAD + n:] == -1).all()), "write after the output"
            assert not bool((bits[PAD:PAD + n] == -1).any()), "output element never written"


def inputs(B, H, Nq, Nk, d, dv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    return mk(B, H, Nq, d), mk(B, H, Nk, d), mk(B, H, Nq, d), mk(B, H, Nk, d), mk(B, H, Nk, dv)


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,causal", [
    (2, 3, 200, 333, 64, 128, True), (1, 2, 77, 130, 64, 128, False), (2, 2, 129, 129, 32, 64, True)])
def test_prefill_and_training_outputs_stay_in_bounds(B, H, Nq, Nk, d, dv, causal):
    q1, k1, q2, k2, v = inputs(B, H, Nq, Nk, d, dv, seed=Nq + Nk)
    c = Canaried()
    out, pre = c((B, H, Nq, dv), torch.bfloat16), c((B, H, Nq, dv), torch.float32)
    da.fwd(q1, k1, q2, k2, v, 0.5, 0.8, causal=causal, out=out, o_prenorm=pre)
    c.check()


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,causal", [(1, 2, 200, 333, 64, 128, True), (2, 1, 130, 70, 32, 64, False)])
def test_backward_gradients_stay_in_bounds(B, H, Nq, Nk, d, dv, causal):
    q1, k1, q2, k2, v = inputs(B, H, Nq, Nk, d, dv, seed=7 + Nq)
    g = torch.Generator(device="cuda").manual_seed(8)
    dy = torch.randn((B, H, Nq, dv), generator=g, device="cuda").to(torch.bfloat16)
    gamma = torch.rand(H * dv, generator=g, device="cuda") + 0.5
    _, saved = da.fwd_train(q1, k1, q2, k2, v, 0.5, 0.8, causal=causal, gamma=gamma)
    c = Canaried()
    grads = {"dq1": c(q1.shape, torch.bfloat16), "dk1": c(k1.shape, torch.bfloat16), "dq2": c(q2.shape, torch.bfloat16),
             "dk2": c(k2.shape, torch.bfloat16), "dv": c(v.shape, torch.bfloat16), "dlambda": c((1,), torch.float32),
             "dgamma": c((H * dv,), torch.float32)}
    da.bwd(q1, k1, q2, k2, v, dy, saved, 0.5, 0.8, causal=causal, gamma=gamma, grads=grads)
    c.check()


@pytest.mark.parametrize("B,H,Nk,d,dv", [(3, 5, 1000, 64, 128), (2, 3, 777, 32, 64)])
def test_decode_outputs_stay_in_bounds(B, H, Nk, d, dv):
    g = torch.Generator(device="cuda").manual_seed(Nk)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    q1, q2, k1, k2, v = mk(B, H, 1, d), mk(B, H, 1, d), mk(B, H, Nk, d), mk(B, H, Nk, d), mk(B, H, Nk, dv)
    c = Canaried()
    out, pre = c((B, H, 1, dv), torch.bfloat16), c((B, H, 1, dv), torch.float32)
    da.decode(q1, k1, q2, k2, v, 0.6, 0.8, out=out, o_prenorm=pre)
    c.check()


def test_standard_attention_outputs_stay_in_bounds():
    g = torch.Generator(device="cuda").manual_seed(5)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = mk(2, 2, 300, 128), mk(2, 2, 300, 128), mk(2, 2, 300, 128)
    c = Canaried()
    out, out32 = c((2, 2, 300, 128), torch.bfloat16), c((2, 2, 300, 128), torch.float32)
    da.standard_fwd(q, k, v, causal=True, out=out, out_f32=out32)
    c.check()
