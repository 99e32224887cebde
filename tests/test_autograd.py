"""The torch.autograd wrapper: it must return exactly what the C-ABI calls it
wraps return (it only marshals tensors), and chain the lambda and gamma
gradients into whatever produced them."""
import pytest
import torch

import transformer_attention_07_b300 as da
from transformer_attention_07_b300.autograd import diff_attn

pytestmark = pytest.mark.gpu


def make(B=1, H=2, Nq=200, Nk=200, d=64, dv=128, seed=3):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16)
    return (mk(B, H, Nq, d), mk(B, H, Nk, d), mk(B, H, Nq, d), mk(B, H, Nk, d), mk(B, H, Nk, dv),
            mk(B, H, Nq, dv), torch.rand(H * dv, generator=g, device="cuda") + 0.5)


@pytest.mark.parametrize("causal,d,dv", [(True, 64, 128), (False, 32, 64)])
def test_autograd_equals_the_direct_calls(causal, d, dv):
    q1, k1, q2, k2, v, dy, gamma = make(d=d, dv=dv, Nk=200 if causal else 150)
    a = torch.tensor(-0.5, device="cuda", requires_grad=True)
    b = torch.tensor(0.1, device="cuda", requires_grad=True)
    lam = torch.exp(a) - b                                  # a learnable lambda, as a function of parameters
    gam = gamma.clone().requires_grad_(True)
    leaves = [t.clone().requires_grad_(True) for t in (q1, k1, q2, k2, v)]
    y = diff_attn(*leaves, lam, 0.8, causal=causal, gamma=gam)
    y.backward(dy)
    torch.cuda.synchronize()
    lam_f = float(lam.detach())
    out, saved = da.fwd_train(q1, k1, q2, k2, v, lam_f, 0.8, causal=causal, gamma=gamma)
    ref = da.bwd(q1, k1, q2, k2, v, dy, saved, lam_f, 0.8, causal=causal, gamma=gamma)
    torch.cuda.synchronize()
    assert da.last_device_error() == 0
    assert torch.equal(y.detach(), out)
    for t, n in zip(leaves, ("dq1", "dk1", "dq2", "dk2", "dv")):
        assert torch.equal(t.grad, ref[n]), n
    assert torch.equal(gam.grad, ref["dgamma"])
    dl = ref["dlambda"].item()
    assert a.grad.item() == pytest.approx(dl * torch.exp(a).item(), rel=1e-6)
    assert b.grad.item() == pytest.approx(-dl, rel=1e-6)


def test_autograd_with_plain_float_lambda_and_no_gain():
    q1, k1, q2, k2, v, dy, _ = make(Nq=130, Nk=130, seed=5)
    leaves = [t.clone().requires_grad_(True) for t in (q1, k1, q2, k2, v)]
    y = diff_attn(*leaves, 0.6, 0.8, causal=True)
    y.backward(dy)
    out, saved = da.fwd_train(q1, k1, q2, k2, v, 0.6, 0.8, causal=True)
    ref = da.bwd(q1, k1, q2, k2, v, dy, saved, 0.6, 0.8, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(y.detach(), out)
    for t, n in zip(leaves, ("dq1", "dk1", "dq2", "dk2", "dv")):
        assert torch.equal(t.grad, ref[n]), n
