"""Pins of the backward oracle (oracle/backward.py): central finite differences of the pinned
forward oracle for every input, autograd of a float64 PyTorch statement of the recurrence, and the
special cases the forward fixes (pads pass gradients through unchanged, L = 1)."""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.backward as ob


def _inputs(B=1, L=5, Hk=1, Hv=2, D=4, seed=3, S0=True):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, L, Hk, D, generator=gen).double().numpy()
    k = torch.randn(B, L, Hk, D, generator=gen).double().numpy()
    v = torch.randn(B, L, Hv, D, generator=gen).double().numpy()
    g = -(0.05 + 0.5 * torch.rand(B, L, Hv, generator=gen)).double().numpy()
    beta = (0.2 + 0.7 * torch.rand(B, L, Hv, generator=gen)).double().numpy()
    s0 = (0.3 * torch.randn(B, Hv, D, D, generator=gen)).double().numpy() if S0 else None
    dO = torch.randn(B, L, Hv, D, generator=gen).double().numpy()
    dS = torch.randn(B, Hv, D, D, generator=gen).double().numpy()
    return q, k, v, g, beta, s0, dO, dS


def _loss(q, k, v, g, beta, S0, dO, dS):
    o, S = oracle.forward(q, k, v, g, beta, S0)
    return float((o * dO).sum() + (S * dS).sum())


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta", "S0"])
def test_backward_matches_central_differences_of_the_forward_oracle(name):
    args = list(_inputs())
    idx = ["q", "k", "v", "g", "beta", "S0"].index(name)
    grads = ob.backward(*args)
    x = args[idx]
    fd = np.zeros_like(x)
    h = 1e-6
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        mi = it.multi_index
        keep = x[mi]
        x[mi] = keep + h
        lp = _loss(*args)
        x[mi] = keep - h
        lm = _loss(*args)
        x[mi] = keep
        fd[mi] = (lp - lm) / (2 * h)
    got = grads[idx]
    assert np.abs(got - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max()), (name, np.abs(got - fd).max())


def _torch_forward(q, k, v, g, beta, S0):
    """A float64 PyTorch statement of the same recurrence, differentiated by autograd."""
    B, L, Hk, D = q.shape
    Hv = v.shape[2]
    r = Hv // Hk
    qn = q / torch.sqrt((q * q).sum(-1, keepdim=True) + 1e-6) / math.sqrt(D)
    kn = k / torch.sqrt((k * k).sum(-1, keepdim=True) + 1e-6)
    outs, states = [], []
    for b in range(B):
        for h in range(Hv):
            S = S0[b, h]
            ob_ = []
            for t in range(L):
                S = torch.exp(g[b, t, h]) * S
                kv = S.T @ kn[b, t, h // r]
                S = S + torch.outer(kn[b, t, h // r], beta[b, t, h] * (v[b, t, h] - kv))
                ob_.append(S.T @ qn[b, t, h // r])
            outs.append(torch.stack(ob_))
            states.append(S)
    return outs, states


def test_backward_matches_autograd_of_a_pytorch_recurrence():
    q, k, v, g, beta, s0, dO, dS = _inputs(B=2, L=7, Hk=2, Hv=4, D=6, seed=5)
    ts = [torch.tensor(a, requires_grad=True) for a in (q, k, v, g, beta, s0)]
    outs, states = _torch_forward(*ts)
    B, L, Hv = q.shape[0], q.shape[1], v.shape[2]
    loss = 0.0
    for i, (o, S) in enumerate(zip(outs, states)):
        b, h = divmod(i, Hv)
        loss = loss + (o * torch.tensor(dO[b, :, h])).sum() + (S * torch.tensor(dS[b, h])).sum()
    auto = torch.autograd.grad(loss, ts)
    mine = ob.backward(q, k, v, g, beta, s0, dO, dS)
    for name, a, m in zip(["q", "k", "v", "g", "beta", "S0"], auto, mine):
        a = a.numpy()
        assert np.abs(a - m).max() <= 1e-12 * max(1.0, np.abs(a).max()), name


def test_pads_pass_the_state_gradient_through_unchanged():
    """At a pad (beta = g = 0) the step is the identity on S, so dS0 of a padded row equals dS0 of
    the row without the pads; the pads' own dv is zero."""
    q, k, v, g, beta, s0, dO, dS = _inputs(L=6, seed=9)
    g[:, 4:] = 0.0
    beta[:, 4:] = 0.0
    dO[:, 4:] = 0.0
    full = ob.backward(q, k, v, g, beta, s0, dO, dS)
    cut = ob.backward(q[:, :4], k[:, :4], v[:, :4], g[:, :4], beta[:, :4], s0, dO[:, :4], dS)
    assert np.allclose(full[5], cut[5], rtol=1e-13, atol=1e-15)
    assert np.all(full[2][:, 4:] == 0.0)


def test_single_token_closed_form_of_dv_and_dbeta():
    """L = 1: S_1 = e^g S0 + k^ beta (v - e^g S0^T k^)^T and o = S_1^T q~, so with dS_T = 0,
    dv = beta (k^ . q~) dO and dbeta = (k^ . q~) dO . (v - e^g S0^T k^)."""
    q, k, v, g, beta, s0, dO, _ = _inputs(L=1, seed=11)
    grads = ob.backward(q, k, v, g, beta, s0, dO, None)
    D = q.shape[-1]
    for h in range(2):
        qt = q[0, 0, 0] / math.sqrt((q[0, 0, 0] ** 2).sum() + 1e-6) / math.sqrt(D)
        kh = k[0, 0, 0] / math.sqrt((k[0, 0, 0] ** 2).sum() + 1e-6)
        Sa = math.exp(g[0, 0, h]) * s0[0, h]
        c = kh @ qt
        assert np.allclose(grads[2][0, 0, h], beta[0, 0, h] * c * dO[0, 0, h], rtol=1e-13)
        assert math.isclose(grads[4][0, 0, h], c * dO[0, 0, h] @ (v[0, 0, h] - Sa.T @ kh), rel_tol=1e-12)
