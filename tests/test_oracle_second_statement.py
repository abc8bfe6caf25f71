"""Pin: the oracle against the second statement of the recurrence on the pages.

The DEG page "model.py" states the same per-token rule a second time, in function
delta_rule_reference: the state is a [B, H, K, V] tensor, the read is a product-and-sum over the
key axis, and the head interleave is repeat_interleave on q and k (function _linear_layer). This
test restates that formulation in float64 PyTorch (broadcast products summed over the key axis,
whole-batch tensors, no per-head loop) and compares it with the oracle's C token loop at D = 8,
with and without an initial state, with pads (beta = g = 0) and with r = 2 head sharing.
"""
import numpy as np
import pytest
import torch

import oracle


def _second_statement(q, k, v, g, beta, S0):
    """float64 restatement of DEG delta_rule_reference after its repeat_interleave head map."""
    r = v.shape[2] // q.shape[2]
    q = torch.repeat_interleave(q, r, dim=2)
    k = torch.repeat_interleave(k, r, dim=2)
    q = q * torch.rsqrt((q * q).sum(-1, keepdim=True) + 1e-6) * q.shape[-1] ** -0.5
    k = k * torch.rsqrt((k * k).sum(-1, keepdim=True) + 1e-6)
    B, L, H, K = k.shape
    state = S0.clone() if S0 is not None else torch.zeros(B, H, K, v.shape[-1], dtype=torch.float64)
    outs = []
    for t in range(L):
        state = state * torch.exp(g[:, t])[:, :, None, None]
        read = (state * k[:, t, :, :, None]).sum(dim=2)                 # [B, H, V]
        delta = beta[:, t][:, :, None] * (v[:, t] - read)
        state = state + k[:, t, :, :, None] * delta[:, :, None, :]
        outs.append((state * q[:, t, :, :, None]).sum(dim=2))
    return torch.stack(outs, dim=1), state


@pytest.mark.parametrize("with_s0,pads", [(True, False), (False, False), (True, True)])
def test_oracle_matches_the_second_statement(with_s0, pads):
    gen = torch.Generator().manual_seed(71 + 2 * with_s0 + pads)
    B, L, Hk, Hv, D = 2, 23, 2, 4, 8
    q = torch.randn(B, L, Hk, D, generator=gen, dtype=torch.float64)
    k = torch.randn(B, L, Hk, D, generator=gen, dtype=torch.float64)
    v = torch.randn(B, L, Hv, D, generator=gen, dtype=torch.float64)
    beta = 0.2 + 0.7 * torch.rand(B, L, Hv, generator=gen, dtype=torch.float64)
    g = -(0.05 + 2.95 * torch.rand(B, L, Hv, generator=gen, dtype=torch.float64))
    S0 = 0.1 * torch.randn(B, Hv, D, D, generator=gen, dtype=torch.float64) if with_s0 else None
    if pads:
        beta[:, 17:] = 0.0
        g[:, 17:] = 0.0
    o_ref, S_ref = _second_statement(q, k, v, g, beta, S0)
    o, S_T = oracle.forward(q, k, v, g, beta, S0)
    np.testing.assert_allclose(o, o_ref.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S_T, S_ref.numpy(), rtol=1e-12, atol=1e-13)
