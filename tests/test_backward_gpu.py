"""GPU parity of the backward (gdr_backward through the C ABI) against the float64 backward oracle.

The kernels compute in float32 throughout (bf16 q, k, v, dO are read as the same values the oracle
is given), so every gradient is held to the float32 path's bound: max|diff| <= 1e-4 max|ref| per
tensor. A float32 restatement of the same reverse pass lands near 1e-6 on these inputs, so the
bound leaves two orders of magnitude for the kernels' other summation orders.
"""
import numpy as np
import pytest
import torch

import oracle.backward as ob
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_F32, assert_close, dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def run(x, dO, dS_T):
    out = gdr.gdr_backward(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(x.S0), dev(dO), dev(dS_T))
    gdr.gdr_sync_status()
    return out


def check(x, dO, dS_T, tol=TOL_F32):
    got = run(x, dO, dS_T)
    want = ob.backward(x.q, x.k, x.v, x.g, x.beta, x.S0, dO, dS_T)
    for name, a, b in zip(NAMES, got, want):
        assert_close(a, b, tol, name)
    return got


@pytest.mark.parametrize("regime", ["R1", "R2", "R3", "R4"])
def test_backward_matches_oracle_f32(regime):
    """Three 32-token segments with a ragged tail of 6, two rows, two value heads per key head."""
    x = inputs.regime(regime, 70, 21, Hk=2, Hv=4, B=2, init_state=True)
    dO, dS_T = inputs.upstream_grads(2, 70, 4, 22)
    check(x, dO, dS_T)


def test_backward_matches_oracle_bf16_inputs():
    x = inputs.regime("R1", 100, 23, Hk=2, Hv=4, B=1, init_state=True, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(1, 100, 4, 24, dtype=torch.bfloat16)
    check(x, dO, dS_T)


@pytest.mark.parametrize("L", [1, 31, 32, 33, 64])
def test_backward_segment_edges_without_S0_or_dS_T(L):
    x = inputs.regime("R2", L, 25 + L, Hk=1, Hv=2, B=1)
    dO, _ = inputs.upstream_grads(1, L, 2, 26 + L, with_dS_T=False)
    check(x, dO, None)


def test_backward_pads_give_zero_dv_and_match_oracle():
    x = inputs.regime("R1", 80, 27, Hk=2, Hv=4, B=2, init_state=True, n_valid=50)
    dO, dS_T = inputs.upstream_grads(2, 80, 4, 28)
    got = check(x, dO, dS_T)
    assert torch.all(got[2][:, 50:] == 0), "dv at pads (beta = 0) must be exactly zero"


def test_backward_is_deterministic():
    x = inputs.regime("R3", 96, 29, Hk=2, Hv=8, B=2, init_state=True, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(2, 96, 8, 30, dtype=torch.bfloat16)
    a = run(x, dO, dS_T)
    b = run(x, dO, dS_T)
    for name, u, w in zip(NAMES, a, b):
        assert torch.equal(u, w), name


def test_backward_full_size_4096_sampled_key_head():
    """L = 4096, Hk = 16, Hv = 32 in bf16 (the prefill workload), checked on key head 0 and its
    two value heads: those gradients depend on no other head, so the oracle runs on that slice."""
    x = inputs.regime("R1", 4096, 31, Hk=16, Hv=32, B=1, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(1, 4096, 32, 32, dtype=torch.bfloat16)
    got = run(x, dO, dS_T)
    want = ob.backward(x.q[:, :, :1], x.k[:, :, :1], x.v[:, :, :2], x.g[:, :, :2], x.beta[:, :, :2], None,
                       dO[:, :, :2], dS_T[:, :2])
    sl = (got[0][:, :, :1], got[1][:, :, :1], got[2][:, :, :2], got[3][:, :, :2], got[4][:, :, :2], got[5][:, :2])
    for name, a, b in zip(NAMES, sl, want):
        assert_close(a, b, TOL_F32, name)
    for t in got:
        assert torch.isfinite(t).all()
