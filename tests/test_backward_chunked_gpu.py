"""GPU parity of the chunked backward (gdr_backward_chunked through the C ABI) against the float64
backward oracle.

The chunked backward runs the forward's chunk factors again, the chunk-entry states and the
adjoint chain dS_c = Gamma_C dS_{c+1} + M'^T dS_{c+1} + Q'^T dO_c on tcgen05, and the chunk-local
gradients on warp-level tensor-core products, all with fp16 operands (bf16 for the raw q, k Gram
products) and float32 accumulation, like the bf16 forward. It is therefore held to the bf16 path's
bound: max|diff| <= 5e-3 max|ref| per gradient. Cases span one and several chunks, ragged tails,
the R1-R4 regimes, pads, no initial state or final-state gradient, and the full-size prefill row
sampled on one key head.
"""
import pytest
import torch

import oracle.backward as ob
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, assert_close, dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def run(x, dO, dS_T):
    out = gdr.gdr_backward_chunked(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(x.S0), dev(dO), dev(dS_T))
    gdr.gdr_sync_status()
    return out


def check(x, dO, dS_T):
    got = run(x, dO, dS_T)
    want = ob.backward(x.q, x.k, x.v, x.g, x.beta, x.S0, dO, dS_T)
    for name, a, b in zip(NAMES, got, want):
        assert_close(a, b, TOL_BF16, name)
    return got


@pytest.mark.parametrize("regime,L", [("R1", 150), ("R2", 200), ("R3", 130), ("R4", 100)])
def test_chunked_backward_matches_oracle(regime, L):
    """Two or more 64-token chunks with a ragged last chunk, two rows, two value heads per key head."""
    x = inputs.regime(regime, L, 41 + L, Hk=2, Hv=4, B=2, init_state=True, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(2, L, 4, 42 + L, dtype=torch.bfloat16)
    check(x, dO, dS_T)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 128])
def test_chunked_backward_chunk_edges_without_S0_or_dS_T(L):
    x = inputs.regime("R1", L, 43 + L, Hk=1, Hv=2, B=1, dtype=torch.bfloat16)
    dO, _ = inputs.upstream_grads(1, L, 2, 44 + L, dtype=torch.bfloat16, with_dS_T=False)
    check(x, dO, None)


def test_chunked_backward_pads_give_zero_dv():
    x = inputs.regime("R1", 150, 45, Hk=2, Hv=4, B=2, init_state=True, n_valid=90, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(2, 150, 4, 46, dtype=torch.bfloat16)
    got = check(x, dO, dS_T)
    assert torch.all(got[2][:, 90:] == 0), "dv at pads (beta = 0) must be exactly zero"


def test_chunked_backward_is_deterministic_and_agrees_with_the_token_loop():
    x = inputs.regime("R3", 192, 47, Hk=2, Hv=8, B=2, init_state=True, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(2, 192, 8, 48, dtype=torch.bfloat16)
    a = run(x, dO, dS_T)
    b = run(x, dO, dS_T)
    for name, u, w in zip(NAMES, a, b):
        assert torch.equal(u, w), name
    ref = gdr.gdr_backward(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(x.S0), dev(dO), dev(dS_T))
    gdr.gdr_sync_status()
    for name, u, w in zip(NAMES, a, ref):
        assert_close(u, w.double().cpu().numpy(), TOL_BF16, name + " against gdr_backward")


def test_chunked_backward_full_size_4096_sampled_key_head():
    """L = 4096, Hk = 16, Hv = 32 (the prefill workload) with S0 and dS_T, checked on key head 3 and
    its two value heads: those gradients depend on no other head, so the oracle runs on that slice."""
    x = inputs.regime("R1", 4096, 49, Hk=16, Hv=32, B=1, init_state=True, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(1, 4096, 32, 50, dtype=torch.bfloat16)
    got = run(x, dO, dS_T)
    kh, vh = slice(3, 4), slice(6, 8)
    want = ob.backward(x.q[:, :, kh], x.k[:, :, kh], x.v[:, :, vh], x.g[:, :, vh], x.beta[:, :, vh],
                       x.S0[:, vh], dO[:, :, vh], dS_T[:, vh])
    sl = (got[0][:, :, kh], got[1][:, :, kh], got[2][:, :, vh], got[3][:, :, vh], got[4][:, :, vh], got[5][:, vh])
    for name, a, b in zip(NAMES, sl, want):
        assert_close(a, b, TOL_BF16, name)
    for t in got:
        assert torch.isfinite(t).all()
