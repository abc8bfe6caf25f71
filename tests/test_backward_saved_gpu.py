"""GPU checks of the chunked backward without recomputation: gdr_chunk_fwd_save keeps the forward's
chunk factors and chunk-entry states, gdr_backward_chunked_saved runs only the adjoint chain and the
chunk-local gradients on them.

Both run the same kernels on the same data as the recomputing forms, so the checks are bit for bit:
the saving forward's o and S_T against gdr_chunk_fwd (rows longer than one chunk: the same two
kernels; rows of one chunk, which gdr_chunk_fwd finishes in one kernel, against the float64 oracle
at the bf16 bound), and the saved backward's gradients against gdr_backward_chunked's.
"""
import pytest
import torch

import oracle
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, assert_close, dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def both(x, dO, dS_T):
    args = [dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    o, S_T, saved = gdr.gdr_chunk_fwd_save(*args)
    got = gdr.gdr_backward_chunked(*args, dev(dO), dev(dS_T), saved=saved)
    want = gdr.gdr_backward_chunked(*args, dev(dO), dev(dS_T))
    gdr.gdr_sync_status()
    return (o, S_T), got, want


@pytest.mark.parametrize("regime,L,init", [("R1", 130, True), ("R3", 200, True), ("R2", 65, False), ("R4", 128, True)])
def test_saved_forward_and_backward_equal_the_recomputing_forms(regime, L, init):
    x = inputs.regime(regime, L, 111 + L, Hk=2, Hv=4, B=2, init_state=init, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(2, L, 4, 112 + L, dtype=torch.bfloat16, with_dS_T=init)
    (o, S_T), got, want = both(x, dO, dS_T)
    o_ref, S_ref = gdr.gdr_chunk_fwd(*[dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)])
    gdr.gdr_sync_status()
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
    for name, a, b in zip(NAMES, got, want):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("L", [1, 40, 64])
def test_saved_forms_on_rows_of_one_chunk(L):
    """gdr_chunk_fwd finishes these rows in one kernel; the saving forward takes the two-kernel path
    (the backward needs the factors): o and S_T against the oracle, the gradients bit for bit."""
    x = inputs.regime("R1", L, 121 + L, Hk=1, Hv=2, B=2, init_state=True, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(2, L, 2, 122 + L, dtype=torch.bfloat16)
    (o, S_T), got, want = both(x, dO, dS_T)
    ro, rS = oracle.forward(x.q, x.k, x.v, x.g, x.beta, x.S0)
    assert_close(o, ro, TOL_BF16, "o")
    assert_close(S_T, rS, TOL_BF16, "S_T")
    for name, a, b in zip(NAMES, got, want):
        assert torch.equal(a, b), name


def test_saved_forms_full_size_4096():
    x = inputs.regime("R1", 4096, 131, Hk=16, Hv=32, B=1, init_state=True, dtype=torch.bfloat16)
    dO, dS_T = inputs.upstream_grads(1, 4096, 32, 132, dtype=torch.bfloat16)
    (o, S_T), got, want = both(x, dO, dS_T)
    o_ref, S_ref = gdr.gdr_chunk_fwd(*[dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)])
    gdr.gdr_sync_status()
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
    for name, a, b in zip(NAMES, got, want):
        assert torch.equal(a, b), name
