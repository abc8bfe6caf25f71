"""GPU parity of the variable-length prefill (gdr_chunk_fwd_varlen; DEG "model.py": Backbone.forward
over right-padded rows with State.lengths): each row runs only its first lengths[b] tokens, whatever g
and beta hold past it; its outputs there match the oracle on the truncated row, its final state is
the oracle's state after its last valid token, and o past the length is left untouched."""
import pytest
import torch

import oracle
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, TOL_F32, assert_close, dev

pytestmark = pytest.mark.gpu


def _check_rows(x, lens, o, S, tol):
    for r, n in enumerate(lens):
        if n > 0:
            sl = lambda t: t[r:r + 1, :n].contiguous()
            ro, rS = oracle.forward(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta), x.S0[r:r + 1])
            assert_close(o[r:r + 1, :n], ro, tol, f"o of row {r} (length {n})")
            assert_close(S[r:r + 1], rS, tol, f"S_T of row {r} (length {n})")
        else:
            assert torch.equal(S[r].cpu(), x.S0[r]), "a row of length 0 keeps its initial state"
        assert torch.all(o[r, n:].float() == 7.0), f"o past the length of row {r} was written"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_varlen_rows_match_their_truncated_rows(dtype):
    lens = [4096, 1000, 1, 0, 2049]
    x = inputs.regime("R1", 4096, 83, Hk=2, Hv=4, B=len(lens), init_state=True, dtype=dtype)
    # g and beta past each length are not pads in the inputs: the lengths alone make them pads
    o = torch.full_like(dev(x.v), 7.0)
    lengths = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, S = gdr.gdr_chunk_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(x.S0), o=o, lengths=lengths)
    gdr.gdr_sync_status()
    _check_rows(x, lens, o, S, TOL_BF16 if dtype == torch.bfloat16 else TOL_F32)


@pytest.mark.parametrize("L", [50, 130])
def test_varlen_short_rows(L):
    lens = [L, L // 2, 0, 1]
    x = inputs.regime("R3", L, 84 + L, Hk=2, Hv=4, B=len(lens), init_state=True, dtype=torch.bfloat16)
    o = torch.full_like(dev(x.v), 7.0)
    lengths = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, S = gdr.gdr_chunk_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(x.S0), o=o, lengths=lengths)
    gdr.gdr_sync_status()
    _check_rows(x, lens, o, S, TOL_BF16)


def test_varlen_full_lengths_equal_the_plain_call_bit_for_bit():
    x = inputs.regime("R1", 300, 85, Hk=2, Hv=4, B=2, init_state=True, dtype=torch.bfloat16)
    args = [dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    o, S = gdr.gdr_chunk_fwd(*args)
    o2, S2 = gdr.gdr_chunk_fwd(*args, lengths=torch.full((2,), 300, dtype=torch.int32, device="cuda"))
    gdr.gdr_sync_status()
    assert torch.equal(o, o2) and torch.equal(S, S2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_varlen_bad_length_reports_and_leaves_the_row_untouched(dtype):
    x = inputs.regime("R1", 130, 86, Hk=2, Hv=4, B=3, init_state=True, dtype=dtype)
    o = torch.full_like(dev(x.v), 7.0)
    S = torch.full((3, 4, 128, 128), 3.0, device="cuda")
    lengths = torch.tensor([130, 131, 64], dtype=torch.int32, device="cuda")
    gdr.gdr_chunk_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(x.S0), o=o, S_T=S, lengths=lengths)
    with pytest.raises(gdr.GdrError) as ei:
        gdr.gdr_sync_status()
    assert ei.value.status == gdr.GDR_ERR_DEVICE_INDEX
    assert torch.all(o[1].float() == 7.0) and torch.all(S[1] == 3.0)
    assert not torch.all(S[0] == 3.0) and not torch.all(S[2] == 3.0)
    gdr.gdr_sync_status()
