"""GPU parity of the GDN prologue fused into the bf16 prefill (gdr_chunk_fwd_prologue through the C
ABI).

The fused call forms q, k, v, g and beta inside the chunk kernel with gdr_prologue's own order of
operations, so for rows longer than one chunk its o, S_T and carry equal those of gdr_prologue
followed by gdr_chunk_fwd bit for bit. Rows of one chunk (L <= 64) take the two-kernel path
through the workspace (gdr_chunk_fwd finishes them in one kernel with another summation order):
there, and everywhere as an independent check, the result is held to the oracle composition
(oracle prologue -> q, k, v rounded to bf16 as the prologue writes them -> oracle recurrence) at the
path's bf16 bound, max|diff| <= 5e-3 max|ref|. The carry is a copy: bit for bit in every case.
"""
import pytest
import torch

import oracle
import oracle.prologue as op
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, assert_close, dev

pytestmark = pytest.mark.gpu


def initial_state(B, Hv, seed):
    gen = torch.Generator().manual_seed(seed)
    return 0.1 * torch.randn(B, Hv, 128, 128, generator=gen)


def fused(x, S0):
    out = gdr.gdr_chunk_fwd_prologue(dev(x.mixed), dev(x.conv_w), dev(x.a), dev(x.b), dev(x.A_log), dev(x.dt_bias),
                                     x.Hk, x.Hv, S0=dev(S0), tail=dev(x.tail))
    gdr.gdr_sync_status()
    return out


def separate(x, S0):
    q, k, v, g, beta, new_tail = gdr.gdr_prologue(dev(x.mixed), dev(x.conv_w), dev(x.a), dev(x.b), dev(x.A_log),
                                                  dev(x.dt_bias), x.Hk, x.Hv, tail=dev(x.tail))
    o, S = gdr.gdr_chunk_fwd(q, k, v, g, beta, dev(S0))
    gdr.gdr_sync_status()
    return o, S, new_tail


def oracle_composition(x, S0):
    rq, rk, rv, rg, rb, rt = op.prologue(x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, x.Hk, x.Hv, tail=x.tail)
    bf = lambda t: torch.from_numpy(t).float().bfloat16()
    ro, rS = oracle.forward(bf(rq), bf(rk), bf(rv), torch.from_numpy(rg).float(), torch.from_numpy(rb).float(), S0)
    return ro, rS, rt


@pytest.mark.parametrize("B,L,with_tail,with_S0", [(2, 130, True, True), (2, 200, True, False), (1, 65, False, True),
                                                   (3, 128, True, True)])
def test_fused_prologue_equals_the_separate_calls_bit_for_bit(B, L, with_tail, with_S0):
    x = inputs.prologue_inputs(B, L, 61 + L, Hk=2, Hv=4, K=4, with_tail=with_tail)
    S0 = initial_state(B, 4, 62 + L) if with_S0 else None
    got = fused(x, S0)
    want = separate(x, S0)
    for name, a, b in zip(("o", "S_T", "new_tail"), got, want):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("Hk,Hv", [(2, 2), (1, 4), (3, 6)])
def test_fused_prologue_head_ratios_equal_the_separate_calls(Hk, Hv):
    """One, four and two value heads per key head: the channel split of the projection (q at key
    head h / r, k after all of q, v after all of k) and the gates' head index, bit for bit."""
    x = inputs.prologue_inputs(2, 150, 101 + Hv, Hk=Hk, Hv=Hv, K=4)
    S0 = initial_state(2, Hv, 102 + Hv)
    got = fused(x, S0)
    want = separate(x, S0)
    for name, a, b in zip(("o", "S_T", "new_tail"), got, want):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("B,L,with_tail", [(2, 200, True), (1, 1, True), (2, 2, True), (1, 3, False), (2, 64, True),
                                           (1, 100, False)])
def test_fused_prologue_matches_the_oracle_composition(B, L, with_tail):
    """Ragged and single-chunk rows, rows shorter than the carry (L < 3: part of the new carry comes
    from the old one), with and without a carry."""
    x = inputs.prologue_inputs(B, L, 71 + L, Hk=2, Hv=4, K=4, with_tail=with_tail)
    S0 = initial_state(B, 4, 72 + L)
    o, S, new_tail = fused(x, S0)
    ro, rS, rt = oracle_composition(x, S0)
    assert_close(o, ro, TOL_BF16, "o")
    assert_close(S, rS, TOL_BF16, "S_T")
    assert torch.equal(new_tail.cpu(), torch.from_numpy(rt).bfloat16()), "carry"


def test_split_fused_calls_continue_through_the_carry():
    """Two fused calls, the second taking the first's carry and final state, against one call over
    the whole row (the same arithmetic, so o agrees within the bf16 bound and S_T too)."""
    x = inputs.prologue_inputs(2, 256, 81, Hk=2, Hv=4, K=4)
    S0 = initial_state(2, 4, 82)
    o_full, S_full, t_full = fused(x, S0)
    L1 = 128
    part = lambda sl, tail: inputs.PrologueInputs(x.mixed[:, sl].contiguous(), x.conv_w, x.a[:, sl].contiguous(),
                                                  x.b[:, sl].contiguous(), x.A_log, x.dt_bias, tail, None, x.Hk, x.Hv)
    o1, S1, t1 = fused(part(slice(0, L1), x.tail), S0)
    o2, S2, t2 = fused(part(slice(L1, None), t1.cpu()), S1.cpu())
    assert torch.equal(torch.cat([o1, o2], 1)[:, :L1], o_full[:, :L1]), "the first half is the same computation"
    ro, rS, _ = oracle_composition(x, S0)
    assert_close(torch.cat([o1, o2], 1), ro, TOL_BF16, "o")
    assert_close(S2, rS, TOL_BF16, "S_T")
    assert torch.equal(t2, t_full)


def test_fused_prologue_full_size_4096():
    """L = 4096, Hk = 16, Hv = 32 with a carry and S0: bit for bit against the separate calls, and key
    head 5 with its two value heads against the oracle composition on that slice (their channels of
    mixed, conv_w and their gates depend on no other head)."""
    x = inputs.prologue_inputs(1, 4096, 91, Hk=16, Hv=32, K=4)
    S0 = initial_state(1, 32, 92)
    got = fused(x, S0)
    want = separate(x, S0)
    for name, a, b in zip(("o", "S_T", "new_tail"), got, want):
        assert torch.equal(a, b), name
    hk, HkD = 5, 16 * 128
    chans = torch.cat([torch.arange(hk * 128, hk * 128 + 128), torch.arange(HkD + hk * 128, HkD + hk * 128 + 128),
                       torch.arange(2 * HkD + 2 * hk * 128, 2 * HkD + 2 * hk * 128 + 256)])
    hv = slice(2 * hk, 2 * hk + 2)
    xs = inputs.PrologueInputs(x.mixed[:, :, chans].contiguous(), x.conv_w[chans].contiguous(), x.a[:, :, hv].contiguous(),
                               x.b[:, :, hv].contiguous(), x.A_log[hv].contiguous(), x.dt_bias[hv].contiguous(),
                               x.tail[:, :, chans].contiguous(), None, 1, 2)
    ro, rS, _ = oracle_composition(xs, S0[:, hv].contiguous())
    assert_close(got[0][:, :, hv], ro, TOL_BF16, "o")
    assert_close(got[1][:, hv], rS, TOL_BF16, "S_T")
