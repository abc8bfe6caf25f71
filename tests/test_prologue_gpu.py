"""GPU parity of the GDN prologue (gdr_prologue through the C ABI) against the float64 oracle.

Tolerances, element by element: q, k, v (one rounding to bf16 of an fp32 result) within
2^-8 |ref| + 1e-6; g and beta (fp32 exp / log1p) within 2e-6 |ref| + 1e-7; the carry (a copy)
and the zero gates at pads bit for bit. The composition prologue -> gdr_chunk_fwd is compared with
the oracle prologue -> oracle recurrence at the path's bf16 tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.prologue as op
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, assert_close, dev

pytestmark = pytest.mark.gpu


def run(x, keep_tail=True):
    out = gdr.gdr_prologue(dev(x.mixed), dev(x.conv_w), dev(x.a), dev(x.b), dev(x.A_log), dev(x.dt_bias), x.Hk, x.Hv,
                           tail=dev(x.tail), lengths=dev(x.lengths), keep_tail=keep_tail)
    gdr.gdr_sync_status()
    return out


def ref(x):
    return op.prologue(x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, x.Hk, x.Hv, tail=x.tail, lengths=x.lengths)


def check(got, want, rtol, atol, what):
    g = got.detach().double().cpu().numpy()
    assert g.shape == want.shape, (what, g.shape, want.shape)
    bad = np.abs(g - want) > rtol * np.abs(want) + atol
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, worst {np.abs(g - want).max():.3e}"


def check_all(got, want, K):
    for i, name in enumerate(("q", "k", "v")):
        check(got[i], want[i], 2.0 ** -8, 1e-6, name)
    check(got[3], want[3], 2e-6, 1e-7, "g")
    check(got[4], want[4], 2e-6, 1e-7, "beta")
    if K > 1:
        assert np.array_equal(got[5].double().cpu().numpy(), want[5]), "carry"


@pytest.mark.parametrize("K", [4, 1, 2, 3, 8])
def test_prologue_matches_oracle_with_lengths_and_carry(K):
    x = inputs.prologue_inputs(2, 130, 31 + K, Hk=2, Hv=4, K=K, lengths=[100, 130])
    got = run(x)
    want = ref(x)
    check_all(got, want, K)
    g = got[3].cpu()
    assert torch.all(g[0, 100:] == 0) and torch.all(got[4].cpu()[0, 100:] == 0), "pads must be exact no-ops"


def test_prologue_rows_of_length_zero_and_full():
    """A row of length 0 is all pads: its gates are zero and its carry is the old carry."""
    x = inputs.prologue_inputs(3, 66, 45, Hk=2, Hv=2, K=4, lengths=[0, 66, 2])
    got = run(x)
    check_all(got, ref(x), 4)
    assert torch.all(got[3][0] == 0) and torch.all(got[4][0] == 0)
    assert torch.equal(got[5][0].cpu(), x.tail[0])


def test_prologue_without_carry_or_lengths():
    x = inputs.prologue_inputs(1, 77, 41, Hk=2, Hv=2, K=4, with_tail=False)
    check_all(run(x), ref(x), 4)


def test_prologue_split_calls_equal_one_call_bit_for_bit():
    x = inputs.prologue_inputs(2, 96, 43, Hk=2, Hv=4, K=4)
    full = run(x)
    L1 = 37
    x1 = inputs.PrologueInputs(x.mixed[:, :L1].contiguous(), x.conv_w, x.a[:, :L1].contiguous(), x.b[:, :L1].contiguous(),
                               x.A_log, x.dt_bias, x.tail, None, x.Hk, x.Hv)
    first = run(x1)
    x2 = inputs.PrologueInputs(x.mixed[:, L1:].contiguous(), x.conv_w, x.a[:, L1:].contiguous(), x.b[:, L1:].contiguous(),
                               x.A_log, x.dt_bias, first[5].cpu(), None, x.Hk, x.Hv)
    second = run(x2)
    for i in range(5):
        assert torch.equal(torch.cat([first[i], second[i]], 1), full[i]), i
    assert torch.equal(second[5], full[5])


def test_prologue_length_out_of_range_reports_and_leaves_the_row():
    x = inputs.prologue_inputs(2, 64, 47, Hk=2, Hv=2, K=4, lengths=[65, 10])
    g = torch.full((2, 64, 2), 7.0, device="cuda")
    beta = torch.full((2, 64, 2), 7.0, device="cuda")
    gdr.gdr_prologue(dev(x.mixed), dev(x.conv_w), dev(x.a), dev(x.b), dev(x.A_log), dev(x.dt_bias), x.Hk, x.Hv,
                     tail=dev(x.tail), lengths=dev(x.lengths), g=g, beta=beta)
    with pytest.raises(gdr.GdrError) as ei:
        gdr.gdr_sync_status()
    assert ei.value.status == gdr.GDR_ERR_DEVICE_INDEX
    assert torch.all(g[0] == 7.0) and torch.all(beta[0] == 7.0)
    want = op.prologue(x.mixed[1:], x.conv_w, x.a[1:], x.b[1:], x.A_log, x.dt_bias, 2, 2, tail=x.tail[1:], lengths=[10])
    check(g[1:], want[3], 2e-6, 1e-7, "g of the valid row")


def test_prologue_full_size_4096():
    x = inputs.prologue_inputs(1, 4096, 3, Hk=16, Hv=32, K=4)
    check_all(run(x), ref(x), 4)


def test_prologue_then_chunked_path_matches_oracle_composition():
    """gdr_prologue -> gdr_chunk_fwd against oracle prologue -> (q, k, v rounded to bf16, as the
    prologue writes them) -> oracle recurrence, with pads from the lengths."""
    x = inputs.prologue_inputs(2, 200, 53, Hk=2, Hv=4, K=4, lengths=[200, 150])
    q, k, v, g, beta, _ = run(x)
    o, S = gdr.gdr_chunk_fwd(q, k, v, g, beta, None)
    gdr.gdr_sync_status()
    rq, rk, rv, rg, rb, _ = ref(x)
    bf = lambda t: torch.from_numpy(t).float().bfloat16()
    ro, rS = oracle.forward(bf(rq), bf(rk), bf(rv), torch.from_numpy(rg).float(), torch.from_numpy(rb).float(), None)
    assert_close(o, ro, TOL_BF16, "o")
    assert_close(S, rS, TOL_BF16, "S_T")
