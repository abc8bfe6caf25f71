"""GPU parity of the gated RMSNorm epilogue (gdr_gated_rmsnorm through the C ABI) against the
float64 oracle: element by element within 2^-8 |ref| + 1e-6 (one rounding to bf16 of an fp32
result); in place equals out of place bit for bit; the composition gdr_chunk_fwd -> epilogue, and the
fused gdr_chunk_fwd_gated, match the oracle recurrence -> oracle epilogue at the path's bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import oracle.epilogue as oe
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, assert_close

pytestmark = pytest.mark.gpu


def _xzw(shape, seed):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=gen).bfloat16()
    z = (2 * torch.randn(*shape, generator=gen)).bfloat16()
    w = 0.5 + torch.rand(shape[-1], generator=gen)
    return x, z, w


def _check(got, want):
    g = got.double().cpu().numpy()
    bad = np.abs(g - want) > 2.0 ** -8 * np.abs(want) + 1e-6
    assert not bad.any(), f"{int(bad.sum())} elements off, worst {np.abs(g - want).max():.3e}"


@pytest.mark.parametrize("shape", [(2, 130, 4, 128), (1, 1, 1, 128), (3, 7, 2, 128)])
def test_gated_rmsnorm_matches_oracle(shape):
    x, z, w = _xzw(shape, sum(shape))
    out = gdr.gdr_gated_rmsnorm(x.cuda(), z.cuda(), w.cuda(), 1e-6)
    gdr.gdr_sync_status()
    _check(out, oe.gated_rms(x, z, w, 1e-6))


def test_gated_rmsnorm_in_place_equals_out_of_place():
    x, z, w = _xzw((2, 64, 4, 128), 5)
    xd, zd, wd = x.cuda(), z.cuda(), w.cuda()
    ref = gdr.gdr_gated_rmsnorm(xd, zd, wd, 1e-6)
    y = xd.clone()
    gdr.gdr_gated_rmsnorm(y, zd, wd, 1e-6, out=y)
    gdr.gdr_sync_status()
    assert torch.equal(y, ref)


def test_gated_rmsnorm_full_size_4096():
    x, z, w = _xzw((1, 4096, 32, 128), 7)
    out = gdr.gdr_gated_rmsnorm(x.cuda(), z.cuda(), w.cuda(), 1e-6)
    gdr.gdr_sync_status()
    _check(out, oe.gated_rms(x, z, w, 1e-6))


def test_chunked_path_then_epilogue_matches_oracle_composition():
    x = inputs.regime("R1", 200, 71, Hk=2, Hv=4, init_state=True, dtype=torch.bfloat16)
    _, z, w = _xzw(tuple(x.v.shape), 72)
    o, _ = gdr.gdr_chunk_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.beta.cuda(), x.S0.cuda())
    out = gdr.gdr_gated_rmsnorm(o, z.cuda(), w.cuda(), 1e-6)
    gdr.gdr_sync_status()
    ro, _ = oracle.forward(x.q, x.k, x.v, x.g, x.beta, x.S0)
    assert_close(out, oe.gated_rms(ro, z, w, 1e-6), TOL_BF16, "normalised output")


@pytest.mark.parametrize("L,B", [(200, 1), (300, 2), (50, 2)])
def test_fused_gated_prefill_matches_oracle_composition(L, B):
    """gdr_chunk_fwd_gated: the gated RMSNorm fused into the recurrence's output (rows of several
    chunks: the four column CTAs of a head reduce the sum of squares in a cluster; rows of one chunk:
    the epilogue over o in place) matches oracle recurrence -> oracle epilogue, and its final state
    equals gdr_chunk_fwd's bit for bit."""
    x = inputs.regime("R1", L, 73 + L, Hk=2, Hv=4, B=B, init_state=True, dtype=torch.bfloat16)
    _, z, w = _xzw(tuple(x.v.shape), 74 + L)
    args = [t.cuda() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    out, S = gdr.gdr_chunk_fwd_gated(*args, z.cuda(), w.cuda(), 1e-6)
    _, S_plain = gdr.gdr_chunk_fwd(*args)
    gdr.gdr_sync_status()
    ro, rS = oracle.forward(x.q, x.k, x.v, x.g, x.beta, x.S0)
    assert_close(out, oe.gated_rms(ro, z, w, 1e-6), TOL_BF16, "fused normalised output")
    assert torch.equal(S, S_plain)


def test_fused_gated_prefill_full_size_4096():
    x = inputs.config3()
    _, z, w = _xzw(tuple(x.v.shape), 75)
    args = [t.cuda() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    out, _ = gdr.gdr_chunk_fwd_gated(*args, z.cuda(), w.cuda(), 1e-6)
    gdr.gdr_sync_status()
    ro, _ = oracle.forward(x.q, x.k, x.v, x.g, x.beta, x.S0)
    assert_close(out, oe.gated_rms(ro, z, w, 1e-6), TOL_BF16, "fused normalised output (L = 4096)")
