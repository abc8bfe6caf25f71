"""gdr_chunk_fwd_noalloc: the prefill call for callers that cannot allocate GPU memory.

Hosts that own the whole device memory budget (a serving process that reserves the GPU at start-up,
or a plugin inside one) and latency-critical loops cannot hand gdr_chunk_fwd a freshly allocated
workspace; this entry point runs the same kernels on a fixed scratch array the library keeps in
device memory. The test calls it through the C ABI several times in a row, on different sizes so
that each call starts from the previous call's leftovers in the scratch (a larger call, then
smaller ones, then a single-chunk row, which needs no scratch at all), and compares each result
with gdr_chunk_fwd given its own workspace. Both calls run the same kernels in the same order, so
the results must be identical bit for bit (a leftover read from the scratch would show here even
if it moved a result by less than the bf16 tolerance). It also checks that a size beyond the
scratch is refused with a clear message and no GPU work.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from gated_deltanet_rule_gb300 import gdr, inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 * 1024 * 1024


def _dev(x):
    return None if x is None else x.cuda().contiguous()


def _noalloc(q, k, v, g, beta, S0, o, S_T):
    B, L, Hk, D = q.shape
    Hv = v.shape[2]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return gdr.lib().gdr_chunk_fwd_noalloc(p(q), p(k), p(v), p(g), p(beta), p(S0), p(o), p(S_T),
                                           B, L, Hk, Hv, D, gdr.GDR_BF16, stream)


def test_noalloc_matches_workspace_call_on_calls_in_a_row():
    cases = [inputs.regime("R1", 1000, 5, Hk=8, Hv=16, B=1, init_state=True, dtype=torch.bfloat16),
             inputs.regime("R3", 700, 6, Hk=4, Hv=8, B=3, init_state=True, n_valid=650, dtype=torch.bfloat16),
             inputs.regime("R2", 300, 7, Hk=2, Hv=4, B=2, init_state=True, dtype=torch.bfloat16),
             inputs.regime("R1", 50, 8, Hk=4, Hv=8, B=2, init_state=True, dtype=torch.bfloat16)]
    for x in cases:
        q, k, v, g, b, S0 = (_dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.S0))
        B, L, Hk, D = q.shape
        assert gdr.workspace_bytes(B, L, Hk, v.shape[2]) <= SCRATCH_BYTES
        ref_o, ref_S = gdr.gdr_chunk_fwd(q, k, v, g, b, S0)
        o = torch.full_like(v, float("nan"))
        S_T = torch.full_like(S0, float("nan"))
        st = _noalloc(q, k, v, g, b, S0, o, S_T)
        assert st == gdr.GDR_OK, gdr.lib().gdr_last_error_message().decode()
        gdr.gdr_sync_status()
        assert torch.equal(o, ref_o), f"o differs from gdr_chunk_fwd (L={L}, Hv={v.shape[2]})"
        assert torch.equal(S_T, ref_S), f"S_T differs from gdr_chunk_fwd (L={L}, Hv={v.shape[2]})"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    B, L, Hk, Hv = 1, 4096, 16, 32                      # 2048 chunk units: 202 MB of scratch
    assert gdr.workspace_bytes(B, L, Hk, Hv) > SCRATCH_BYTES
    q = torch.zeros(B, L, Hk, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(B, L, Hv, 128, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(B, L, Hv, device="cuda")
    o = torch.full_like(v, 3.0)
    st = _noalloc(q, q, v, g, g, None, o, None)
    assert st == gdr.GDR_ERR_UNSUPPORTED
    msg = gdr.lib().gdr_last_error_message().decode()
    assert "scratch" in msg and str(SCRATCH_BYTES) in msg
    torch.cuda.synchronize()
    assert torch.all(o == 3.0)
