"""GPU parity of the fork and decode rows beyond the single-chunk bf16 forks of the fork workload:
forks of two and three chunks (the prep and state kernels, with the initial state gathered from
the trunk by index), float32 forks (the token loop with the same gather) and float32 decode steps.

Tolerances as elsewhere: max|diff| <= 5e-3 max|ref| for bf16 q/k/v, <= 1e-4 max|ref| for float32;
the bookkeeping (trunk gather, batch independence, idle rows) is checked bit for bit.
"""
import pytest
import torch

import oracle
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, TOL_F32, assert_close, dev

pytestmark = pytest.mark.gpu


def _forks(L_pad, seed, F=9, N=3, Hk=4, Hv=8, dtype=torch.bfloat16):
    """F forks whose real lengths fill the last of L_pad / 64 chunks (so every chunk is used), N
    trunk states, random trunk indices."""
    c = inputs.config5(seed=seed, F=F, steps=2, Hk=Hk, Hv=Hv, len_lo=L_pad - 60, len_hi=L_pad)
    assert c.fork.q.shape[1] == L_pad
    gen = torch.Generator().manual_seed(seed + 1)
    trunk = torch.randn(N, Hv, 128, 128, generator=gen) * 0.1
    idx = torch.randint(0, N, (F,), generator=gen)
    x = c.fork
    if dtype == torch.float32:
        x.q, x.k, x.v = x.q.float(), x.k.float(), x.v.float()
    return x, trunk, idx


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("L_pad", [128, 192])
def test_multichunk_forks_match_oracle(L_pad, dtype):
    x, trunk, idx = _forks(L_pad, seed=40 + L_pad, dtype=dtype)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    args = [dev(t) for t in (x.q, x.k, x.v, x.g, x.beta)]
    o, S = gdr.gdr_fork_fwd(*args, dev(trunk), dev(idx))
    gdr.gdr_sync_status()
    ro, rS = oracle.fork(x.q, x.k, x.v, x.g, x.beta, trunk, idx)
    assert_close(o, ro, tol, f"fork o (L_pad={L_pad})")
    assert_close(S, rS, tol, f"fork states (L_pad={L_pad})")
    # bookkeeping: fork f is the prefill of its own row from trunk[idx[f]], bit for bit
    for f in (0, 4, 8):
        row = [t[f:f + 1].contiguous() for t in args]
        o1, S1 = gdr.gdr_chunk_fwd(*row, dev(trunk[idx[f]:idx[f] + 1]))
        gdr.gdr_sync_status()
        assert torch.equal(o1, o[f:f + 1]) and torch.equal(S1, S[f:f + 1]), f


def test_multichunk_forks_do_not_depend_on_batch_composition():
    x, trunk, idx = _forks(192, seed=77)
    args = [dev(t) for t in (x.q, x.k, x.v, x.g, x.beta)]
    o, S = gdr.gdr_fork_fwd(*args, dev(trunk), dev(idx))
    perm = torch.tensor([5, 1, 8])
    sub = [t[perm.to(t.device)].contiguous() for t in args]
    o2, S2 = gdr.gdr_fork_fwd(*sub, dev(trunk), dev(idx[perm]))
    gdr.gdr_sync_status()
    assert torch.equal(o2, o[perm.cuda()]) and torch.equal(S2, S[perm.cuda()])


def test_float32_decode_steps_match_oracle_and_idle_rows_are_unchanged():
    c = inputs.config5(seed=23, F=12, steps=4, Hk=4, Hv=8)
    gen = torch.Generator().manual_seed(29)
    states = torch.randn(12, 8, 128, 128, generator=gen) * 0.1
    st_dev = dev(states).clone()
    ref = states.double().numpy()
    for step in c.decode:
        step.q, step.k, step.v = step.q.float(), step.k.float(), step.v.float()
        step.beta[5] = 0.0
        step.g[5] = 0.0
        idle_before = st_dev[5].clone()
        o = gdr.gdr_decode_step(dev(step.q), dev(step.k), dev(step.v), dev(step.g), dev(step.beta), st_dev)
        gdr.gdr_sync_status()
        assert o.dtype == torch.float32
        ro, ref = oracle.decode_step(step.q, step.k, step.v, step.g, step.beta, ref)
        assert_close(o, ro, TOL_F32, "float32 decode o")
        assert torch.equal(st_dev[5], idle_before)
    assert_close(st_dev, ref, TOL_F32, "float32 decode states")
