"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle on seeded inputs.

Tolerances: max|diff| <= 1e-4 max|ref| for float32 q/k/v, <= 5e-3 max|ref| for bf16 q/k/v, on the
outputs at every position and on the final states. Bookkeeping (pads, fork indices, idle decode
rows, state handoff, power-of-two scaling) is checked bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_rule_gb300 import gdr, inputs
from tests.gpu_util import TOL_BF16, TOL_F32, assert_close, dev

pytestmark = pytest.mark.gpu


def run_chunk(x, final_state=True, S0=True):
    o, S = gdr.gdr_chunk_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta),
                             dev(x.S0) if S0 else None, final_state=final_state)
    gdr.gdr_sync_status()
    return o, S


def ref_chunk(x, S0=True):
    return oracle.forward(x.q, x.k, x.v, x.g, x.beta, x.S0 if S0 else None)


def tol_of(x):
    return TOL_BF16 if x.q.dtype == torch.bfloat16 else TOL_F32


def test_config1_fp32_single_row():
    x = inputs.config1()
    o, S = run_chunk(x)
    ro, rS = ref_chunk(x)
    assert_close(o, ro, TOL_F32, "o")
    assert_close(S, rS, TOL_F32, "S_T")


@pytest.mark.parametrize("which", ["a", "b", "c"])
def test_config2_fp32_padded_regimes(which):
    x = inputs.config2(which)
    o, S = run_chunk(x)
    ro, rS = ref_chunk(x)
    assert_close(o, ro, TOL_F32, "o (all positions)")
    assert_close(o[:, :100], ro[:, :100], TOL_F32, "o (real positions)")
    assert_close(S, rS, TOL_F32, "S_T")


def test_config2_joint_scale_2_pow_8_bit_exact():
    x = inputs.config2("a")
    o, S = run_chunk(x)
    x.v, x.S0 = x.v * 256.0, x.S0 * 256.0
    o8, S8 = run_chunk(x)
    assert torch.equal(o8, o * 256.0) and torch.equal(S8, S * 256.0)


@pytest.mark.parametrize("L,B", [(50, 2), (130, 1), (300, 2)])
def test_bf16_joint_scale_2_pow_8_bit_exact(L, B):
    """The tensor-core path forms every fp16 operand that depends on v or the state from a tile
    divided by its own power of two (v per chunk, the initial state per head, the running state by
    the largest of those seen so far), so scaling (v, S0) by 2^8 leaves every operand bit-identical
    and scales o and S_T by exactly 2^8: on single-chunk rows (one kernel) and multi-chunk rows."""
    x = inputs.regime("R2", L, 22 + L, Hk=4, Hv=8, B=B, init_state=True, n_valid=L - 30, dtype=torch.bfloat16)
    o, S = run_chunk(x)
    x.v, x.S0 = x.v * 256.0, x.S0 * 256.0
    o8, S8 = run_chunk(x)
    assert torch.equal(o8, o * 256.0) and torch.equal(S8, S * 256.0)
    # negative control: v scaled alone is not a scaling of the result
    x.S0 = x.S0 / 256.0
    o9, _ = run_chunk(x)
    assert not torch.equal(o9, o * 256.0)


@pytest.mark.parametrize("L", [50, 300])
def test_bf16_large_inputs_stay_in_range(L):
    """q, k, v and S0 with entries in the thousands (well inside bf16's range, beyond what fp16
    operands hold unscaled): the tensor-core path scales its operands by powers of two, so o and
    S_T still match the oracle at the bf16 tolerance and nothing overflows to inf."""
    x = inputs.regime("R1", L, 91 + L, Hk=2, Hv=4, B=2, init_state=True, dtype=torch.bfloat16)
    x.q = (x.q.float() * 2000.0).bfloat16()
    x.k = (x.k.float() * 4000.0).bfloat16()
    x.v = (x.v.float() * 3000.0).bfloat16()
    x.S0 = x.S0 * 30000.0
    o, S = run_chunk(x)
    ro, rS = ref_chunk(x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()
    assert_close(o, ro, TOL_BF16, "o")
    assert_close(S, rS, TOL_BF16, "S_T")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 130, 200])
def test_lengths_and_ragged_tails(dtype, L):
    x = inputs.regime("R1", L, 100 + L, Hk=2, Hv=4, init_state=True, dtype=dtype)
    o, S = run_chunk(x)
    ro, rS = ref_chunk(x)
    assert_close(o, ro, tol_of(x), f"o L={L}")
    assert_close(S, rS, tol_of(x), f"S_T L={L}")


@pytest.mark.parametrize("name,seed", [("R1", 11), ("R2", 21), ("R3", 31), ("R4", 42)])
def test_regimes_bf16_multi_row(name, seed):
    x = inputs.regime(name, 256, seed, Hk=4, Hv=8, B=2, init_state=True, n_valid=200, dtype=torch.bfloat16)
    o, S = run_chunk(x)
    ro, rS = ref_chunk(x)
    assert_close(o, ro, TOL_BF16, "o")
    assert_close(S, rS, TOL_BF16, "S_T")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_no_initial_state_and_no_final_state(dtype):
    x = inputs.regime("R2", 100, 5, Hk=2, Hv=2, init_state=False, dtype=dtype)
    o, S = run_chunk(x, S0=False)
    ro, rS = ref_chunk(x, S0=False)
    assert_close(o, ro, tol_of(x), "o")
    assert_close(S, rS, tol_of(x), "S_T")
    o2, S2 = run_chunk(x, final_state=False, S0=False)
    assert S2 is None and torch.equal(o2, o)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_split_sequence_handoff_bit_exact(dtype):
    x = inputs.regime("R1", 256, 7, Hk=2, Hv=4, init_state=True, dtype=dtype)
    q, k, v, g, b = (dev(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    o, S = gdr.gdr_chunk_fwd(q, k, v, g, b, dev(x.S0))
    cut = 128
    o1, S1 = gdr.gdr_chunk_fwd(*(t[:, :cut].contiguous() for t in (q, k, v, g, b)), dev(x.S0))
    o2, S2 = gdr.gdr_chunk_fwd(*(t[:, cut:].contiguous() for t in (q, k, v, g, b)), S1)
    gdr.gdr_sync_status()
    assert torch.equal(torch.cat([o1, o2], 1), o) and torch.equal(S2, S)


def test_final_state_may_alias_initial_state():
    x = inputs.regime("R1", 70, 8, Hk=2, Hv=4, init_state=True, dtype=torch.bfloat16)
    o, S = run_chunk(x)
    S_io = dev(x.S0).clone()
    o2, S2 = gdr.gdr_chunk_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), S_io, S_T=S_io)
    gdr.gdr_sync_status()
    assert S2.data_ptr() == S_io.data_ptr()
    assert torch.equal(S2, S) and torch.equal(o2, o)


# ------------------------------------------------------------------------------------------------
# forks and decode
# ------------------------------------------------------------------------------------------------

def _fork_case(F=12, seed=9, N=3):
    c = inputs.config5(seed=seed, F=F, steps=3)
    gen = torch.Generator().manual_seed(seed)
    trunk = torch.randn(N, 32, 128, 128, generator=gen) * 0.1
    idx = torch.randint(0, N, (F,), generator=gen)
    return c, trunk, idx


def test_fork_batch_matches_oracle():
    c, trunk, idx = _fork_case()
    x = c.fork
    o, S = gdr.gdr_fork_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(trunk), dev(idx))
    gdr.gdr_sync_status()
    ro, rS = oracle.fork(x.q, x.k, x.v, x.g, x.beta, trunk, idx)
    assert_close(o, ro, TOL_BF16, "fork o")
    assert_close(S, rS, TOL_BF16, "fork states")


def test_fork_results_do_not_depend_on_batch_composition():
    c, trunk, idx = _fork_case(F=10, seed=13)
    x = c.fork
    args = [dev(t) for t in (x.q, x.k, x.v, x.g, x.beta)]
    o, S = gdr.gdr_fork_fwd(*args, dev(trunk), dev(idx))
    perm = torch.tensor([7, 2, 9, 0])
    sub = [t[perm.to(t.device)].contiguous() for t in args]
    o2, S2 = gdr.gdr_fork_fwd(*sub, dev(trunk), dev(idx[perm]))
    gdr.gdr_sync_status()
    assert torch.equal(o2, o[perm.cuda()]) and torch.equal(S2, S[perm.cuda()])
    # the trunk is read in place and never written
    t_dev = dev(trunk)
    before = t_dev.clone()
    gdr.gdr_fork_fwd(*args, t_dev, dev(idx))
    gdr.gdr_sync_status()
    assert torch.equal(t_dev, before)


def test_fork_index_out_of_range_reports_and_leaves_row_untouched():
    c, trunk, idx = _fork_case(F=4, seed=17, N=2)
    x = c.fork
    bad = idx.clone()
    bad[2] = 5
    o = torch.full_like(dev(x.v), 7.0)
    S = torch.full((4, 32, 128, 128), 3.0, device="cuda")
    gdr.gdr_fork_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(trunk), dev(bad), o=o,
                     states_out=S)
    with pytest.raises(gdr.GdrError) as ei:
        gdr.gdr_sync_status()
    assert ei.value.status == gdr.GDR_ERR_DEVICE_INDEX
    assert torch.all(o[2] == 7.0) and torch.all(S[2] == 3.0)
    assert not torch.all(o[1] == 7.0)
    gdr.gdr_sync_status()          # the error word was cleared


def test_decode_steps_match_oracle_and_idle_rows_are_unchanged():
    c, trunk, idx = _fork_case(F=16, seed=21, N=1)
    gen = torch.Generator().manual_seed(3)
    states = torch.randn(16, 32, 128, 128, generator=gen) * 0.1
    st_dev = dev(states).clone()
    ref = states.double().numpy()
    for step in c.decode:
        x = step
        x.beta[3] = 0.0      # row 3 idle: lens 0 => beta = g = 0
        x.g[3] = 0.0
        before_idle = st_dev[3].clone()
        o = gdr.gdr_decode_step(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), st_dev)
        gdr.gdr_sync_status()
        ro, ref = oracle.decode_step(x.q, x.k, x.v, x.g, x.beta, ref)
        assert_close(o, ro, TOL_BF16, "decode o")
        assert torch.equal(st_dev[3], before_idle)
    assert_close(st_dev, ref, TOL_BF16, "decode states")


def test_forced_wait_timeout_reports_and_the_next_call_recovers():
    """Failure detection without a fault: with a wait budget of 0 the kernels give up at their
    first unsatisfied wait, drain their own copies in flight and report GDR_ERR_TIMEOUT through the
    device error word; with the budget restored the same call is correct again."""
    x = inputs.regime("R1", 256, 61, Hk=2, Hv=4, init_state=True, dtype=torch.bfloat16)
    args = [dev(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    gdr.debug_set_wait_budget(0)
    try:
        gdr.gdr_chunk_fwd(*args)
        with pytest.raises(gdr.GdrError) as ei:
            gdr.gdr_sync_status()
        assert ei.value.status == gdr.GDR_ERR_TIMEOUT
    finally:
        gdr.debug_set_wait_budget(-1)
    o, S = gdr.gdr_chunk_fwd(*args)
    gdr.gdr_sync_status()
    ro, rS = ref_chunk(x)
    assert_close(o, ro, TOL_BF16, "o after recovery")
    assert_close(S, rS, TOL_BF16, "S_T after recovery")


# ------------------------------------------------------------------------------------------------
# the full-size workloads, in the launch configuration the benchmark times
# ------------------------------------------------------------------------------------------------

def test_config3_prefill_4096_full_size():
    x = inputs.config3()
    o, S = run_chunk(x)
    ro, rS = ref_chunk(x)
    assert_close(o, ro, TOL_BF16, "o")
    assert_close(S, rS, TOL_BF16, "S_T")


def test_config4_long_prefill_8192_full_size():
    x = inputs.config4()
    o, S = run_chunk(x, S0=False)
    ro, rS = ref_chunk(x, S0=False)
    assert_close(o, ro, TOL_BF16, "o")
    assert_close(S, rS, TOL_BF16, "S_T")


def test_config5_forks_and_decode_full_size_sampled():
    c = inputs.config5()
    x = c.fork
    o, S = gdr.gdr_fork_fwd(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.beta), dev(c.trunk), dev(c.trunk_idx))
    for step in c.decode:
        gdr.gdr_decode_step(dev(step.q), dev(step.k), dev(step.v), dev(step.g), dev(step.beta), S)
    gdr.gdr_sync_status()
    # oracle on a sample of 24 forks (each fork is independent of the others)
    pick = torch.arange(0, 256, 11)
    sub = lambda t: t[pick].contiguous()
    ro, rS = oracle.fork(sub(x.q), sub(x.k), sub(x.v), sub(x.g), sub(x.beta), c.trunk, c.trunk_idx[pick])
    assert_close(o[pick.cuda()], ro, TOL_BF16, "fork o")
    for step in c.decode:
        _, rS = oracle.decode_step(sub(step.q), sub(step.k), sub(step.v), sub(step.g), sub(step.beta), rS)
    assert_close(S[pick.cuda()], rS, TOL_BF16, "states after 32 decode steps")


def test_variable_length_rows_match_their_truncated_rows():
    """Rows of different real lengths in one call (right-padded with beta = g = 0): each row's final
    state equals the oracle's state after that row's last real token alone, and its outputs at
    real positions match the oracle on the truncated row."""
    lens = [256, 130, 64, 1]
    x = inputs.regime("R1", 256, 81, Hk=2, Hv=4, B=len(lens), init_state=True, dtype=torch.bfloat16)
    for r, n in enumerate(lens):
        x.beta[r, n:] = 0.0
        x.g[r, n:] = 0.0
    o, S = run_chunk(x)
    for r, n in enumerate(lens):
        sl = lambda t: t[r:r + 1, :n].contiguous()
        ro, rS = oracle.forward(sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta), x.S0[r:r + 1])
        assert_close(o[r:r + 1, :n], ro, TOL_BF16, f"o of row {r} (length {n})")
        assert_close(S[r:r + 1], rS, TOL_BF16, f"S_T of row {r} (length {n})")
