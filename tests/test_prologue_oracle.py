"""Pins of the GDN prologue oracle (oracle/prologue.py) against facts that do not come from it:
closed forms of the gates, single-tap convolutions, a brute-force convolution written as a
sum over input positions, and the carry handoff between two calls."""
import math

import numpy as np
import pytest
import torch

from gated_deltanet_rule_gb300 import inputs
import oracle.prologue as op

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _small(B=2, L=9, Hk=1, Hv=2, K=4, D=4, seed=7, tail=True):
    gen = torch.Generator().manual_seed(seed)
    C = (2 * Hk + Hv) * D
    mixed = torch.randn(B, L, C, generator=gen).double().numpy()
    t = torch.randn(B, K - 1, C, generator=gen).double().numpy() if tail else None
    w = torch.randn(C, K, generator=gen).double().numpy()
    a = torch.randn(B, L, Hv, generator=gen).double().numpy()
    b = torch.randn(B, L, Hv, generator=gen).double().numpy()
    A_log = torch.randn(Hv, generator=gen).double().numpy()
    dt_bias = torch.randn(Hv, generator=gen).double().numpy()
    return mixed, t, w, a, b, A_log, dt_bias


def _silu_scalar(x):
    return x / (1.0 + math.exp(-x))


def test_last_tap_alone_gives_silu_of_the_input():
    mixed, tail, w, a, b, A_log, dt_bias = _small()
    w[:] = 0.0
    w[:, -1] = 1.0
    q, k, v, *_ = op.prologue(mixed, w, a, b, A_log, dt_bias, 1, 2, D=4, tail=tail)
    y = np.concatenate([q.reshape(2, 9, -1), k.reshape(2, 9, -1), v.reshape(2, 9, -1)], axis=-1)
    ref = np.vectorize(_silu_scalar)(mixed)
    assert np.allclose(y, ref, rtol=1e-15, atol=0)


def test_first_tap_alone_reads_the_carry_then_the_input():
    K = 4
    mixed, tail, w, a, b, A_log, dt_bias = _small(K=K)
    w[:] = 0.0
    w[:, 0] = 1.0
    q, k, v, *_ = op.prologue(mixed, w, a, b, A_log, dt_bias, 1, 2, D=4, tail=tail)
    y = np.concatenate([q.reshape(2, 9, -1), k.reshape(2, 9, -1), v.reshape(2, 9, -1)], axis=-1)
    for t in range(9):
        src = tail[:, t] if t < K - 1 else mixed[:, t - (K - 1)]
        assert np.allclose(y[:, t], np.vectorize(_silu_scalar)(src), rtol=1e-15, atol=0)


@pytest.mark.parametrize("K", [1, 2, 4])
def test_convolution_by_brute_force_over_input_positions(K):
    """y[t][c] = silu(sum over input positions s <= t, s > t - K, of x[s][c] w[c][K-1-(t-s)]), with
    x indexed from -(K-1) (the carry) to L-1 (the new inputs)."""
    B, L, Hk, Hv, D = 1, 6, 1, 2, 2
    mixed, tail, w, a, b, A_log, dt_bias = _small(B=B, L=L, K=K, D=D, seed=11)
    C = mixed.shape[-1]

    def x_at(s, c):
        return tail[0, s + K - 1, c] if s < 0 else mixed[0, s, c]

    ref = np.zeros((L, C))
    for t in range(L):
        for c in range(C):
            acc = 0.0
            for s in range(t - K + 1, t + 1):
                acc += x_at(s, c) * w[c, K - 1 - (t - s)]
            ref[t, c] = _silu_scalar(acc)
    q, k, v, *_ = op.prologue(mixed, w, a, b, A_log, dt_bias, Hk, Hv, D=D, tail=tail)
    y = np.concatenate([q.reshape(B, L, -1), k.reshape(B, L, -1), v.reshape(B, L, -1)], axis=-1)[0]
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-15)


def test_channel_split_into_heads():
    """Channels [0, Hk D) are q, [Hk D, 2 Hk D) are k and the rest v, head-major within each."""
    B, L, Hk, Hv, D = 1, 3, 2, 4, 2
    mixed, tail, w, a, b, A_log, dt_bias = _small(B=B, L=L, Hk=Hk, Hv=Hv, D=D, K=1, tail=False)
    w[:] = 1.0
    q, k, v, *_ = op.prologue(mixed, w, a, b, A_log, dt_bias, Hk, Hv, D=D)
    s = np.vectorize(_silu_scalar)
    assert np.allclose(q[0, 1, 1, 0], s(mixed[0, 1, 1 * D + 0]))
    assert np.allclose(k[0, 2, 0, 1], s(mixed[0, 2, Hk * D + 1]))
    assert np.allclose(v[0, 0, 3, 1], s(mixed[0, 0, 2 * Hk * D + 3 * D + 1]))


def test_gates_closed_forms_and_pads():
    B, L, Hv = 1, 4, 3
    a = np.array([[[0.0, 0.0, 0.0], [1.5, -2.0, 30.0], [0.0, 0.0, 0.0], [5.0, 5.0, 5.0]]])
    b = np.array([[[0.0, 0.0, 0.0], [2.0, -1.0, 0.5], [0.0, 0.0, 0.0], [1.0, 1.0, 1.0]]])
    A_log = np.array([0.0, math.log(2.0), math.log(16.0)])
    dt_bias = np.zeros(Hv)
    valid = np.array([[1.0, 1.0, 1.0, 0.0]])
    beta, g = op.dn_gates(a, b, A_log, dt_bias, valid)
    assert np.allclose(beta[0, 0], 0.5, rtol=0, atol=1e-16)                       # sigmoid(0)
    assert np.allclose(g[0, 0], -np.exp(A_log) * math.log(2.0), rtol=1e-15)        # softplus(0)
    assert np.isclose(beta[0, 1, 0], 1 / (1 + math.exp(-2.0)), rtol=1e-15)
    assert np.isclose(g[0, 1, 1], -2.0 * math.log1p(math.exp(-2.0)), rtol=1e-15)
    assert np.isclose(g[0, 1, 2], -16.0 * (30.0 + math.log1p(math.exp(-30.0))), rtol=1e-15)  # softplus(x) ~ x
    assert np.all(beta[0, 3] == 0.0) and np.all(g[0, 3] == 0.0)                     # pads: exact no-ops
    assert np.all(g[0, :3] < 0) and np.all((beta[0, :3] > 0) & (beta[0, :3] < 1))


def test_gates_do_not_depend_on_the_convolution_inputs():
    x = inputs.prologue_inputs(1, 8, 3, Hk=1, Hv=2, K=4, lengths=[5])
    r1 = op.prologue(x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, 1, 2, tail=x.tail, lengths=x.lengths)
    r2 = op.prologue(x.mixed * 3, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, 1, 2, tail=None, lengths=x.lengths)
    assert np.array_equal(r1[3], r2[3]) and np.array_equal(r1[4], r2[4])
    assert np.all(r1[3][0, 5:] == 0) and np.all(r1[4][0, 5:] == 0)


@pytest.mark.parametrize("K", [2, 4])
def test_carry_handoff_equals_one_call(K):
    """Running [0, L1) and then [L1, L) with the first call's new_tail as the second call's tail gives
    the same q, k, v as one call over [0, L), bit for bit."""
    x = inputs.prologue_inputs(2, 12, 5, Hk=1, Hv=2, K=K)
    L1 = 5
    full = op.prologue(x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, 1, 2, tail=x.tail)
    first = op.prologue(x.mixed[:, :L1], x.conv_w, x.a[:, :L1], x.b[:, :L1], x.A_log, x.dt_bias, 1, 2, tail=x.tail)
    second = op.prologue(x.mixed[:, L1:], x.conv_w, x.a[:, L1:], x.b[:, L1:], x.A_log, x.dt_bias, 1, 2,
                         tail=first[5])
    for i in range(3):
        assert np.array_equal(np.concatenate([first[i], second[i]], axis=1), full[i])
    assert np.array_equal(second[5], full[5])


def test_carry_of_a_short_row_keeps_the_old_carry():
    K = 4
    x = inputs.prologue_inputs(1, 6, 9, Hk=1, Hv=2, K=K, lengths=[1])
    *_, new_tail = op.prologue(x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, 1, 2, tail=x.tail, lengths=x.lengths)
    t = x.tail.double().numpy()
    m = x.mixed.double().numpy()
    assert np.array_equal(new_tail[0, 0], t[0, 1]) and np.array_equal(new_tail[0, 1], t[0, 2])
    assert np.array_equal(new_tail[0, 2], m[0, 0])


def test_row_of_length_zero_keeps_the_carry_and_zeroes_the_gates():
    x = inputs.prologue_inputs(2, 5, 13, Hk=1, Hv=2, K=4, lengths=[0, 5])
    q, k, v, g, beta, new_tail = op.prologue(x.mixed, x.conv_w, x.a, x.b, x.A_log, x.dt_bias, 1, 2,
                                              tail=x.tail, lengths=x.lengths)
    assert np.array_equal(new_tail[0], x.tail[0].double().numpy())
    assert np.all(g[0] == 0) and np.all(beta[0] == 0)
    assert np.array_equal(new_tail[1], x.mixed[1, 2:5].double().numpy())
