"""Pins for the float64 oracle: each test checks it against something other than itself.

Pins (the recurrence is the one of the Kev-4B-LiteRT page "r15_kernel_test.py", truth_f64):
  * L = 1 closed form: o = e^g S0^T q~ + (k^.q~) beta (v - e^g S0^T k^), S1 = e^g S0 + k^ delta^T
  * 50-digit brute force at D = 4 using the matrix form S_t = e^g (I - beta k k^T) S + beta k v^T
  * pad invariance (beta = g = 0 leaves the state bit-identical; DEG "model.py" _dn_gates)
  * split-sequence equivalence (state handed off between two calls; DEG chunked prefill)
  * exact 2^8 joint linearity in (v, S0) and its negative control (the vs<k> contract)
  * closed form of the one-key, no-decay regime R4
  * head map h -> h // r (repeat_interleave order, not tiling)
  * eps inside the square root of the l2 norm; zero key gives k^ = 0
"""
import math

import mpmath
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_rule_gb300 import inputs


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _l2n(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)


def _small(B=2, L=9, Hk=2, Hv=4, Dk=8, Dv=6, seed=0, s0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, L, Hk, Dk))
    k = rng.standard_normal((B, L, Hk, Dk))
    v = rng.standard_normal((B, L, Hv, Dv))
    g = -rng.uniform(0.05, 3.0, (B, L, Hv))
    beta = rng.uniform(0.2, 0.9, (B, L, Hv))
    S0 = 0.1 * rng.standard_normal((B, Hv, Dk, Dv)) if s0 else None
    return q, k, v, g, beta, S0


def test_l1_closed_form():
    q, k, v, g, beta, S0 = _small(L=1, seed=1)
    o, S1 = oracle.forward(q, k, v, g, beta, S0)
    r = v.shape[2] // q.shape[2]
    qh = np.repeat(_l2n(q[:, 0]), r, axis=1) / math.sqrt(q.shape[-1])   # [B, Hv, Dk]
    kh = np.repeat(_l2n(k[:, 0]), r, axis=1)
    e = np.exp(g[:, 0])[..., None]                                      # [B, Hv, 1]
    read = np.einsum("bhij,bhi->bhj", S0, kh)
    delta = beta[:, 0][..., None] * (v[:, 0] - e * read)
    o_ref = e * np.einsum("bhij,bhi->bhj", S0, qh) + (kh * qh).sum(-1, keepdims=True) * delta
    S_ref = e[..., None] * S0 + kh[..., :, None] * delta[..., None, :]
    np.testing.assert_allclose(o[:, 0], o_ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S1, S_ref, rtol=1e-13, atol=1e-14)


def test_bruteforce_d4_matrix_form_50_digits():
    """Different formulation (a product of matrices), 50 significant digits, D = 4, r = 2."""
    mpmath.mp.dps = 50
    B, L, Hk, Hv, D = 1, 8, 1, 2, 4
    q, k, v, g, beta, S0 = _small(B, L, Hk, Hv, D, D, seed=7)
    o, ST = oracle.forward(q, k, v, g, beta, S0)
    for h in range(Hv):
        S = mpmath.matrix(S0[0, h].tolist())
        for t in range(L):
            kt = mpmath.matrix(k[0, t, h // 2].tolist())
            qt = mpmath.matrix(q[0, t, h // 2].tolist())
            kn = kt / mpmath.sqrt(sum(x * x for x in kt) + mpmath.mpf("1e-6"))
            qn = qt / mpmath.sqrt(sum(x * x for x in qt) + mpmath.mpf("1e-6")) / mpmath.sqrt(D)
            b = mpmath.mpf(beta[0, t, h])
            M = mpmath.exp(mpmath.mpf(g[0, t, h])) * (mpmath.eye(D) - b * kn * kn.T)
            S = M * S + b * kn * mpmath.matrix(v[0, t, h].tolist()).T
            ot = S.T * qn
            for j in range(D):
                assert abs(float(ot[j]) - o[0, t, h, j]) <= 1e-13 * max(1.0, abs(float(ot[j])))
        for i in range(D):
            for j in range(D):
                assert abs(float(S[i, j]) - ST[0, h, i, j]) <= 1e-13 * max(1.0, abs(float(S[i, j])))


def test_pad_invariance_bit_exact():
    q, k, v, g, beta, S0 = _small(L=12, seed=2)
    n = 7
    g2, b2 = g.copy(), beta.copy()
    g2[:, n:] = 0.0
    b2[:, n:] = 0.0
    o_full, S_full = oracle.forward(q, k, v, g2, b2, S0)
    o_n, S_n = oracle.forward(q[:, :n], k[:, :n], v[:, :n], g[:, :n], beta[:, :n], S0)
    assert np.array_equal(S_full, S_n)                  # pads leave the state untouched
    assert np.array_equal(o_full[:, :n], o_n)
    # the state after a pad equals the state before it; the output at a pad reads that state
    o_p, _ = oracle.forward(q[:, n:n + 1], k[:, n:n + 1], v[:, n:n + 1], g2[:, n:n + 1],
                            b2[:, n:n + 1], S_n)
    assert np.array_equal(o_p[:, 0], o_full[:, n])


def test_split_sequence_handoff_bit_exact():
    q, k, v, g, beta, S0 = _small(L=13, seed=3)
    o, S = oracle.forward(q, k, v, g, beta, S0)
    for cut in (1, 6, 12):
        o1, S1 = oracle.forward(q[:, :cut], k[:, :cut], v[:, :cut], g[:, :cut], beta[:, :cut], S0)
        o2, S2 = oracle.forward(q[:, cut:], k[:, cut:], v[:, cut:], g[:, cut:], beta[:, cut:], S1)
        assert np.array_equal(np.concatenate([o1, o2], 1), o)
        assert np.array_equal(S2, S)


def test_joint_scale_2_pow_8_exact_and_negative_control():
    q, k, v, g, beta, S0 = _small(L=10, seed=4)
    o, S = oracle.forward(q, k, v, g, beta, S0)
    o8, S8 = oracle.forward(q, k, v * 256.0, g, beta, S0 * 256.0)
    assert np.array_equal(o8, o * 256.0) and np.array_equal(S8, S * 256.0)
    # the wrong contract (v scaled, state not) must not reproduce the scaled result
    o_bad, _ = oracle.forward(q, k, v * 256.0, g, beta, S0)
    assert np.abs(o_bad - o8).max() > 1e-3 * np.abs(o8).max()


def test_r4_one_key_no_decay_closed_form():
    """R4: one key, g = 0. With kappa = |k^|^2 and m_t = S_t^T k^:
    m_t = (1 - kappa beta) m_{t-1} + kappa beta v_t, S_t = S0 + k^ (m_t - m_0)^T / kappa."""
    x = inputs.regime("R4", 40, 41, Hk=2, Hv=4, Dk=16, init_state=True)
    o, S = oracle.forward(x.q, x.k, x.v, x.g, x.beta, x.S0)
    q, k, v = (t.double().numpy() for t in (x.q, x.k, x.v))
    beta, S0 = x.beta.double().numpy(), x.S0.double().numpy()
    for h in range(4):
        kk = k[0, 0, h // 2]
        kh = kk / math.sqrt((kk * kk).sum() + 1e-6)
        kap = (kh * kh).sum()
        m0 = S0[0, h].T @ kh
        m = m0.copy()
        for t in range(40):
            m = (1 - kap * beta[0, t, h]) * m + kap * beta[0, t, h] * v[0, t, h]
            qq = q[0, t, h // 2]
            qt = qq / math.sqrt((qq * qq).sum() + 1e-6) / 4.0
            o_ref = S0[0, h].T @ qt + (kh @ qt) * (m - m0) / kap
            np.testing.assert_allclose(o[0, t, h], o_ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(S[0, h], S0[0, h] + np.outer(kh, (m - m0) / kap), rtol=1e-10, atol=1e-12)


def test_head_map_is_interleave_not_tiling():
    q, k, v, g, beta, S0 = _small(B=1, L=6, Hk=3, Hv=6, seed=5)
    o, S = oracle.forward(q, k, v, g, beta, S0)
    # explicit interleave (each key head copied to 2 adjacent value heads), then r = 1
    qi, ki = np.repeat(q, 2, axis=2), np.repeat(k, 2, axis=2)
    assert np.array_equal(qi[:, :, 0::2], qi[:, :, 1::2])   # head pairs identical
    o1, S1 = oracle.forward(qi, ki, v, g, beta, S0)
    assert np.array_equal(o, o1) and np.array_equal(S, S1)
    # tiling (h -> h % Hk) is a different map and gives a different answer
    qt, kt = np.tile(q, (1, 1, 2, 1)), np.tile(k, (1, 1, 2, 1))
    o2, _ = oracle.forward(qt, kt, v, g, beta, S0)
    assert np.abs(o2 - o).max() > 1e-3


def test_eps_inside_sqrt_and_zero_key():
    B, L, Hk, Hv, D = 1, 1, 1, 1, 4
    q = np.array([[[[1e-4, 0, 0, 0]]]])
    k = np.array([[[[1e-4, 0, 0, 0]]]])
    v = np.array([[[[1.0, 2.0, 3.0, 4.0]]]])
    g = np.zeros((1, 1, 1))
    beta = np.ones((1, 1, 1))
    o, S = oracle.forward(q, k, v, g, beta, None)
    kh = 1e-4 / math.sqrt(1e-8 + 1e-6)        # eps added to the sum of squares, then sqrt
    qh = kh / 2.0                              # D^-0.5 = 1/2
    np.testing.assert_allclose(S[0, 0, 0], kh * v[0, 0, 0], rtol=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], kh * qh * v[0, 0, 0], rtol=1e-14)
    # zero key: k^ = 0, nothing is written, no NaN
    o0, S0 = oracle.forward(q, np.zeros_like(k), v, g, beta, None)
    assert np.all(S0 == 0) and np.all(o0 == 0)


def test_fork_and_decode_wrappers():
    q, k, v, g, beta, _ = _small(B=3, L=5, seed=6, s0=False)
    trunk = 0.1 * _rand((2, 4, 8, 6), 9)
    idx = np.array([1, 0, 1])
    o, S = oracle.fork(q, k, v, g, beta, trunk, idx)
    for f in range(3):
        of, Sf = oracle.forward(q[f:f + 1], k[f:f + 1], v[f:f + 1], g[f:f + 1], beta[f:f + 1],
                                trunk[idx[f]][None])
        assert np.array_equal(of, o[f:f + 1]) and np.array_equal(Sf, S[f:f + 1])
    with pytest.raises(IndexError):
        oracle.fork(q, k, v, g, beta, trunk, np.array([0, 2, 1]))
    od, Sd = oracle.decode_step(q[:, :1], k[:, :1], v[:, :1], g[:, :1], beta[:, :1], S)
    of, Sf = oracle.forward(q[:, :1], k[:, :1], v[:, :1], g[:, :1], beta[:, :1], S)
    assert np.array_equal(od, of) and np.array_equal(Sd, Sf)


def test_bf16_inputs_are_widened_exactly():
    x = inputs.regime("R1", 5, 1, Hk=1, Hv=2, Dk=8, dtype=torch.bfloat16)
    o1, _ = oracle.forward(x.q, x.k, x.v, x.g, x.beta)
    o2, _ = oracle.forward(x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(),
                           x.g.double().numpy(), x.beta.double().numpy())
    assert np.array_equal(o1, o2)
