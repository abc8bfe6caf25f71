"""Float64 chunked (WY) form of the gated delta rule, checked against the token oracle.

The pages print no chunk code; their kernel forms ("R64": 64-token chunks and a triangular
inverse; "ec": exp clamp; "dd": direct decay) are named in the Kev-4B-LiteRT page
"r15_kernel_test.py". The algebra below is derived from the recurrence and is what the CUDA
path computes per chunk. Within a chunk with entering state S, cumulative log-decay gamma_i
and Gamma_i = exp(gamma_i):

  A_ij  = beta_i (k^_i . k^_j) exp(gamma_i - gamma_j)          j < i, else 0
  T     = (I + A)^-1                                           unit lower triangular
  W     = T diag(beta Gamma) K^ ,  U = T diag(beta) V
  Vnew  = U - W S                                              the chunk's delta rows
  P_ij  = (q~_i . k^_j) exp(gamma_i - gamma_j)                 j <= i, else 0
  O     = diag(Gamma) Q~ S + P Vnew
  S'    = Gamma_C S + (diag(exp(gamma_C - gamma)) K^)^T Vnew

This file is test code: it pins the oracle with an independent formulation (agreement to
~1e-12) and shows why the pair decay must be computed directly (the ratio of cumulative
decays underflows to 0/0 in fp32 at the strong-decay regime).
"""
import math

import numpy as np

import oracle
from gated_deltanet_rule_gb300 import inputs


def chunked_f64(q, k, v, g, beta, S0, C=64):
    B, L, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    r = Hv // Hk
    o = np.zeros((B, L, Hv, Dv))
    ST = np.zeros((B, Hv, Dk, Dv))
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6) / math.sqrt(Dk)
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    for b in range(B):
        for h in range(Hv):
            S = np.zeros((Dk, Dv)) if S0 is None else S0[b, h].copy()
            for c0 in range(0, L, C):
                c1 = min(c0 + C, L)
                Q, K, V = qn[b, c0:c1, h // r], kn[b, c0:c1, h // r], v[b, c0:c1, h]
                be, gam = beta[b, c0:c1, h], np.cumsum(g[b, c0:c1, h])
                n = c1 - c0
                diff = gam[:, None] - gam[None, :]
                low = np.tril(np.ones((n, n)), -1)
                A = be[:, None] * (K @ K.T) * np.exp(np.where(low > 0, diff, 0.0)) * low
                T = np.linalg.inv(np.eye(n) + A)
                Gam = np.exp(gam)
                W = T @ ((be * Gam)[:, None] * K)
                U = T @ (be[:, None] * V)
                Vn = U - W @ S
                lowd = np.tril(np.ones((n, n)))
                P = (Q @ K.T) * np.exp(np.where(lowd > 0, diff, 0.0)) * lowd
                o[b, c0:c1, h] = Gam[:, None] * (Q @ S) + P @ Vn
                S = Gam[-1] * S + (np.exp(gam[-1] - gam)[:, None] * K).T @ Vn
            ST[b, h] = S
    return o, ST


def _rel(a, b):
    return np.abs(a - b).max() / np.abs(b).max()


def test_chunked_matches_oracle_ragged_strong_decay():
    x = inputs.regime("R1", 150, 12, Hk=2, Hv=4, Dk=32, init_state=True)
    args = [t.double().numpy() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    o, S = oracle.forward(*args)
    for C in (16, 64):
        oc, Sc = chunked_f64(*args, C=C)
        assert _rel(oc, o) < 1e-12 and _rel(Sc, S) < 1e-12


def test_chunked_matches_oracle_pads_and_correlated_keys():
    for name, seed in (("R3", 32), ("R4", 41), ("R2", 22)):
        x = inputs.regime(name, 130, seed, Hk=2, Hv=4, Dk=32, init_state=True, n_valid=100)
        args = [t.double().numpy() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
        o, S = oracle.forward(*args)
        oc, Sc = chunked_f64(*args, C=64)
        assert _rel(oc, o) < 1e-11 and _rel(Sc, S) < 1e-11


def test_ratio_of_cumulative_decays_fails_in_fp32_direct_form_does_not():
    # g = -1.7 per token lies inside R1's range [-3.0, -0.05]; after 64 tokens gamma = -108.8,
    # below the smallest fp32 subnormal (about exp(-103.3)), so Gamma underflows to exactly 0
    g = np.full(64, -1.7, dtype=np.float32)
    gam = np.cumsum(g).astype(np.float32)
    Gam = np.exp(gam)
    assert Gam[-1] == 0.0
    with np.errstate(all="ignore"):
        ratio = Gam[:, None] / Gam[None, :]             # Gamma_i / Gamma_j
    i, j = np.tril_indices(64)
    assert not np.isfinite(ratio[i, j]).all()           # 0/0 late in the chunk
    direct = np.exp(gam[i] - gam[j])                    # computed per pair: finite, <= 1
    assert np.isfinite(direct).all() and direct.max() <= 1.0
    np.testing.assert_allclose(direct, np.exp(-1.7 * (i - j).astype(np.float64)), rtol=1e-4, atol=1e-30)
