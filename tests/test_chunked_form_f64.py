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


def chunk_factors_f64(q, k, v, g, beta, b, h, r, C=64):
    """Per chunk of row b, value head h: (Gamma_C, M', N, Q', P U) of the folded form the CUDA path
    evaluates: o = Q' S + P U and S' = Gamma_C S + M' S + N, with Q' = diag(Gamma) Q~ - P W,
    M' = -(diag(exp(gamma_C - gamma)) K^)^T W and N = (diag(exp(gamma_C - gamma)) K^)^T U."""
    L, Dk = q.shape[1], q.shape[3]
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6) / math.sqrt(Dk)
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    out = []
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
        lowd = np.tril(np.ones((n, n)))
        P = (Q @ K.T) * np.exp(np.where(lowd > 0, diff, 0.0)) * lowd
        Ks = np.exp(gam[-1] - gam)[:, None] * K
        out.append((Gam[-1], -Ks.T @ W, Ks.T @ U, Gam[:, None] * Q - P @ W, P @ U))
    return out


def test_folded_form_matches_oracle():
    """The form the CUDA kernels evaluate: one state product per chunk on the chain."""
    x = inputs.regime("R1", 200, 14, Hk=2, Hv=4, Dk=32, init_state=True)
    q, k, v, g, beta, S0 = [t.double().numpy() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    o_ref, S_ref = oracle.forward(q, k, v, g, beta, S0)
    for h in range(4):
        S = S0[0, h].copy()
        for ci, (Gc, M, N, Qp, PU) in enumerate(chunk_factors_f64(q, k, v, g, beta, 0, h, 2)):
            o = Qp @ S + PU
            assert _rel(o, o_ref[0, 64 * ci:64 * ci + len(o), h]) < 1e-12
            S = Gc * S + M @ S + N
        assert _rel(S, S_ref[0, h]) < 1e-12


def test_chunk_pairs_compose_into_one_step():
    """Two chunks compose into one step of the same form, S'' = G1 G2 S + M'' S + N'', with
    M'' = G2 M1 + G1 M2 + M2 M1 and N'' = G2 N1 + M2 N1 + N2, and the second chunk's output from the
    pair's entering state, o2 = (G1 Q'2 + Q'2 M1) S + (Q'2 N1 + P U2): the algebra a chain of
    half the steps would use."""
    x = inputs.regime("R1", 256, 15, Hk=2, Hv=4, Dk=32, init_state=True)
    q, k, v, g, beta, S0 = [t.double().numpy() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0)]
    o_ref, S_ref = oracle.forward(q, k, v, g, beta, S0)
    for h in range(4):
        f = chunk_factors_f64(q, k, v, g, beta, 0, h, 2)
        S = S0[0, h].copy()
        for p in range(0, len(f), 2):
            (G1, M1, N1, Q1, PU1), (G2, M2, N2, Q2, PU2) = f[p], f[p + 1]
            o1 = Q1 @ S + PU1
            o2 = (G1 * Q2 + Q2 @ M1) @ S + (Q2 @ N1 + PU2)
            assert _rel(o1, o_ref[0, 64 * p:64 * p + 64, h]) < 1e-12
            assert _rel(o2, o_ref[0, 64 * p + 64:64 * p + 128, h]) < 1e-12
            Mpp = G2 * M1 + G1 * M2 + M2 @ M1
            Npp = G2 * N1 + M2 @ N1 + N2
            S = G1 * G2 * S + Mpp @ S + Npp
        assert _rel(S, S_ref[0, h]) < 1e-12
