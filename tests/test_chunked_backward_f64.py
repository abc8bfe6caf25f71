"""Float64 chunked form of the gated delta rule backward, checked against the backward oracle.

The pages train through the recurrence but print no backward. The chunked forward (the algebra
the CUDA path computes, pinned in ``test_chunked_form_f64.py``) is, per 64-token chunk with
entering state S:

    A_ij = beta_i (k^_i . k^_j) e^{gamma_i - gamma_j} (j < i),  T = (I + A)^-1
    W = T diag(beta Gamma) K^,  U = T diag(beta) V,  Delta = U - W S
    P_ij = (q~_i . k^_j) e^{gamma_i - gamma_j} (j <= i)
    O = diag(Gamma) Q~ S + P Delta,   S' = Gamma_C S + K^T diag(e) Delta,  e_i = e^{gamma_C - gamma_i}

Its reverse, given dO and the adjoint dS' of the exiting state, is what the chunked backward
kernels compute. The sequential part is the adjoint chain, the forward chain transposed:

    dS = Gamma_C dS' + M'^T dS' + Q'^T dO     (M' = -K^T diag(e) W,  Q' = diag(Gamma) Q~ - P W)

and everything else is local to the chunk once S and dS' are known:

    dDelta = P^T dO + diag(e) K^ dS';   dU = dDelta;   dW = -dDelta S^T
    dQ~ = diag(Gamma) dO S^T + (dP o E) K^,   dP = dO Delta^T (j <= i),  E_ij = e^{gamma_i - gamma_j}
    dK^ = (dP o E)^T Q~ + diag(e) Delta dS'^T + diag(beta Gamma) T^T dW + (dA~ + dA~^T) K^
    dT = dU (diag(beta) V)^T + dW (diag(beta Gamma) K^)^T,   dA = -T^T dT T^T (j < i),
    dA~_ij = dA_ij beta_i E_ij,   dV = diag(beta) T^T dU
    dbeta_i = V_i . (T^T dU)_i + Gamma_i K^_i . (T^T dW)_i + sum_j dA_ij (k^_i . k^_j) E_ij
    dgamma_i = Gamma_i q~_i . (dO S^T)_i + sum_j (dP o P)_ij - sum_j (dP o P)_ji
               + beta_i Gamma_i K^_i . (T^T dW)_i + sum_j (dA o A)_ij - sum_j (dA o A)_ji
               - e_i k^_i . (dS' Delta_i)        (+ Gamma_C <S, dS'> + sum_j e_j k^_j . (dS' Delta_j) at i = C-1)
    dg_j = sum_{i >= j} dgamma_i  (within the chunk)

then the normalisations' backward and the sum over the value heads of a key head, as in the
oracle. Test code only: agreement with the token-level oracle to ~1e-11 pins the derivation.
"""
import math

import numpy as np

import oracle.backward as ob
from gated_deltanet_rule_gb300 import inputs

EPS = 1e-6


def chunked_backward_f64(q, k, v, g, beta, S0, dO, dS_T, C=64):
    B, L, Hk, D = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    r = Hv // Hk
    sq = 1.0 / np.sqrt((q * q).sum(-1) + EPS)
    sk = 1.0 / np.sqrt((k * k).sum(-1) + EPS)
    qt = q * sq[..., None] / math.sqrt(D)
    kh = k * sk[..., None]
    dqt = np.zeros((B, L, Hv, D))   # per value head, summed over the key head's value heads below
    dkh = np.zeros((B, L, Hv, D))
    dv = np.zeros_like(v)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dS0 = np.zeros((B, Hv, D, Dv))
    NC = (L + C - 1) // C
    for b in range(B):
        for h in range(Hv):
            hk = h // r
            # forward: the chunk-entry states
            S = np.zeros((D, Dv)) if S0 is None else S0[b, h].copy()
            states, loc = [], []
            for c in range(NC):
                c0, c1 = c * C, min(c * C + C, L)
                n = c1 - c0
                Q, K, V = qt[b, c0:c1, hk], kh[b, c0:c1, hk], v[b, c0:c1, h]
                be, gam = beta[b, c0:c1, h], np.cumsum(g[b, c0:c1, h])
                E = np.exp(np.where(np.tril(np.ones((n, n))) > 0, gam[:, None] - gam[None, :], -np.inf))
                A = be[:, None] * (K @ K.T) * np.tril(E, -1)
                T = np.linalg.inv(np.eye(n) + A)
                Gam = np.exp(gam)
                e = np.exp(gam[-1] - gam)
                W = T @ ((be * Gam)[:, None] * K)
                U = T @ (be[:, None] * V)
                P = (Q @ K.T) * E
                states.append(S.copy())
                Dl = U - W @ S
                loc.append((c0, c1, Q, K, V, be, gam, E, A, T, Gam, e, W, P, Dl))
                S = Gam[-1] * S + (e[:, None] * K).T @ Dl
            # backward: the adjoint chain, last chunk first
            dS = np.zeros((D, Dv)) if dS_T is None else dS_T[b, h].copy()
            for c in reversed(range(NC)):
                c0, c1, Q, K, V, be, gam, E, A, T, Gam, e, W, P, Dl = loc[c]
                S = states[c]
                dOc = dO[b, c0:c1, h]
                n = c1 - c0
                # chain: dS_c = Gamma_C dS' + M'^T dS' + Q'^T dO
                Mp = -K.T @ (e[:, None] * W)
                Qp = Gam[:, None] * Q - P @ W
                dS_prev = Gam[-1] * dS + Mp.T @ dS + Qp.T @ dOc
                # chunk-local gradients
                dDl = P.T @ dOc + e[:, None] * (K @ dS)
                dW = -dDl @ S.T
                dP = (dOc @ Dl.T) * np.tril(np.ones((n, n)))
                dPE = dP * E
                dQ = Gam[:, None] * (dOc @ S.T) + dPE @ K
                dK = dPE.T @ Q + e[:, None] * (Dl @ dS.T)
                TtdW = T.T @ dW
                TtdU = T.T @ dDl
                dT = dDl @ (be[:, None] * V).T + dW @ ((be * Gam)[:, None] * K).T
                dA = -(T.T @ dT @ T.T) * np.tril(np.ones((n, n)), -1)
                dAt = dA * be[:, None] * E
                dK += (be * Gam)[:, None] * TtdW + dAt @ K + dAt.T @ K
                dV = be[:, None] * TtdU
                dbe = (V * TtdU).sum(1) + Gam * (K * TtdW).sum(1) + (dA * (K @ K.T) * E).sum(1)
                dPP, dAA = dP * P, dA * A
                de = (K * (Dl @ dS.T)).sum(1) * e
                dgam = (Gam * (Q * (dOc @ S.T)).sum(1) + dPP.sum(1) - dPP.sum(0) + be * Gam * (K * TtdW).sum(1)
                        + dAA.sum(1) - dAA.sum(0) - de)
                dgam[-1] += Gam[-1] * (S * dS).sum() + de.sum()
                dg[b, c0:c1, h] = np.cumsum(dgam[::-1])[::-1]
                dqt[b, c0:c1, h] = dQ
                dkh[b, c0:c1, h] = dK
                dv[b, c0:c1, h] = dV
                dbeta[b, c0:c1, h] = dbe
                dS = dS_prev
            dS0[b, h] = dS
    # normalisations and the key-head sum
    dqt_k = dqt.reshape(B, L, Hk, r, D).sum(3)
    dkh_k = dkh.reshape(B, L, Hk, r, D).sum(3)
    dq = (sq[..., None] * dqt_k - sq[..., None] ** 3 * (q * dqt_k).sum(-1, keepdims=True) * q) / math.sqrt(D)
    dk = sk[..., None] * dkh_k - sk[..., None] ** 3 * (k * dkh_k).sum(-1, keepdims=True) * k
    return dq, dk, dv, dg, dbeta, dS0


def _rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


def _case(regime, L, seed, n_valid=None, init=True, dS=True, Dk=32):
    x = inputs.regime(regime, L, seed, Hk=2, Hv=4, B=2, Dk=Dk, init_state=init, n_valid=n_valid)
    dO, dS_T = inputs.upstream_grads(2, L, 4, seed + 1, Dk=Dk, with_dS_T=dS)
    args = [None if t is None else t.double().numpy() for t in (x.q, x.k, x.v, x.g, x.beta, x.S0, dO, dS_T)]
    return args


def test_chunked_backward_matches_oracle_ragged_multichunk():
    for regime, seed in (("R1", 61), ("R3", 62)):
        args = _case(regime, 150, seed)
        want = ob.backward(*args)
        got = chunked_backward_f64(*args, C=64)
        for name, a, w in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), got, want):
            assert _rel(a, w) < 1e-10, (regime, name, _rel(a, w))


def test_chunked_backward_small_chunks_pads_no_state():
    args = _case("R2", 70, 63, n_valid=50, init=False, dS=False)
    want = ob.backward(*args)
    for C in (16, 64):
        got = chunked_backward_f64(*args, C=C)
        for name, a, w in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), got, want):
            assert _rel(a, w) < 1e-10, (C, name, _rel(a, w))
