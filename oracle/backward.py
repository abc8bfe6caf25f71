"""Gated delta rule backward oracle (float64, CPU, numpy).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may use it. It shares no code with ``gated_deltanet_rule_gb300``.

Reverse mode through the token recurrence of the forward oracle (Kev-4B-LiteRT
"r15_kernel_test.py", ``truth_f64``; DEG "model.py", ``delta_rule_reference``), per row and value
head h with key head h // r:

    k^ = k / sqrt(|k|^2 + 1e-6),  q~ = q / sqrt(|q|^2 + 1e-6) D^-1/2
    S_a = e^{g_t} S_{t-1};  kv = S_a^T k^;  delta = beta_t (v_t - kv);  S_t = S_a + k^ delta^T;  o_t = S_t^T q~

Given the upstream gradients dO (of o) and dS_T (of the final state), the adjoint dS of S_t is
carried from the last token to the first, each step undone in reverse order:

    dq~ = S_t dO_t;  dS += q~ dO_t^T
    dk^ += dS delta;  ddelta = dS^T k^
    dbeta = ddelta . (v - kv);  dv = beta ddelta;  dkv = -beta ddelta
    dS_a = dS + k^ dkv^T;  dk^ += S_a dkv
    dg = <S_a, dS_a>;  dS <- e^{g_t} dS_a                     (the adjoint of S_{t-1})

then through the normalisations (dx = s (dx^ - s^2 (x . dx^) x), s = (|x|^2 + eps)^-1/2, and D^-1/2
for q), summing dq, dk over the value heads that share a key head; dS0 is the final dS. The pages
train through the recurrence but print no backward; this is the plain reverse of the forward.
Pinned by ``tests/test_backward_oracle.py`` (central finite differences of the forward oracle and
autograd of a float64 PyTorch recurrence).
"""
from __future__ import annotations

import math

import numpy as np

EPS = 1e-6


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        return x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def backward(q, k, v, g, beta, S0, dO, dS_T=None):
    """Returns (dq [B,L,Hk,D], dk [B,L,Hk,D], dv [B,L,Hv,Dv], dg [B,L,Hv], dbeta [B,L,Hv],
    dS0 [B,Hv,D,Dv]) in float64. S0 None means zeros; dS_T None means no gradient on the state."""
    q, k, v, g, beta, S0, dO, dS_T = (_f64(t) for t in (q, k, v, g, beta, S0, dO, dS_T))
    B, L, Hk, D = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    r = Hv // Hk
    sq = 1.0 / np.sqrt((q * q).sum(-1) + EPS)            # [B, L, Hk]
    sk = 1.0 / np.sqrt((k * k).sum(-1) + EPS)
    qt = q * sq[..., None] / math.sqrt(D)
    kh = k * sk[..., None]
    dqt = np.zeros_like(q)
    dkh = np.zeros_like(k)
    dv = np.zeros_like(v)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dS0 = np.zeros((B, Hv, D, Dv))
    for b in range(B):
        for h in range(Hv):
            hk = h // r
            # forward, keeping every S_a and S_t (the test sizes are small)
            S = np.zeros((D, Dv)) if S0 is None else S0[b, h].copy()
            Sa_all, St_all, kv_all, dl_all = [], [], [], []
            for t in range(L):
                Sa = math.exp(g[b, t, h]) * S
                kv = Sa.T @ kh[b, t, hk]
                dl = beta[b, t, h] * (v[b, t, h] - kv)
                S = Sa + np.outer(kh[b, t, hk], dl)
                Sa_all.append(Sa)
                St_all.append(S)
                kv_all.append(kv)
                dl_all.append(dl)
            # reverse
            dS = np.zeros((D, Dv)) if dS_T is None else dS_T[b, h].copy()
            for t in range(L - 1, -1, -1):
                St, Sa, kv, dl = St_all[t], Sa_all[t], kv_all[t], dl_all[t]
                k1, q1 = kh[b, t, hk], qt[b, t, hk]
                dqt[b, t, hk] += St @ dO[b, t, h]
                dS = dS + np.outer(q1, dO[b, t, h])
                dkh[b, t, hk] += dS @ dl
                ddl = dS.T @ k1
                dbeta[b, t, h] = ddl @ (v[b, t, h] - kv)
                dv[b, t, h] = beta[b, t, h] * ddl
                dkv = -beta[b, t, h] * ddl
                dSa = dS + np.outer(k1, dkv)
                dkh[b, t, hk] += Sa @ dkv
                dg[b, t, h] = float((Sa * dSa).sum())
                dS = math.exp(g[b, t, h]) * dSa
            dS0[b, h] = dS
    # through the normalisations
    dq = (sq[..., None] * dqt - (sq ** 3)[..., None] * (q * dqt).sum(-1, keepdims=True) * q) / math.sqrt(D)
    dk = sk[..., None] * dkh - (sk ** 3)[..., None] * (k * dkh).sum(-1, keepdims=True) * k
    return dq, dk, dv, dg, dbeta, dS0
