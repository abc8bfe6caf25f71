"""GDN prologue oracle (float64, CPU, numpy).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may use it. It shares no code with ``gated_deltanet_rule_gb300``.

What it computes, step by step as DEG "model.py" writes it in ``_linear_layer``:
  - ``_conv_silu(ext, w)``: ext = [tail; mixed] along positions (K-1 carried inputs, then the L new
    ones); out[t] = sum_{j < K} ext[t + j] w[:, j]; result silu(out) = out / (1 + exp(-out)).
  - the channel split of the result into q (Hk D channels), k (Hk D) and v (Hv D), as heads.
  - ``_dn_gates(b, a, A_log, dt_bias, valid)``: beta = sigmoid(b) valid,
    g = -exp(A_log) softplus(a + dt_bias) valid (softplus(x) = log(1 + e^x)).
  - the carry: new_tail = ext[len_b + j], j < K-1 (the ``gather`` at lengths_new + arange(K-1)).
Inputs are widened exactly to float64 (bf16 -> float32 -> float64). Pinned by
``tests/test_prologue_oracle.py`` (closed forms, a brute-force convolution, the carry handoff).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))                         # never overflows
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def softplus(x):
    return np.logaddexp(0.0, np.asarray(x, dtype=np.float64))   # log(1 + e^x), exact in float64


def silu(x):
    return np.asarray(x, dtype=np.float64) * sigmoid(x)


def conv_silu(ext, w):
    """ext [B, K-1+L, C], w [C, K] -> silu of the depthwise causal convolution, [B, L, C]."""
    ext, w = _f64(ext), _f64(w)
    K = w.shape[1]
    L = ext.shape[1] - K + 1
    out = ext[:, 0:L] * w[:, 0]
    for j in range(1, K):
        out = out + ext[:, j:j + L] * w[:, j]
    return silu(out)


def dn_gates(a, b, A_log, dt_bias, valid):
    """a, b [B, L, Hv]; A_log, dt_bias [Hv]; valid [B, L] (1 real, 0 pad) -> (beta, g)."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    v = _f64(valid)[..., None]
    beta = sigmoid(b) * v
    g = -np.exp(A_log) * softplus(a + dt_bias) * v
    return beta, g


def prologue(mixed, conv_w, a, b, A_log, dt_bias, Hk, Hv, D=128, tail=None, lengths=None):
    """Returns (q [B,L,Hk,D], k [B,L,Hk,D], v [B,L,Hv,D], g [B,L,Hv], beta [B,L,Hv], new_tail
    [B,K-1,C]) in float64. ``tail`` None means zeros; ``lengths`` None means L for every row."""
    mixed, w = _f64(mixed), _f64(conv_w)
    B, L, C = mixed.shape
    K = w.shape[1]
    assert C == (2 * Hk + Hv) * D and w.shape[0] == C
    tail = np.zeros((B, K - 1, C)) if tail is None else _f64(tail)
    ext = np.concatenate([tail, mixed], axis=1)
    y = conv_silu(ext, w)
    q = y[..., :Hk * D].reshape(B, L, Hk, D)
    k = y[..., Hk * D:2 * Hk * D].reshape(B, L, Hk, D)
    v = y[..., 2 * Hk * D:].reshape(B, L, Hv, D)
    lens = np.full(B, L, dtype=np.int64) if lengths is None else np.asarray(_f64(lengths), dtype=np.int64)
    valid = (np.arange(L)[None, :] < lens[:, None]).astype(np.float64)
    beta, g = dn_gates(a, b, A_log, dt_bias, valid)
    new_tail = np.stack([ext[i, lens[i]:lens[i] + K - 1] for i in range(B)]) if K > 1 else np.zeros((B, 0, C))
    return q, k, v, g, beta, new_tail
