"""Gated RMSNorm epilogue oracle (float64, CPU, numpy).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may use it. It shares no code with ``gated_deltanet_rule_gb300``.

DEG "model.py", ``_gated_rms(x, gate, w, eps)``, over the last dimension of x:
    x_hat = x / sqrt(mean(x^2) + eps);   out = w * x_hat * silu(gate),   silu(z) = z / (1 + e^-z).
The pages round x_hat and w * x_hat to the activation dtype on the way; this oracle keeps float64
throughout. Pinned by ``tests/test_epilogue_oracle.py``.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def silu(z):
    z = _f64(z)
    e = np.exp(-np.abs(z))
    sig = np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    return z * sig


def gated_rms(x, z, w, eps: float = 1e-6):
    x, w = _f64(x), _f64(w)
    x_hat = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return w * x_hat * silu(z)
