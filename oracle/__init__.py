"""Gated delta rule oracle (float64, CPU).

TEST INFRASTRUCTURE ONLY: this package is the checker that the CUDA library is compared
against. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import it. It shares no code with ``gated_deltanet_rule_gb300`` and never imports it.

The arithmetic lives in ``gdr_oracle.c`` (a plain token-by-token recurrence, the function
``truth_f64`` of the Kev-4B-LiteRT page "r15_kernel_test.py"); this module only widens inputs
to float64, calls it and returns numpy arrays. ``fork`` and ``decode_step`` are the same
recurrence with the initial state gathered by index (DEG "model.py", ``fork_delta_rule(h0,
h0_idx, store)``) and with L = 1 and the state updated in place (DEG ``DecodeGraph``).

Every function here is pinned by ``tests/test_oracle_pins.py`` and
``tests/test_chunked_form_f64.py`` against closed forms, a 50-digit brute force and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB = os.path.join(_HERE, "libgdr_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gdr_oracle.c with gcc (OpenMP, -O2, no -ffast-math) into libgdr_oracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math", "-ffp-contract=off",
               "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdr_oracle_forward.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp] + [ctypes.c_int] * 7
        lib.gdr_oracle_forward.restype = ctypes.c_int
        lib.gdr_oracle_max_threads.argtypes = []
        lib.gdr_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    """Widen any array-like (numpy, or a torch CPU tensor of any float dtype) to float64 exactly."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor of any float dtype: the conversion to float64 is exact
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().gdr_oracle_max_threads())


def forward(q, k, v, g, beta, S0=None, nthreads: int = 0):
    """o, S_T = recurrence over q,k [B,L,Hk,Dk], v [B,L,Hv,Dv], g,beta [B,L,Hv], S0 [B,Hv,Dk,Dv].

    Returns float64 numpy arrays o [B,L,Hv,Dv] and S_T [B,Hv,Dk,Dv].
    """
    q, k, v, g, beta, S0 = (_f64(x) for x in (q, k, v, g, beta, S0))
    B, L, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, L)
    assert g.shape == (B, L, Hv) and beta.shape == (B, L, Hv)
    if S0 is not None:
        assert S0.shape == (B, Hv, Dk, Dv)
    o = np.zeros((B, L, Hv, Dv), dtype=np.float64)
    S_T = np.zeros((B, Hv, Dk, Dv), dtype=np.float64)
    rc = _load().gdr_oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                    _ptr(o), _ptr(S_T), B, L, Hk, Hv, Dk, Dv, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_forward failed with code {rc}")
    return o, S_T


def fork(q, k, v, g, beta, trunk, trunk_idx, nthreads: int = 0):
    """Fork f continues its own copy of trunk[trunk_idx[f]] over its L_pad tokens.

    q,k [F,L,Hk,Dk], v [F,L,Hv,Dv], g,beta [F,L,Hv], trunk [N,Hv,Dk,Dv], trunk_idx [F] ints.
    Returns o [F,L,Hv,Dv] and the per-fork final states [F,Hv,Dk,Dv].
    """
    trunk = _f64(trunk)
    idx = np.asarray(trunk_idx.cpu() if hasattr(trunk_idx, "cpu") else trunk_idx, dtype=np.int64)
    if idx.min(initial=0) < 0 or idx.max(initial=0) >= trunk.shape[0]:
        raise IndexError("trunk index out of range")
    return forward(q, k, v, g, beta, trunk[idx], nthreads=nthreads)


def decode_step(q, k, v, g, beta, states, nthreads: int = 0):
    """One token per row (L = 1): returns o [F,1,Hv,Dv] and the updated states [F,Hv,Dk,Dv]."""
    return forward(q, k, v, g, beta, states, nthreads=nthreads)


if __name__ == "__main__":  # `python -m oracle` builds the library
    print(build(force="--force" in sys.argv))
