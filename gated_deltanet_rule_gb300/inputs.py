"""Seeded synthetic inputs for the gated delta rule.

This module draws random numbers and lays them out; it holds none of the method's
arithmetic (no normalisation, no head interleave, no decay, no recurrence). Both the
oracle tests and the CUDA tests draw their inputs here, so the two sides see the same
values without sharing any other code.

Recipes follow the input generator ``regime`` of the Kev-4B-LiteRT page
"r15_kernel_test.py" (draw order q, k, v, beta, g, S0; regimes R1..R4), with two
differences: q and k stay at the key-head count (value head h reads key head h // r by
index, so no copy is made here), and positions at or after ``n_valid`` are pads with
beta = g = 0 (DEG "model.py", ``_dn_gates``: pads are exact no-ops). q, k, v at pads keep
their drawn values.

All tensors are CPU torch tensors. q, k, v are float32 or bfloat16 (drawn in float32,
then rounded); g, beta and states are always float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D = 128  # key and value head dimension at the Qwen3.5 4B / 0.8B shapes


@dataclass
class GdrInputs:
    q: torch.Tensor            # [B, L, Hk, D]
    k: torch.Tensor            # [B, L, Hk, D]
    v: torch.Tensor            # [B, L, Hv, D]
    g: torch.Tensor            # [B, L, Hv] float32, natural-log decay (<= 0)
    beta: torch.Tensor         # [B, L, Hv] float32, write strength
    S0: torch.Tensor | None    # [B, Hv, D, D] float32 or None (zeros)
    n_valid: int | None = None  # positions >= n_valid are pads (beta = g = 0)
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, L, Hk, Dk = self.q.shape
        return B, L, Hk, self.v.shape[2], Dk


def regime(name: str, L: int, seed: int, Hk: int = 16, Hv: int = 32, Dk: int = D, B: int = 1,
           init_state: bool = False, n_valid: int | None = None,
           dtype: torch.dtype = torch.float32) -> GdrInputs:
    """One of the four regimes R1..R4.

    R1: random keys, strong decay      beta = 0.2 + 0.7 U, g = -(0.05 + 2.95 U)
    R2: random keys, weak decay        beta = 0.2 + 0.7 U, g = -0.02 U
    R3: correlated keys (u sqrt(D)/|u| + 0.3 N), weak decay, beta = 0.3 + 0.7 U
    R4: one key at every token, no decay, beta = 0.5
    """
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, L, Hk, Dk, generator=gen)
    if name in ("R1", "R2"):
        k = torch.randn(B, L, Hk, Dk, generator=gen)
    elif name == "R3":
        u = torch.randn(B, 1, Hk, Dk, generator=gen)
        u = u / u.norm(dim=-1, keepdim=True) * Dk ** 0.5
        k = u + 0.3 * torch.randn(B, L, Hk, Dk, generator=gen)
    elif name == "R4":
        k = torch.randn(B, 1, Hk, Dk, generator=gen).expand(B, L, Hk, Dk).contiguous()
    else:
        raise ValueError(name)
    v = torch.randn(B, L, Hv, Dk, generator=gen)
    if name == "R1":
        beta = 0.2 + 0.7 * torch.rand(B, L, Hv, generator=gen)
        g = -(0.05 + 2.95 * torch.rand(B, L, Hv, generator=gen))
    elif name in ("R2", "R3"):
        beta = (0.2 if name == "R2" else 0.3) + 0.7 * torch.rand(B, L, Hv, generator=gen)
        g = -0.02 * torch.rand(B, L, Hv, generator=gen)
    else:
        beta = torch.full((B, L, Hv), 0.5)
        g = torch.zeros(B, L, Hv)
    S0 = torch.randn(B, Hv, Dk, Dk, generator=gen) * 0.1 if init_state else None
    if n_valid is not None and n_valid < L:
        beta[:, n_valid:] = 0.0
        g[:, n_valid:] = 0.0
    q, k, v = (x.to(dtype) for x in (q, k, v))
    return GdrInputs(q, k, v, g.contiguous(), beta.contiguous(), S0, n_valid,
                     {"regime": name, "seed": seed})


def upstream_grads(B: int, L: int, Hv: int, seed: int, dtype: torch.dtype = torch.float32, Dk: int = D,
                   with_dS_T: bool = True):
    """Seeded upstream gradients for the backward: dO ~ N(0, 1) [B, L, Hv, D] in ``dtype`` and
    dS_T ~ 0.1 N(0, 1) [B, Hv, D, D] float32 (None when ``with_dS_T`` is False)."""
    gen = torch.Generator().manual_seed(seed)
    dO = torch.randn(B, L, Hv, Dk, generator=gen).to(dtype)
    dS_T = 0.1 * torch.randn(B, Hv, Dk, Dk, generator=gen) if with_dS_T else None
    return dO, dS_T


# ---------------------------------------------------------------------------------------------
# The five workloads (single row fp32, padded fp32 regimes, 4B prefill, 0.8B long prefill, forks)
# ---------------------------------------------------------------------------------------------

def config1(seed: int = 11) -> GdrInputs:
    """fp32, one row, L = 64, 16 key heads -> 32 value heads, R1 distributions, no S0, no pads."""
    x = regime("R1", 64, seed, 16, 32, D, init_state=False, dtype=torch.float32)
    x.meta["workload"] = "single row fp32 L=64 Hk=16 Hv=32 D=128"
    return x


CONFIG2_REGIMES = {"a": ("R2", 22), "b": ("R3", 32), "c": ("R4", 41)}


def config2(which: str = "a") -> GdrInputs:
    """fp32, L = 130 with 100 valid tokens then pads, S0 = 0.1 N; (a) R2, (b) R3, (c) R4."""
    name, seed = CONFIG2_REGIMES[which]
    x = regime(name, 130, seed, 16, 32, D, init_state=True, n_valid=100, dtype=torch.float32)
    x.meta["workload"] = f"padded fp32 L=130 valid=100 regime {name}"
    return x


def config3(seed: int = 3, L: int = 4096) -> GdrInputs:
    """bf16 prefill row at 4B shapes: L = 4096, 16 -> 32 heads, R1 distributions, S0 = 0.1 N."""
    x = regime("R1", L, seed, 16, 32, D, init_state=True, dtype=torch.bfloat16)
    x.meta["workload"] = f"prefill bf16 L={L} Hk=16 Hv=32 D=128 with S0"
    return x


def config4(seed: int = 4, L: int = 8192) -> GdrInputs:
    """bf16 long prefill at 0.8B shapes: L = 8192, 16 = 16 heads, weak decay, no S0."""
    x = regime("R2", L, seed, 16, 16, D, init_state=False, dtype=torch.bfloat16)
    x.meta["workload"] = f"long prefill bf16 L={L} Hk=16 Hv=16 D=128"
    return x


@dataclass
class ForkInputs:
    trunk: torch.Tensor        # [N, Hv, D, D] float32
    trunk_idx: torch.Tensor    # [F] int64
    lengths: torch.Tensor      # [F] int64 real tokens per fork
    fork: GdrInputs            # [F, L_pad, ...] with beta = g = 0 at pads
    decode: list               # per step: GdrInputs with L = 1 (all rows active)
    meta: dict = field(default_factory=dict)


def config5(seed: int = 5, F: int = 256, steps: int = 32, Hk: int = 16, Hv: int = 32,
            len_lo: int = 8, len_hi: int = 64) -> ForkInputs:
    """One trunk state copied into F forks of length U{len_lo..len_hi}, padded to a multiple of 64
    with beta = g = 0, then ``steps`` decode steps (L = 1) per fork. bf16 q/k/v, R1 gates."""
    gen = torch.Generator().manual_seed(seed)
    trunk = torch.randn(1, Hv, D, D, generator=gen) * 0.1
    lengths = torch.randint(len_lo, len_hi + 1, (F,), generator=gen, dtype=torch.int64)
    L_pad = 64 * math.ceil(int(lengths.max()) / 64)
    q = torch.randn(F, L_pad, Hk, D, generator=gen)
    k = torch.randn(F, L_pad, Hk, D, generator=gen)
    v = torch.randn(F, L_pad, Hv, D, generator=gen)
    beta = 0.2 + 0.7 * torch.rand(F, L_pad, Hv, generator=gen)
    g = -(0.05 + 2.95 * torch.rand(F, L_pad, Hv, generator=gen))
    pad = torch.arange(L_pad)[None, :] >= lengths[:, None]          # [F, L_pad]
    beta[pad] = 0.0
    g[pad] = 0.0
    fork = GdrInputs(q.bfloat16(), k.bfloat16(), v.bfloat16(), g, beta, None, None,
                     {"regime": "R1", "seed": seed})
    dec = []
    for _ in range(steps):
        dq = torch.randn(F, 1, Hk, D, generator=gen)
        dk = torch.randn(F, 1, Hk, D, generator=gen)
        dv = torch.randn(F, 1, Hv, D, generator=gen)
        db = 0.2 + 0.7 * torch.rand(F, 1, Hv, generator=gen)
        dg = -(0.05 + 2.95 * torch.rand(F, 1, Hv, generator=gen))
        dec.append(GdrInputs(dq.bfloat16(), dk.bfloat16(), dv.bfloat16(), dg, db, None))
    trunk_idx = torch.zeros(F, dtype=torch.int64)
    return ForkInputs(trunk, trunk_idx, lengths, fork, dec,
                      {"workload": f"fork batch F={F} L_pad={L_pad} + {steps} decode steps",
                       "L_pad": L_pad})


@dataclass
class PrologueInputs:
    mixed: torch.Tensor            # [B, L, C] bfloat16, C = (2 Hk + Hv) D: the q|k|v projection
    conv_w: torch.Tensor           # [C, K] float32 depthwise causal weights
    a: torch.Tensor                # [B, L, Hv] float32 decay projection
    b: torch.Tensor                # [B, L, Hv] float32 write-strength projection
    A_log: torch.Tensor            # [Hv] float32
    dt_bias: torch.Tensor          # [Hv] float32
    tail: torch.Tensor | None      # [B, K-1, C] bfloat16 carried inputs, or None (zeros)
    lengths: torch.Tensor | None   # [B] int32 valid tokens per row, or None (all L)
    Hk: int = 16
    Hv: int = 32


def prologue_inputs(B: int, L: int, seed: int, Hk: int = 16, Hv: int = 32, K: int = 4,
                    with_tail: bool = True, lengths=None) -> PrologueInputs:
    """Synthetic GDN-prologue inputs (the pages print no initialisation): mixed, tail, a, b ~ N(0, 1)
    (mixed and tail rounded to bf16), conv_w ~ U(-1, 1) / sqrt(K), A_log = log U(1, 16),
    dt_bias ~ U(-5, 0); ``lengths`` a list of valid token counts per row (None = all L)."""
    gen = torch.Generator().manual_seed(seed)
    C = (2 * Hk + Hv) * D
    mixed = torch.randn(B, L, C, generator=gen).bfloat16()
    tail = torch.randn(B, K - 1, C, generator=gen).bfloat16() if with_tail else None
    conv_w = (2 * torch.rand(C, K, generator=gen) - 1) / math.sqrt(K)
    a = torch.randn(B, L, Hv, generator=gen)
    b = torch.randn(B, L, Hv, generator=gen)
    A_log = torch.log(1 + 15 * torch.rand(Hv, generator=gen))
    dt_bias = -5 * torch.rand(Hv, generator=gen)
    lens = None if lengths is None else torch.tensor(lengths, dtype=torch.int32)
    return PrologueInputs(mixed, conv_w, a, b, A_log, dt_bias, tail, lens, Hk, Hv)
