"""Python binding of libgdr (the C ABI in include/gdr.h): argument marshalling only.

Each function checks tensor devices, dtypes, shapes and contiguity, allocates outputs the
caller did not pass (torch.empty: memory plumbing, no arithmetic), hands raw device pointers
and the current CUDA stream to the library and raises ``GdrError`` on a non-OK status. Every
step of the computation runs in the library's kernels; there is no CPU fallback: if
``libgdr.so`` is missing this module raises instead of computing anything.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr.so")

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_CUDA, GDR_ERR_DEVICE_INDEX, GDR_ERR_TIMEOUT = range(6)
GDR_F32, GDR_BF16 = 0, 1
D = 128

EXPORTS = ["gdr_chunk_workspace_bytes", "gdr_chunk_fwd", "gdr_chunk_fwd_varlen", "gdr_chunk_fwd_gated",
           "gdr_chunk_fwd_noalloc", "gdr_chunk_fwd_prologue_workspace_bytes", "gdr_chunk_fwd_prologue",
           "gdr_fork_workspace_bytes",
           "gdr_fork_fwd", "gdr_decode_step", "gdr_prologue", "gdr_gated_rmsnorm",
           "gdr_backward_workspace_bytes", "gdr_backward",
           "gdr_backward_chunked_workspace_bytes", "gdr_backward_chunked",
           "gdr_chunk_fwd_save", "gdr_backward_chunked_saved",
           "gdr_sync_status", "gdr_status_string", "gdr_last_error_message",
           "gdr_stage_timer_enable", "gdr_stage_timer_collect", "gdr_kernel_name", "gdr_debug_set_wait_budget"]


class GdrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libgdr.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "or python -m gated_deltanet_rule_gb300.build")
    L = ctypes.CDLL(LIB_PATH)
    vp, fp, i, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.gdr_chunk_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.gdr_chunk_workspace_bytes.restype = sz
    L.gdr_chunk_fwd.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, i, vp, sz, vp]
    L.gdr_chunk_fwd.restype = i
    L.gdr_chunk_fwd_varlen.argtypes = [vp, vp, vp, fp, fp, fp, vp, vp, fp, i, i, i, i, i, i, vp, sz, vp]
    L.gdr_chunk_fwd_varlen.restype = i
    L.gdr_chunk_fwd_gated.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, ctypes.c_float, vp, fp, i, i, i, i, i, i, vp, sz, vp]
    L.gdr_chunk_fwd_gated.restype = i
    L.gdr_chunk_fwd_noalloc.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, i, vp]
    L.gdr_chunk_fwd_noalloc.restype = i
    L.gdr_fork_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.gdr_fork_workspace_bytes.restype = sz
    L.gdr_fork_fwd.argtypes = [vp, vp, vp, fp, fp, fp, vp, i, vp, fp, i, i, i, i, i, i, vp, sz, vp]
    L.gdr_fork_fwd.restype = i
    L.gdr_decode_step.argtypes = [vp, vp, vp, fp, fp, fp, vp, i, i, i, i, i, vp]
    L.gdr_decode_step.restype = i
    L.gdr_prologue.argtypes = [vp, vp, fp, fp, fp, fp, fp, vp, vp, vp, vp, fp, fp, vp, i, i, i, i, i, i, vp]
    L.gdr_prologue.restype = i
    L.gdr_chunk_fwd_prologue_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.gdr_chunk_fwd_prologue_workspace_bytes.restype = sz
    L.gdr_chunk_fwd_prologue.argtypes = [vp, vp, fp, fp, fp, fp, fp, fp, vp, fp, vp, i, i, i, i, i, i, vp, sz, vp]
    L.gdr_chunk_fwd_prologue.restype = i
    L.gdr_gated_rmsnorm.argtypes = [vp, vp, fp, ctypes.c_float, vp, ctypes.c_longlong, i, vp]
    L.gdr_gated_rmsnorm.restype = i
    L.gdr_backward_workspace_bytes.argtypes = [i, i, i, i, i]
    L.gdr_backward_workspace_bytes.restype = sz
    L.gdr_backward.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, i, vp, sz, vp]
    L.gdr_backward.restype = i
    L.gdr_backward_chunked_workspace_bytes.argtypes = [i, i, i, i, i]
    L.gdr_backward_chunked_workspace_bytes.restype = sz
    L.gdr_backward_chunked.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, i, vp, sz,
                                       vp]
    L.gdr_backward_chunked.restype = i
    L.gdr_backward_chunked_saved.argtypes = L.gdr_backward_chunked.argtypes
    L.gdr_backward_chunked_saved.restype = i
    L.gdr_chunk_fwd_save.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, i, vp, sz, vp]
    L.gdr_chunk_fwd_save.restype = i
    L.gdr_sync_status.argtypes = [vp]
    L.gdr_sync_status.restype = i
    L.gdr_status_string.argtypes = [i]
    L.gdr_status_string.restype = ctypes.c_char_p
    L.gdr_last_error_message.argtypes = []
    L.gdr_last_error_message.restype = ctypes.c_char_p
    L.gdr_stage_timer_enable.argtypes = [i, i]
    L.gdr_stage_timer_enable.restype = i
    L.gdr_stage_timer_collect.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int), i]
    L.gdr_stage_timer_collect.restype = i
    L.gdr_debug_set_wait_budget.argtypes = [ctypes.c_longlong]
    L.gdr_debug_set_wait_budget.restype = i
    L.gdr_kernel_name.argtypes = [i]
    L.gdr_kernel_name.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int) -> None:
    if status != GDR_OK:
        L = lib()
        name = L.gdr_status_string(status).decode()
        msg = L.gdr_last_error_message().decode()
        raise GdrError(status, f"{name}: {msg}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GDR_F32
    if t.dtype == torch.bfloat16:
        return GDR_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _check_inputs(q, k, v, g, beta, device_check=True):
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _need(isinstance(t, torch.Tensor), f"{name} must be a tensor")
        if device_check:
            _need(t.is_cuda, f"{name} must be a CUDA tensor")
        _need(t.is_contiguous(), f"{name} must be contiguous")
    _need(q.dtype == k.dtype == v.dtype, "q, k, v must share one dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g and beta must be float32")
    _need(q.dim() == 4 and k.shape == q.shape and v.dim() == 4, "q, k [B,L,Hk,D] and v [B,L,Hv,D]")
    B, L, Hk, Dk = q.shape
    _need(v.shape[0] == B and v.shape[1] == L, "v must be [B, L, Hv, D]")
    Hv = v.shape[2]
    _need(g.shape == (B, L, Hv) and beta.shape == (B, L, Hv), "g and beta must be [B, L, Hv]")
    return B, L, Hk, Hv, Dk


def workspace_bytes(B: int, L: int, Hk: int, Hv: int, D: int = D, dtype=torch.bfloat16) -> int:
    code = GDR_BF16 if dtype == torch.bfloat16 else GDR_F32
    return int(lib().gdr_chunk_workspace_bytes(B, L, Hk, Hv, D, code))


def gdr_chunk_fwd(q, k, v, g, beta, S0=None, o=None, S_T=None, ws=None, stream=None,
                  final_state: bool = True, lengths=None):
    """Prefill of B rows: returns (o [B,L,Hv,D] in v's dtype, S_T [B,Hv,D,D] float32 or None).

    lengths: optional CUDA int32 [B], each row's valid tokens (gdr_chunk_fwd_varlen): positions past
    a row's length are pads, not run, and their o is left as it was (pass o to control it)."""
    B, L, Hk, Hv, Dk = _check_inputs(q, k, v, g, beta)
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty_like(v)
    if S_T is None and final_state:
        S_T = torch.empty(B, Hv, Dk, v.shape[3], device=v.device, dtype=torch.float32)
    for name, t in (("S0", S0), ("S_T", S_T)):
        if t is not None:
            _need(t.dtype == torch.float32 and t.is_contiguous() and t.is_cuda, f"{name} must be contiguous CUDA float32")
    need = workspace_bytes(B, L, Hk, Hv, Dk, q.dtype)
    if need and ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    if lengths is None:
        _check(lib().gdr_chunk_fwd(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(o), _p(S_T),
                                   B, L, Hk, Hv, Dk, dt, _p(ws), ws_bytes, _stream(stream)))
    else:
        _need(lengths.is_cuda and lengths.dtype == torch.int32 and lengths.shape == (B,) and lengths.is_contiguous(),
              "lengths must be a contiguous CUDA int32 tensor of shape [B]")
        _check(lib().gdr_chunk_fwd_varlen(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(lengths), _p(o),
                                          _p(S_T), B, L, Hk, Hv, Dk, dt, _p(ws), ws_bytes, _stream(stream)))
    return o, S_T


def gdr_chunk_fwd_gated(q, k, v, g, beta, S0, z, w, eps: float, out=None, S_T=None, ws=None, stream=None,
                        final_state: bool = True):
    """Prefill with the gated RMSNorm fused into its output: returns (out [B,L,Hv,D] bf16 =
    w * o / rms(o) * silu(z), S_T [B,Hv,D,D] float32 or None)."""
    B, L, Hk, Hv, Dk = _check_inputs(q, k, v, g, beta)
    dt = _dtype_code(q)
    _need(z.is_cuda and z.dtype == torch.bfloat16 and z.shape == v.shape and z.is_contiguous(), "z: contiguous CUDA bf16 like v")
    _need(w.is_cuda and w.dtype == torch.float32 and w.shape == (Dk,) and w.is_contiguous(), "w: contiguous CUDA float32 [D]")
    if out is None:
        out = torch.empty_like(v)
    if S_T is None and final_state:
        S_T = torch.empty(B, Hv, Dk, v.shape[3], device=v.device, dtype=torch.float32)
    need = workspace_bytes(B, L, Hk, Hv, Dk, q.dtype)
    if need and ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().gdr_chunk_fwd_gated(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(z), _p(w), float(eps), _p(out),
                                     _p(S_T), B, L, Hk, Hv, Dk, dt, _p(ws), ws_bytes, _stream(stream)))
    return out, S_T


def fork_workspace_bytes(F: int, L_pad: int, Hk: int, Hv: int, D: int = D, dtype=torch.bfloat16) -> int:
    code = GDR_BF16 if dtype == torch.bfloat16 else GDR_F32
    return int(lib().gdr_fork_workspace_bytes(F, L_pad, Hk, Hv, D, code))


def gdr_fork_fwd(q, k, v, g, beta, trunk, trunk_idx, o=None, states_out=None, stream=None,
                 keep: bool = True, ws=None):
    """Fork batch: returns (o [F,L_pad,Hv,D], states_out [F,Hv,D,D] or None)."""
    F, L, Hk, Hv, Dk = _check_inputs(q, k, v, g, beta)
    dt = _dtype_code(q)
    _need(trunk.is_cuda and trunk.dtype == torch.float32 and trunk.is_contiguous(), "trunk: CUDA float32")
    _need(trunk_idx.is_cuda and trunk_idx.dtype == torch.int64 and trunk_idx.shape == (F,), "trunk_idx: CUDA int64 [F]")
    if o is None:
        o = torch.empty_like(v)
    if states_out is None and keep:
        states_out = torch.empty(F, Hv, Dk, v.shape[3], device=v.device, dtype=torch.float32)
    need = fork_workspace_bytes(F, L, Hk, Hv, Dk, q.dtype)
    if need and ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().gdr_fork_fwd(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(trunk), _p(trunk_idx),
                              trunk.shape[0], _p(o), _p(states_out), F, L, Hk, Hv, Dk, dt,
                              _p(ws), ws_bytes, _stream(stream)))
    return o, states_out


def gdr_decode_step(q, k, v, g, beta, states, o=None, stream=None):
    """One token per row; ``states`` [F,Hv,D,D] float32 is updated in place. Returns o [F,1,Hv,D]."""
    F, L, Hk, Hv, Dk = _check_inputs(q, k, v, g, beta)
    _need(L == 1, "decode takes one token per row")
    dt = _dtype_code(q)
    _need(states.is_cuda and states.dtype == torch.float32 and states.is_contiguous(), "states: CUDA float32")
    if o is None:
        o = torch.empty_like(v)
    _check(lib().gdr_decode_step(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(states), _p(o),
                                 F, Hk, Hv, Dk, dt, _stream(stream)))
    return o


def gdr_prologue(mixed, conv_w, a, b, A_log, dt_bias, Hk: int, Hv: int, tail=None, lengths=None,
                 q=None, k=None, v=None, g=None, beta=None, new_tail=None, stream=None,
                 keep_tail: bool = True):
    """GDN prologue: conv + SiLU of ``mixed`` [B,L,C] bf16 (with the carry ``tail`` [B,K-1,C]),
    gates from ``a``, ``b`` [B,L,Hv]. Returns (q, k, v, g, beta, new_tail or None)."""
    for name, t in (("mixed", mixed), ("conv_w", conv_w), ("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias)):
        _need(isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(mixed.dtype == torch.bfloat16 and mixed.dim() == 3, "mixed must be bfloat16 [B, L, C]")
    B, L, C = mixed.shape
    _need(C == (2 * Hk + Hv) * D, f"mixed has {C} channels, expected (2 Hk + Hv) D = {(2 * Hk + Hv) * D}")
    _need(conv_w.dtype == torch.float32 and conv_w.dim() == 2 and conv_w.shape[0] == C, "conv_w must be float32 [C, K]")
    K = conv_w.shape[1]
    for name, t in (("a", a), ("b", b)):
        _need(t.dtype == torch.float32 and t.shape == (B, L, Hv), f"{name} must be float32 [B, L, Hv]")
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias)):
        _need(t.dtype == torch.float32 and t.shape == (Hv,), f"{name} must be float32 [Hv]")
    if tail is not None:
        _need(tail.is_cuda and tail.is_contiguous() and tail.dtype == torch.bfloat16 and tail.shape == (B, K - 1, C),
              "tail must be contiguous CUDA bfloat16 [B, K-1, C]")
    if lengths is not None:
        _need(lengths.is_cuda and lengths.dtype == torch.int32 and lengths.shape == (B,), "lengths must be CUDA int32 [B]")
    dev = mixed.device
    if q is None:
        q = torch.empty(B, L, Hk, D, device=dev, dtype=torch.bfloat16)
    if k is None:
        k = torch.empty(B, L, Hk, D, device=dev, dtype=torch.bfloat16)
    if v is None:
        v = torch.empty(B, L, Hv, D, device=dev, dtype=torch.bfloat16)
    if g is None:
        g = torch.empty(B, L, Hv, device=dev, dtype=torch.float32)
    if beta is None:
        beta = torch.empty(B, L, Hv, device=dev, dtype=torch.float32)
    if new_tail is None and keep_tail and K > 1:
        new_tail = torch.empty(B, K - 1, C, device=dev, dtype=torch.bfloat16)
    _check(lib().gdr_prologue(_p(mixed), _p(tail), _p(conv_w), _p(a), _p(b), _p(A_log), _p(dt_bias), _p(lengths),
                              _p(q), _p(k), _p(v), _p(g), _p(beta), _p(new_tail), B, L, Hk, Hv, D, K,
                              _stream(stream)))
    return q, k, v, g, beta, new_tail


def prologue_workspace_bytes(B: int, L: int, Hk: int, Hv: int, K: int = 4, D: int = D) -> int:
    return int(lib().gdr_chunk_fwd_prologue_workspace_bytes(B, L, Hk, Hv, D, K))


def gdr_chunk_fwd_prologue(mixed, conv_w, a, b, A_log, dt_bias, Hk: int, Hv: int, S0=None, tail=None,
                           o=None, S_T=None, new_tail=None, ws=None, stream=None, final_state: bool = True,
                           keep_tail: bool = True):
    """The GDN prologue fused into the bf16 prefill: gdr_prologue(mixed, ...) then gdr_chunk_fwd on its
    outputs, in one pass. Returns (o [B,L,Hv,D] bf16, S_T [B,Hv,D,D] float32 or None, new_tail
    [B,3,C] bf16 or None)."""
    for name, t in (("mixed", mixed), ("conv_w", conv_w), ("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias)):
        _need(isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(mixed.dtype == torch.bfloat16 and mixed.dim() == 3, "mixed must be bfloat16 [B, L, C]")
    B, L, C = mixed.shape
    _need(C == (2 * Hk + Hv) * D, f"mixed has {C} channels, expected (2 Hk + Hv) D = {(2 * Hk + Hv) * D}")
    _need(conv_w.dtype == torch.float32 and conv_w.dim() == 2 and conv_w.shape[0] == C, "conv_w must be float32 [C, K]")
    K = conv_w.shape[1]
    for name, t in (("a", a), ("b", b)):
        _need(t.dtype == torch.float32 and t.shape == (B, L, Hv), f"{name} must be float32 [B, L, Hv]")
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias)):
        _need(t.dtype == torch.float32 and t.shape == (Hv,), f"{name} must be float32 [Hv]")
    if tail is not None:
        _need(tail.is_cuda and tail.is_contiguous() and tail.dtype == torch.bfloat16 and tail.shape == (B, K - 1, C),
              "tail must be contiguous CUDA bfloat16 [B, K-1, C]")
    for name, t in (("S0", S0), ("S_T", S_T)):
        if t is not None:
            _need(t.dtype == torch.float32 and t.is_contiguous() and t.is_cuda and t.shape == (B, Hv, D, D),
                  f"{name} must be contiguous CUDA float32 [B, Hv, D, D]")
    dev = mixed.device
    if o is None:
        o = torch.empty(B, L, Hv, D, device=dev, dtype=torch.bfloat16)
    if S_T is None and final_state:
        S_T = torch.empty(B, Hv, D, D, device=dev, dtype=torch.float32)
    if new_tail is None and keep_tail and K > 1:
        new_tail = torch.empty(B, K - 1, C, device=dev, dtype=torch.bfloat16)
    need = prologue_workspace_bytes(B, L, Hk, Hv, K)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().gdr_chunk_fwd_prologue(_p(mixed), _p(tail), _p(conv_w), _p(a), _p(b), _p(A_log), _p(dt_bias),
                                        _p(S0), _p(o), _p(S_T), _p(new_tail), B, L, Hk, Hv, D, K, _p(ws), ws_bytes,
                                        _stream(stream)))
    return o, S_T, new_tail


def gdr_gated_rmsnorm(x, z, w, eps: float = 1e-6, out=None, stream=None):
    """Gated RMSNorm over the last dimension (D = 128) of ``x`` with gate ``z`` (both bf16, same
    shape, e.g. o [B, L, Hv, D]) and weight ``w`` [D] float32; returns ``out`` (x's shape, bf16)."""
    for name, t in (("x", x), ("z", z), ("w", w)):
        _need(isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(x.dtype == torch.bfloat16 and z.dtype == torch.bfloat16 and z.shape == x.shape, "x and z: bfloat16, same shape")
    _need(w.dtype == torch.float32 and w.shape == (x.shape[-1],), "w must be float32 [D]")
    if out is None:
        out = torch.empty_like(x)
    rows = x.numel() // x.shape[-1]
    _check(lib().gdr_gated_rmsnorm(_p(x), _p(z), _p(w), float(eps), _p(out), rows, x.shape[-1], _stream(stream)))
    return out


def backward_workspace_bytes(B: int, L: int, Hk: int, Hv: int, D: int = D) -> int:
    return int(lib().gdr_backward_workspace_bytes(B, L, Hk, Hv, D))


def gdr_backward(q, k, v, g, beta, S0, dO, dS_T=None, ws=None, stream=None, want_dS0: bool = True):
    """Gradients of gdr_chunk_fwd: returns (dq, dk [B,L,Hk,D], dv [B,L,Hv,D], dg, dbeta [B,L,Hv],
    dS0 [B,Hv,D,D] or None), all float32, given dO (o's shape, q's dtype) and dS_T (None = 0)."""
    B, L, Hk, Hv, Dk = _check_inputs(q, k, v, g, beta)
    dt = _dtype_code(q)
    _need(isinstance(dO, torch.Tensor) and dO.is_cuda and dO.is_contiguous() and dO.dtype == q.dtype
          and dO.shape == v.shape, "dO must be a contiguous CUDA tensor of v's shape and q's dtype")
    for name, t in (("S0", S0), ("dS_T", dS_T)):
        if t is not None:
            _need(t.dtype == torch.float32 and t.is_contiguous() and t.is_cuda and t.shape == (B, Hv, Dk, v.shape[3]),
                  f"{name} must be contiguous CUDA float32 [B, Hv, D, D]")
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty(q.shape, **f32)
    dk = torch.empty(k.shape, **f32)
    dv = torch.empty(v.shape, **f32)
    dg = torch.empty(g.shape, **f32)
    dbeta = torch.empty(beta.shape, **f32)
    dS0 = torch.empty(B, Hv, Dk, v.shape[3], **f32) if want_dS0 else None
    need = backward_workspace_bytes(B, L, Hk, Hv, Dk)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = ws.numel() * ws.element_size()
    _check(lib().gdr_backward(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(dO), _p(dS_T), _p(dq), _p(dk),
                              _p(dv), _p(dg), _p(dbeta), _p(dS0), B, L, Hk, Hv, Dk, dt, _p(ws), ws_bytes,
                              _stream(stream)))
    return dq, dk, dv, dg, dbeta, dS0


def backward_chunked_workspace_bytes(B: int, L: int, Hk: int, Hv: int, D: int = 128) -> int:
    return int(lib().gdr_backward_chunked_workspace_bytes(B, L, Hk, Hv, D))


def gdr_chunk_fwd_save(q, k, v, g, beta, S0=None, saved=None, o=None, S_T=None, stream=None,
                       final_state: bool = True):
    """gdr_chunk_fwd for bf16 rows that also keeps, in ``saved`` (a uint8 CUDA buffer of
    backward_chunked_workspace_bytes; allocated if None), what gdr_backward_chunked would recompute.
    Returns (o, S_T or None, saved); pass saved to gdr_backward_chunked(..., saved=saved)."""
    B, L, Hk, Hv, Dk = _check_inputs(q, k, v, g, beta)
    _need(q.dtype == torch.bfloat16, "gdr_chunk_fwd_save takes bf16 q, k, v")
    if o is None:
        o = torch.empty_like(v)
    if S_T is None and final_state:
        S_T = torch.empty(B, Hv, Dk, v.shape[3], device=v.device, dtype=torch.float32)
    for name, t in (("S0", S0), ("S_T", S_T)):
        if t is not None:
            _need(t.dtype == torch.float32 and t.is_contiguous() and t.is_cuda, f"{name} must be contiguous CUDA float32")
    need = backward_chunked_workspace_bytes(B, L, Hk, Hv, Dk)
    if saved is None:
        saved = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(lib().gdr_chunk_fwd_save(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(o), _p(S_T), B, L, Hk, Hv, Dk,
                                    _dtype_code(q), _p(saved), saved.numel() * saved.element_size(), _stream(stream)))
    return o, S_T, saved


def gdr_backward_chunked(q, k, v, g, beta, S0, dO, dS_T=None, ws=None, stream=None, want_dS0: bool = True,
                         saved=None):
    """gdr_backward's gradients for bf16 q, k, v, dO, computed chunk by chunk on the tensor cores
    (bf16-path accuracy); same arguments and results. With ``saved`` (the buffer gdr_chunk_fwd_save
    filled on the same q, k, v, g, beta, S0) the forward passes are not run again
    (gdr_backward_chunked_saved)."""
    B, L, Hk, Hv, Dk = _check_inputs(q, k, v, g, beta)
    _need(q.dtype == torch.bfloat16, "gdr_backward_chunked takes bf16 q, k, v, dO (float32: gdr_backward)")
    _need(isinstance(dO, torch.Tensor) and dO.is_cuda and dO.is_contiguous() and dO.dtype == q.dtype
          and dO.shape == v.shape, "dO must be a contiguous CUDA tensor of v's shape and q's dtype")
    for name, t in (("S0", S0), ("dS_T", dS_T)):
        if t is not None:
            _need(t.dtype == torch.float32 and t.is_contiguous() and t.is_cuda and t.shape == (B, Hv, Dk, v.shape[3]),
                  f"{name} must be contiguous CUDA float32 [B, Hv, D, D]")
    f32 = dict(dtype=torch.float32, device=q.device)
    dq = torch.empty(q.shape, **f32)
    dk = torch.empty(k.shape, **f32)
    dv = torch.empty(v.shape, **f32)
    dg = torch.empty(g.shape, **f32)
    dbeta = torch.empty(beta.shape, **f32)
    dS0 = torch.empty(B, Hv, Dk, v.shape[3], **f32) if want_dS0 else None
    need = backward_chunked_workspace_bytes(B, L, Hk, Hv, Dk)
    if saved is not None:
        _need(ws is None, "pass either ws or saved")
        ws = saved
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = ws.numel() * ws.element_size()
    fn = lib().gdr_backward_chunked_saved if saved is not None else lib().gdr_backward_chunked
    _check(fn(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0), _p(dO), _p(dS_T), _p(dq), _p(dk), _p(dv), _p(dg),
              _p(dbeta), _p(dS0), B, L, Hk, Hv, Dk, _dtype_code(q), _p(ws), ws_bytes, _stream(stream)))
    return dq, dk, dv, dg, dbeta, dS0


def gdr_sync_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    _check(lib().gdr_sync_status(_stream(stream)))


def kernel_names() -> list[str]:
    names, i = [], 0
    while True:
        n = lib().gdr_kernel_name(i)
        if n is None:
            return names
        names.append(n.decode())
        i += 1


def debug_set_wait_budget(cycles: int) -> None:
    """Testing aid: cycles a kernel wait may take before it gives up (0: at once; < 0: default)."""
    _check(lib().gdr_debug_set_wait_budget(int(cycles)))


def stage_timer_enable(on: bool = True, capacity: int = 8192) -> None:
    _check(lib().gdr_stage_timer_enable(int(on), int(capacity)))


def stage_timer_collect() -> dict:
    """{kernel name: (total ms, launches)} for the launches recorded since the last collect."""
    names = kernel_names()
    n = len(names)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    _check(lib().gdr_stage_timer_collect(ms, cnt, n))
    return {names[i]: (ms[i], cnt[i]) for i in range(n)}
