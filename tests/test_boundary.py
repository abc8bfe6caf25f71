"""The C ABI without a GPU: the library loads, exports every function include/gdr.h declares, and
rejects bad arguments on the host (status codes and messages) before touching CUDA."""
import ctypes
import os
import re

import pytest

from gated_deltanet_rule_gb300 import build as gbuild
from gated_deltanet_rule_gb300 import gdr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdr.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "gdr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert "gdr_chunk_fwd" in declared and "gdr_fork_fwd" in declared and "gdr_decode_step" in declared
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(gdr.EXPORTS) == declared


def test_status_strings(L):
    for code, name in enumerate(["GDR_OK", "GDR_ERR_INVALID_ARG", "GDR_ERR_UNSUPPORTED", "GDR_ERR_CUDA",
                                 "GDR_ERR_DEVICE_INDEX", "GDR_ERR_TIMEOUT"]):
        assert L.gdr_status_string(code).decode() == name
    assert gdr.kernel_names()[0] == "gdr_recurrent"


P = ctypes.c_void_p(1 << 20)       # a 16-byte aligned address; never dereferenced on the host
BAD = ctypes.c_void_p((1 << 20) + 4)


def _chunk(L, q=P, g=P, o=P, S0=None, B=1, Lt=64, Hk=16, Hv=32, D=128, dt=1, ws=None, ws_bytes=0):
    return L.gdr_chunk_fwd(q, P, P, g, P, S0, o, None, B, Lt, Hk, Hv, D, dt, ws, ws_bytes, None)


def test_chunk_rejects_bad_arguments(L):
    assert _chunk(L, q=None) == gdr.GDR_ERR_INVALID_ARG
    assert b"non-NULL" in L.gdr_last_error_message()
    assert _chunk(L, Lt=0) == gdr.GDR_ERR_INVALID_ARG
    assert _chunk(L, B=0) == gdr.GDR_ERR_INVALID_ARG
    assert _chunk(L, Hk=3, Hv=32) == gdr.GDR_ERR_INVALID_ARG
    assert b"multiple" in L.gdr_last_error_message()
    assert _chunk(L, D=64) == gdr.GDR_ERR_UNSUPPORTED
    assert _chunk(L, dt=7) == gdr.GDR_ERR_INVALID_ARG
    assert _chunk(L, q=BAD) == gdr.GDR_ERR_INVALID_ARG
    assert b"aligned" in L.gdr_last_error_message()
    assert _chunk(L, S0=BAD) == gdr.GDR_ERR_INVALID_ARG


def test_chunk_rejects_small_workspace(L):
    need = L.gdr_chunk_workspace_bytes(1, 4096, 16, 32, 128, 1)
    if need == 0:
        pytest.skip("this path needs no workspace")
    assert _chunk(L, Lt=4096, ws=P, ws_bytes=need - 1) == gdr.GDR_ERR_INVALID_ARG
    assert b"workspace" in L.gdr_last_error_message()
    assert _chunk(L, Lt=4096, ws=None, ws_bytes=need) == gdr.GDR_ERR_INVALID_ARG


def test_workspace_query(L):
    assert L.gdr_chunk_workspace_bytes(1, 64, 16, 32, 64, 1) == 0      # unsupported D
    assert L.gdr_chunk_workspace_bytes(1, 64, 3, 32, 128, 1) == 0      # bad head ratio
    assert L.gdr_chunk_workspace_bytes(1, 64, 16, 32, 128, 0) == 0     # float32 path needs none
    a = L.gdr_chunk_workspace_bytes(1, 4096, 16, 32, 128, 1)
    b = L.gdr_chunk_workspace_bytes(2, 4096, 16, 32, 128, 1)
    assert b >= a


def test_fork_rejects_bad_arguments(L):
    def fork(trunk=P, idx=P, N=1, states=None, F=4, ws=P, ws_bytes=1 << 40):
        return L.gdr_fork_fwd(P, P, P, P, P, trunk, idx, N, P, states, F, 64, 16, 32, 128, 1, ws, ws_bytes, None)
    assert fork(trunk=None) == gdr.GDR_ERR_INVALID_ARG
    assert fork(idx=None) == gdr.GDR_ERR_INVALID_ARG
    assert fork(N=0) == gdr.GDR_ERR_INVALID_ARG
    assert fork(idx=ctypes.c_void_p((1 << 20) + 4)) == gdr.GDR_ERR_INVALID_ARG
    # states_out overlapping the trunk is rejected
    assert fork(trunk=P, states=ctypes.c_void_p((1 << 20) + 1024)) == gdr.GDR_ERR_INVALID_ARG
    assert b"overlaps" in L.gdr_last_error_message()
    # bf16 forks run on the tensor-core kernels: single-chunk forks need no workspace, longer ones
    # need the caller's
    assert L.gdr_fork_workspace_bytes(4, 64, 16, 32, 128, 1) == 0
    need = L.gdr_fork_workspace_bytes(4, 128, 16, 32, 128, 1)
    assert need == L.gdr_chunk_workspace_bytes(4, 128, 16, 32, 128, 1) > 0
    assert L.gdr_fork_workspace_bytes(4, 128, 16, 32, 128, 0) == 0

    def fork128(ws, ws_bytes):
        return L.gdr_fork_fwd(P, P, P, P, P, P, P, 1, P, None, 4, 128, 16, 32, 128, 1, ws, ws_bytes, None)
    assert fork128(None, 0) == gdr.GDR_ERR_INVALID_ARG
    assert b"workspace" in L.gdr_last_error_message()
    assert fork128(P, need - 1) == gdr.GDR_ERR_INVALID_ARG


def test_decode_rejects_bad_arguments(L):
    assert L.gdr_decode_step(P, P, P, P, P, None, P, 4, 16, 32, 128, 1, None) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_decode_step(P, P, P, P, P, P, P, 4, 16, 32, 100, 1, None) == gdr.GDR_ERR_UNSUPPORTED
    assert L.gdr_decode_step(P, P, P, P, P, BAD, P, 4, 16, 32, 128, 1, None) == gdr.GDR_ERR_INVALID_ARG


def test_stage_timer_argument_checks(L):
    assert L.gdr_stage_timer_enable(1, 0) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_stage_timer_enable(0, 0) == gdr.GDR_OK
    assert L.gdr_stage_timer_collect(None, None, 0) == gdr.GDR_ERR_INVALID_ARG


def _prologue(L, mixed=P, tail=None, w=P, a=P, lengths=None, q=P, new_tail=None, B=1, Lt=64, Hk=16, Hv=32,
              D=128, K=4):
    return L.gdr_prologue(mixed, tail, w, a, P, P, P, lengths, q, P, P, P, P, new_tail, B, Lt, Hk, Hv, D, K, None)


def test_prologue_rejects_bad_arguments(L):
    assert _prologue(L, mixed=None) == gdr.GDR_ERR_INVALID_ARG
    assert b"non-NULL" in L.gdr_last_error_message()
    assert _prologue(L, q=None) == gdr.GDR_ERR_INVALID_ARG
    assert _prologue(L, Lt=0) == gdr.GDR_ERR_INVALID_ARG
    assert _prologue(L, Hk=3) == gdr.GDR_ERR_INVALID_ARG
    assert _prologue(L, K=0) == gdr.GDR_ERR_INVALID_ARG
    assert _prologue(L, K=9) == gdr.GDR_ERR_INVALID_ARG
    assert b"conv width" in L.gdr_last_error_message()
    assert _prologue(L, D=64) == gdr.GDR_ERR_UNSUPPORTED
    assert _prologue(L, mixed=BAD) == gdr.GDR_ERR_INVALID_ARG
    assert b"aligned" in L.gdr_last_error_message()
    assert _prologue(L, w=ctypes.c_void_p((1 << 20) + 2)) == gdr.GDR_ERR_INVALID_ARG
    # the carry is gathered from tail and mixed, so it may overlap neither
    assert _prologue(L, tail=P, new_tail=P) == gdr.GDR_ERR_INVALID_ARG
    assert b"overlap" in L.gdr_last_error_message()
    assert _prologue(L, new_tail=ctypes.c_void_p((1 << 20) + 4096)) == gdr.GDR_ERR_INVALID_ARG
    assert _prologue(L, Lt=16 * 65535 + 1) == gdr.GDR_ERR_UNSUPPORTED
    assert _prologue(L, B=65536) == gdr.GDR_ERR_UNSUPPORTED


def test_gated_rmsnorm_rejects_bad_arguments(L):
    f = L.gdr_gated_rmsnorm
    Q = ctypes.c_void_p((1 << 24))   # a second, distant aligned address
    assert f(None, P, P, 1e-6, Q, 4, 128, None) == gdr.GDR_ERR_INVALID_ARG
    assert f(P, P, P, 1e-6, Q, 0, 128, None) == gdr.GDR_ERR_INVALID_ARG
    assert f(P, P, P, 1e-6, Q, 4, 64, None) == gdr.GDR_ERR_UNSUPPORTED
    assert f(P, Q, P, 1e-6, P, (1 << 34) + 1, 128, None) == gdr.GDR_ERR_UNSUPPORTED
    assert f(P, P, P, -1.0, Q, 4, 128, None) == gdr.GDR_ERR_INVALID_ARG
    assert f(BAD, P, P, 1e-6, Q, 4, 128, None) == gdr.GDR_ERR_INVALID_ARG
    assert b"aligned" in L.gdr_last_error_message()
    # out may be x itself, but not a shifted view of it
    assert f(P, Q, P, 1e-6, ctypes.c_void_p((1 << 20) + 256), 4, 128, None) == gdr.GDR_ERR_INVALID_ARG
    assert b"overlaps" in L.gdr_last_error_message()


def _bwd(L, q=P, dO=P, dq=P, dg=P, S0=None, dS0=None, B=1, Lt=64, Hk=2, Hv=4, D=128, dt=1, ws=P, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = L.gdr_backward_workspace_bytes(B, Lt, Hk, Hv, 128)
    return L.gdr_backward(q, P, P, P, P, S0, dO, None, dq, P, P, dg, P, dS0, B, Lt, Hk, Hv, D, dt, ws, ws_bytes, None)


def test_backward_rejects_bad_arguments(L):
    assert _bwd(L, dO=None) == gdr.GDR_ERR_INVALID_ARG
    assert b"dO" in L.gdr_last_error_message()
    assert _bwd(L, q=None) == gdr.GDR_ERR_INVALID_ARG
    assert _bwd(L, dq=None) == gdr.GDR_ERR_INVALID_ARG
    assert b"dq" in L.gdr_last_error_message()
    assert _bwd(L, Hk=3, Hv=4) == gdr.GDR_ERR_INVALID_ARG
    assert _bwd(L, D=64) == gdr.GDR_ERR_UNSUPPORTED
    assert _bwd(L, dt=5) == gdr.GDR_ERR_INVALID_ARG
    assert _bwd(L, dg=BAD) == gdr.GDR_ERR_INVALID_ARG
    assert b"aligned" in L.gdr_last_error_message()
    assert _bwd(L, dS0=BAD) == gdr.GDR_ERR_INVALID_ARG
    assert _bwd(L, B=65536, ws_bytes=1 << 62) == gdr.GDR_ERR_UNSUPPORTED
    assert _bwd(L, B=2, Lt=1 << 30, ws_bytes=1 << 62) == gdr.GDR_ERR_UNSUPPORTED
    need = L.gdr_backward_workspace_bytes(1, 64, 2, 4, 128)
    assert _bwd(L, ws_bytes=need - 1) == gdr.GDR_ERR_INVALID_ARG
    assert b"workspace" in L.gdr_last_error_message()
    assert _bwd(L, ws=None) == gdr.GDR_ERR_INVALID_ARG


def test_backward_workspace_query(L):
    assert L.gdr_backward_workspace_bytes(1, 64, 2, 4, 64) == 0
    assert L.gdr_backward_workspace_bytes(1, 64, 3, 4, 128) == 0
    assert L.gdr_backward_workspace_bytes(0, 64, 2, 4, 128) == 0
    # checkpoints (ceil(L/32) slices) + one segment (32 slices) per (row, value head, column block),
    # 8 column blocks of 16 value columns, a slice being 128 x 16 floats; then the partials:
    # 8 column blocks x (2 D + 2) floats per token and value head
    for B, Lt, Hv in ((1, 64, 4), (2, 70, 8), (1, 4096, 32)):
        n_seg = -(-Lt // 32)
        want = 4 * (8 * B * Hv * (n_seg + 32) * 128 * 16 + B * Lt * Hv * 8 * (2 * 128 + 2))
        assert L.gdr_backward_workspace_bytes(B, Lt, 2, Hv, 128) == want


def test_backward_rejects_overlapping_outputs(L):
    """Outputs that overlap each other, the workspace or an input are refused before any CUDA call
    (each case below overlaps exactly one pair; every other pointer is far from the rest)."""
    B, Lt, Hk, Hv = 1, 64, 2, 4
    need = L.gdr_backward_workspace_bytes(B, Lt, Hk, Hv, 128)
    base = {n: ctypes.c_void_p((i + 1) << 32) for i, n in enumerate(
        ["q", "k", "v", "g", "beta", "S0", "dO", "dS_T", "dq", "dk", "dv", "dg", "dbeta", "dS0", "ws"])}

    def call(**over):
        p = dict(base, **{n: ctypes.c_void_p(v) for n, v in over.items()})
        return L.gdr_backward(p["q"], p["k"], p["v"], p["g"], p["beta"], p["S0"], p["dO"], p["dS_T"], p["dq"],
                              p["dk"], p["dv"], p["dg"], p["dbeta"], p["dS0"], B, Lt, Hk, Hv, 128, 1, p["ws"],
                              need, None)

    cases = [dict(dv=base["dq"].value + 256),          # two outputs
             dict(ws=base["dg"].value + 16),           # an output and the workspace
             dict(dq=base["q"].value + 4096),          # an output and an input
             dict(dS0=base["S0"].value),               # the state gradient over the initial state
             dict(dbeta=base["dO"].value + 1024)]
    for over in cases:
        assert call(**over) == gdr.GDR_ERR_INVALID_ARG, over
        assert b"overlaps" in L.gdr_last_error_message(), over


def test_varlen_and_gated_reject_bad_arguments(L):
    """The variable-length and gated prefill calls check their extra arguments on the host."""
    B, Lt, Hk, Hv = 1, 64, 2, 4
    # gdr_chunk_fwd_varlen(q, k, v, g, beta, S0, lengths, o, S_T, B, L, Hk, Hv, D, dt, ws, ws_bytes, stream)
    f = L.gdr_chunk_fwd_varlen
    assert f(P, P, P, P, P, None, None, P, None, B, Lt, Hk, Hv, 128, 1, None, 0, None) == gdr.GDR_ERR_INVALID_ARG
    assert b"lengths" in L.gdr_last_error_message()
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert f(P, P, P, P, P, None, odd, P, None, B, Lt, Hk, Hv, 128, 1, None, 0, None) == gdr.GDR_ERR_INVALID_ARG
    assert b"aligned" in L.gdr_last_error_message()
    # gdr_chunk_fwd_gated(q, k, v, g, beta, S0, z, w, eps, out, S_T, B, L, Hk, Hv, D, dt, ws, ws_bytes, stream)
    f = L.gdr_chunk_fwd_gated
    Z = ctypes.c_void_p(1 << 32)
    assert f(P, P, P, P, P, None, None, P, 1e-6, P, None, B, Lt, Hk, Hv, 128, 1, None, 0, None) == gdr.GDR_ERR_INVALID_ARG
    assert f(P, P, P, P, P, None, Z, P, 1e-6, P, None, B, Lt, Hk, Hv, 128, 0, None, 0, None) == gdr.GDR_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, None, Z, P, -1.0, P, None, B, Lt, Hk, Hv, 128, 1, None, 0, None) == gdr.GDR_ERR_INVALID_ARG
    assert f(P, P, P, P, P, None, Z, P, 1e-6, ctypes.c_void_p((1 << 32) + 4096), None, B, Lt, Hk, Hv, 128, 1, None, 0,
             None) == gdr.GDR_ERR_INVALID_ARG
    assert b"overlaps" in L.gdr_last_error_message()


def test_chunked_backward_rejects_bad_arguments_and_sizes_its_workspace(L):
    """gdr_backward_chunked: bf16 only, the backward's host checks, and a workspace of the forward's
    chunk factors plus the chunk-entry states and adjoints (fp16 with one scale per 32-column slice)."""
    f = L.gdr_backward_chunked
    need = L.gdr_backward_chunked_workspace_bytes(1, 64, 2, 4, 128)
    args = lambda dt=1, dO=P, ws_bytes=need, dq=P: (P, P, P, P, P, None, dO, None, dq, P, P, P, P, None, 1, 64, 2,
                                                     4, 128, dt, P, ws_bytes, None)
    assert f(*args(dt=0)) == gdr.GDR_ERR_UNSUPPORTED
    assert b"bf16" in L.gdr_last_error_message()
    assert f(*args(dO=None)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(dq=None)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(ws_bytes=need - 1)) == gdr.GDR_ERR_INVALID_ARG
    assert b"workspace" in L.gdr_last_error_message()
    assert L.gdr_backward_chunked_workspace_bytes(1, 64, 3, 4, 128) == 0
    for B, Lt, Hv in ((1, 64, 4), (2, 130, 8), (1, 4096, 32)):
        NC = -(-Lt // 64)
        units = B * Hv * NC * 98816 + 1024
        a256 = lambda x: -(-x // 256) * 256
        want = (a256(units) + 2 * a256(B * Hv * NC * 128 * 128 * 2) + 2 * a256(B * Hv * NC * 4 * 4)
                + a256(B * Hv * NC * 8 * 4))
        assert L.gdr_backward_chunked_workspace_bytes(B, Lt, 2, Hv, 128) == want


def test_fused_prologue_rejects_bad_arguments_and_sizes_its_workspace(L):
    """gdr_chunk_fwd_prologue: the prologue's and the prefill's host checks, a 4-tap conv only, o and
    new_tail clear of the inputs, and a workspace of the per-chunk factors for every L (rows of one
    chunk included: with the prologue fused they go through the two-kernel path)."""
    f = L.gdr_chunk_fwd_prologue
    need = L.gdr_chunk_fwd_prologue_workspace_bytes(1, 64, 2, 4, 128, 4)
    assert need == 1 * 4 * 1 * 98816 + 1024
    O = ctypes.c_void_p(1 << 30)   # an output far from P's inputs

    def args(mixed=P, conv_w=P, a=P, o=O, new_tail=None, tail=None, B=1, Lt=64, Hk=2, Hv=4, D=128, K=4,
             ws=P, ws_bytes=need):
        return (mixed, tail, conv_w, a, P, P, P, None, o, None, new_tail, B, Lt, Hk, Hv, D, K, ws, ws_bytes, None)

    assert f(*args(mixed=None)) == gdr.GDR_ERR_INVALID_ARG
    assert b"non-NULL" in L.gdr_last_error_message()
    assert f(*args(o=None)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(Lt=0)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(Hk=3)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(K=9)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(K=3)) == gdr.GDR_ERR_UNSUPPORTED
    assert b"4-tap" in L.gdr_last_error_message()
    assert f(*args(D=64)) == gdr.GDR_ERR_UNSUPPORTED
    assert f(*args(B=65536)) == gdr.GDR_ERR_UNSUPPORTED
    assert f(*args(mixed=BAD)) == gdr.GDR_ERR_INVALID_ARG
    assert b"aligned" in L.gdr_last_error_message()
    assert f(*args(conv_w=BAD)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(a=ctypes.c_void_p((1 << 20) + 2))) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(o=P)) == gdr.GDR_ERR_INVALID_ARG
    assert b"overlap" in L.gdr_last_error_message()
    assert f(*args(new_tail=ctypes.c_void_p((1 << 20) + 4096))) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(tail=ctypes.c_void_p(1 << 31), new_tail=ctypes.c_void_p((1 << 31) + 1024))) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(ws_bytes=need - 1)) == gdr.GDR_ERR_INVALID_ARG
    assert b"workspace" in L.gdr_last_error_message()
    assert f(*args(ws=None)) == gdr.GDR_ERR_INVALID_ARG
    assert L.gdr_chunk_fwd_prologue_workspace_bytes(1, 64, 2, 4, 128, 3) == 0
    assert L.gdr_chunk_fwd_prologue_workspace_bytes(1, 64, 3, 4, 128, 4) == 0
    for B, Lt, Hv in ((1, 1, 4), (2, 130, 8), (1, 4096, 32)):
        NC = -(-Lt // 64)
        assert L.gdr_chunk_fwd_prologue_workspace_bytes(B, Lt, 2, Hv, 128, 4) == B * Hv * NC * 98816 + 1024
    # rows longer than one chunk take the prefill's own workspace
    assert L.gdr_chunk_fwd_prologue_workspace_bytes(1, 4096, 16, 32, 128, 4) == \
        L.gdr_chunk_workspace_bytes(1, 4096, 16, 32, 128, 1)


def test_saving_forward_and_saved_backward_reject_bad_arguments(L):
    """gdr_chunk_fwd_save: bf16 only, a saved buffer of the chunked backward's workspace size clear of
    every input and output; gdr_backward_chunked_saved: the chunked backward's checks."""
    f = L.gdr_chunk_fwd_save
    need = L.gdr_backward_chunked_workspace_bytes(1, 130, 2, 4, 128)
    W = ctypes.c_void_p(1 << 32)   # far from P
    args = lambda dt=1, saved=W, nbytes=need, o=P, q=P: (q, P, P, P, P, None, o, None, 1, 130, 2, 4, 128, dt, saved,
                                                        nbytes, None)
    assert f(*args(dt=0)) == gdr.GDR_ERR_UNSUPPORTED
    assert f(*args(q=None)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(saved=None)) == gdr.GDR_ERR_INVALID_ARG
    assert f(*args(nbytes=need - 1)) == gdr.GDR_ERR_INVALID_ARG
    assert b"saved" in L.gdr_last_error_message()
    assert f(*args(saved=P)) == gdr.GDR_ERR_INVALID_ARG
    assert b"overlaps" in L.gdr_last_error_message()
    assert f(*args(saved=BAD)) == gdr.GDR_ERR_INVALID_ARG
    b = L.gdr_backward_chunked_saved
    bargs = lambda dt=1, dO=P, nbytes=need: (P, P, P, P, P, None, dO, None, W, ctypes.c_void_p((1 << 32) + (1 << 28)),
                                             ctypes.c_void_p((1 << 32) + (2 << 28)), ctypes.c_void_p((1 << 32) + (3 << 28)),
                                             ctypes.c_void_p((1 << 32) + (4 << 28)), None, 1, 130, 2, 4, 128, dt,
                                             ctypes.c_void_p(1 << 34), nbytes, None)
    assert b(*bargs(dt=0)) == gdr.GDR_ERR_UNSUPPORTED
    assert b(*bargs(dO=None)) == gdr.GDR_ERR_INVALID_ARG
    assert b(*bargs(nbytes=need - 1)) == gdr.GDR_ERR_INVALID_ARG
