"""The C-ABI library loads, exports every symbol include/dfa.h declares, and
rejects bad arguments on the host before touching a GPU (CPU only)."""
import ctypes

import pytest

from long_context_causal_gb300 import dfa

lib = dfa.library()
A = 0x10000          # an aligned stand-in address: validation fails before any use
MIS = 0x10004        # not 16-byte aligned


def test_every_header_function_is_exported():
    names = dfa.header_functions()
    assert "dfa_attn_fwd" in names and "dfa_attn_bwd" in names
    assert "dfa_chunk_attn_fwd" in names and "dfa_merge_partials" in names
    for n in names:
        assert hasattr(lib, n), n


def chunk(**kw):
    a = dict(q=A, k=A, v=A, dt=dfa.DFA_BF16, B=1, H=2, Hkv=1, Lq=128, Lkv=128, D=128,
             qs=None, ks=None, qo=0, ko=0, causal=1, scale=0.1, O=A, lse=A, stream=None)
    a.update(kw)
    st = lib.dfa_chunk_attn_fwd(a["q"], a["k"], a["v"], a["dt"], a["B"], a["H"], a["Hkv"], a["Lq"],
                                a["Lkv"], a["D"], a["qs"], a["ks"], a["qo"], a["ko"], a["causal"],
                                a["scale"], a["O"], a["lse"], a["stream"])
    return st, lib.dfa_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), dfa.DFA_ERR_UNSUPPORTED),
    (dict(H=3, Hkv=2), dfa.DFA_ERR_INVALID_ARG),
    (dict(scale=0.0), dfa.DFA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), dfa.DFA_ERR_INVALID_ARG),
    (dict(q=None), dfa.DFA_ERR_INVALID_ARG),
    (dict(O=MIS), dfa.DFA_ERR_INVALID_ARG),
    (dict(Lq=-1), dfa.DFA_ERR_INVALID_ARG),
    (dict(qo=-5), dfa.DFA_ERR_INVALID_ARG),
    (dict(dt=7), dfa.DFA_ERR_INVALID_ARG),
    (dict(qs=(ctypes.c_int64 * 3)(128 * 256, 256, 12)), dfa.DFA_ERR_INVALID_ARG),   # head stride not /8
])
def test_chunk_fwd_validation(kw, code):
    st, msg = chunk(**kw)
    assert st == code and msg


def test_empty_chunk_is_a_no_op():
    st, _ = chunk(Lq=0, q=None, O=None, lse=None)
    assert st == dfa.DFA_OK
    st, _ = chunk(B=0, q=None, O=None, lse=None)
    assert st == dfa.DFA_OK


def test_whole_sequence_validation():
    f = lib.dfa_attn_fwd
    ws = dfa.dfa_attn_workspace_size(1, 4, 2, 1024, 128, 4, 0)
    assert ws > 0 and ws % 256 == 0
    # n_chunks that leaves the last chunk empty (S = 9: chunks of 3, 3, 3 and 0); a
    # ragged last chunk is valid (S = 1000, 3 chunks of 334, 334, 332)
    assert f(A, A, A, 1, 1, 4, 2, 9, 128, 4, 1, 0.1, 0, A, A, A, ws, None) == dfa.DFA_ERR_INVALID_ARG
    assert f(A, A, A, 1, 1, 4, 2, 8, 128, 9, 1, 0.1, 0, A, A, A, ws, None) == dfa.DFA_ERR_INVALID_ARG
    assert dfa.dfa_attn_workspace_size(1, 4, 2, 1000, 128, 3, 0) > 0
    # workspace too small / missing
    assert f(A, A, A, 1, 1, 4, 2, 1024, 128, 4, 1, 0.1, 0, A, A, A, ws - 256, None) == dfa.DFA_ERR_WORKSPACE
    assert f(A, A, A, 1, 1, 4, 2, 1024, 128, 4, 1, 0.1, 0, A, A, None, ws, None) == dfa.DFA_ERR_WORKSPACE
    # bad schedule
    assert f(A, A, A, 1, 1, 4, 2, 1024, 128, 4, 1, 0.1, 9, A, A, A, ws, None) == dfa.DFA_ERR_INVALID_ARG
    # empty problem: OK without touching anything
    assert f(None, None, None, 1, 0, 4, 2, 1024, 128, 4, 1, 0.1, 0, None, None, None, 0, None) == dfa.DFA_OK
    b = lib.dfa_attn_bwd
    wsb = dfa.dfa_attn_workspace_size(1, 4, 2, 1024, 128, 4, 1)
    assert wsb > ws
    assert b(A, A, A, A, A, A, 1, 1, 4, 2, 1024, 128, 4, 1, 0.1, 0, A, A, A, A, wsb - 1, None) == dfa.DFA_ERR_WORKSPACE
    assert b(A, A, A, A, A, MIS, 1, 1, 4, 2, 1024, 128, 4, 1, 0.1, 0, A, A, A, A, wsb, None) == dfa.DFA_ERR_INVALID_ARG


def test_workspace_size_rejects_bad_shapes():
    assert dfa.dfa_attn_workspace_size(1, 3, 2, 128, 128, 1, 0) == 0
    assert dfa.dfa_attn_workspace_size(1, 4, 2, 9, 128, 4, 0) == 0
    assert dfa.dfa_attn_workspace_size(1, 4, 2, 100, 128, 0, 0) == 0
    assert dfa.dfa_attn_workspace_size(1, 4, 2, 128, 80, 1, 1) == 0


def test_merge_validation():
    f = lib.dfa_merge_partials
    assert f(1, 2, 8, 6, A, A, A, A, A, A, None) == dfa.DFA_ERR_INVALID_ARG        # D % 4
    assert f(1, 2, 8, 64, A, A, None, A, A, A, None) == dfa.DFA_ERR_INVALID_ARG
    assert f(0, 2, 8, 64, None, None, None, None, None, None, None) == dfa.DFA_OK


def test_launch_counters_exist():
    for kind in dfa.KERNEL_KINDS:
        assert dfa.dfa_launch_count(kind) >= 0
    assert lib.dfa_launch_count(99) == -1
