"""dfa_attn_fwd_noalloc: the forward for callers that cannot allocate device
memory (a plugin whose host framework owns all device memory, a service that
forbids allocation after start-up).  It keeps its work list in a static device
array instead of a caller workspace.

Checked through the C ABI against dfa_attn_fwd on the same inputs and the same
schedule.  Both run the same kernel over the same work list, so O and lse must
be bit-equal.  Every shape is called twice in a row, and the shapes are visited
in both orders, so that a call always finds another shape's (or its own) list
in the shared array.  Also checked: a ragged chunk split, the refusals (a
problem beyond the array's capacity, a split whose last chunk is empty, a call
on a capturing stream).  This file is collected last so that a
stop-at-first-failure run has already run every other test.
"""
import pytest
import torch

from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import make

pytestmark = pytest.mark.gpu

# (B, H, H_kv, S, D, n_chunks, schedule)
SHAPES = [
    (1, 8, 2, 2048, 128, 1, "balanced"),
    (2, 4, 4, 1000, 64, 1, "unbalanced"),
    (1, 4, 2, 1000, 128, 3, "balanced"),     # ragged: chunks of 334, 334, 332 tokens
]


def _inputs(shape):
    B, H, Hkv, S, D, P, sched = shape
    q, k, v, _ = make(B, H, Hkv, S, D, torch.bfloat16, seed=31, device="cuda")
    O_ref, l_ref = dfa.dfa_attn_fwd(q, k, v, n_chunks=P, sched=sched)
    return q, k, v, O_ref, l_ref


@pytest.mark.parametrize("order", ["forward", "reverse"])
def test_noalloc_forward_is_bit_equal_to_the_workspace_forward(order):
    shapes = SHAPES if order == "forward" else SHAPES[::-1]
    cases = [(s, _inputs(s)) for s in shapes]
    for (B, H, Hkv, S, D, P, sched), (q, k, v, O_ref, l_ref) in cases:
        for call in range(2):
            O = torch.full_like(q, float("nan"))
            lse = torch.full((B, H, S), float("nan"), device="cuda")
            dfa.dfa_attn_fwd_noalloc(q, k, v, O, lse, n_chunks=P, sched=sched)
            dfa.dfa_check_errors()
            assert torch.equal(O, O_ref), (B, H, S, P, sched, call, "O")
            assert torch.equal(lse, l_ref), (B, H, S, P, sched, call, "lse")


def test_noalloc_forward_refuses_problems_beyond_its_static_capacity():
    A = 0x10000   # never dereferenced: the size check comes first
    lib = dfa.library()
    st = lib.dfa_attn_fwd_noalloc(A, A, A, dfa.DFA_BF16, 1, 64, 64, 1 << 22, 128, 1, 1, 0.1,
                                  dfa.DFA_SCHED_BALANCED, A, A, None)
    assert st == dfa.DFA_ERR_INVALID_ARG
    assert "static work list" in dfa.dfa_last_error()


def test_noalloc_forward_refuses_a_split_with_an_empty_last_chunk():
    # S = 9 into 4 chunks of ceil(9/4) = 3 tokens leaves the last chunk empty.
    q, k, v, _ = make(1, 2, 2, 9, 128, torch.bfloat16, seed=1, device="cuda")
    O = torch.empty_like(q)
    lse = torch.empty((1, 2, 9), device="cuda")
    with pytest.raises(dfa.DfaError) as e:
        dfa.dfa_attn_fwd_noalloc(q, k, v, O, lse, n_chunks=4)
    assert e.value.status == dfa.DFA_ERR_INVALID_ARG


def test_noalloc_forward_refuses_a_capturing_stream():
    # Its upload reads a host array shared by every call, which a captured
    # graph would read again at replay time: the call must refuse and enqueue
    # nothing, leaving the capture intact.
    B, H, Hkv, S, D = 1, 2, 2, 512, 128
    q, k, v, _ = make(B, H, Hkv, S, D, torch.bfloat16, seed=2, device="cuda")
    O = torch.empty_like(q)
    lse = torch.empty((B, H, S), device="cuda")
    dfa.dfa_attn_fwd_noalloc(q, k, v, O, lse)     # first call: set-up outside any capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    refused = None
    with torch.cuda.graph(g, stream=s):
        try:
            dfa.dfa_attn_fwd_noalloc(q, k, v, O, lse)
        except dfa.DfaError as e:
            refused = e
    assert refused is not None and refused.status == dfa.DFA_ERR_INVALID_ARG
    assert "captured" in str(refused)
