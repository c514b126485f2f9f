"""Local sliding window (DISTFLASHATTN App. F) through the C ABI against the
fp64 oracle: a query sees its own chunk and the window - 1 chunks before it.

Cases cover chunk lengths that are multiples of the 256-row forward block, of
the 128-row tile only (a block straddles two windows), and of neither (the
window edge cuts through tiles), a ragged last chunk (S not a multiple of
n_chunks), head dims 128 and 64, GQA, and fp32 on the CUDA-core kernels.  Tolerances as in the other parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import make

pytestmark = pytest.mark.gpu
DEV = "cuda"


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check(O, lse, grads, Or, lr, refs, dtype, what):
    if dtype == torch.float32:
        assert np.max(np.abs(np64(O) - Or)) <= 1e-4, f"{what}: O"
        assert np.max(np.abs(np64(lse) - lr)) <= 1e-5, f"{what}: lse"
    else:
        assert np.max(np.abs(np64(O) - Or)) <= 2e-2, f"{what}: O"
        assert np.max(np.abs(np64(lse) - lr)) <= 1e-3, f"{what}: lse"
    for name, g, r in zip(("dQ", "dK", "dV"), grads, refs):
        err = np.max(np.abs(np64(g) - r))
        if dtype == torch.float32:
            assert err <= 1e-3, f"{what}: {name} abs err {err}"
        else:
            rel = err / max(np.max(np.abs(r)), 1e-2)
            assert rel <= 3e-2, f"{what}: {name} rel err {rel}"


# (B, H, Hkv, S, D, dtype, n_chunks, window, note)
CASES = [
    (1, 4, 2, 1024, 128, torch.bfloat16, 4, 2, "C=256, two chunks"),
    (1, 2, 1, 1536, 128, torch.bfloat16, 4, 1, "C=384: a 256-row block straddles windows"),
    (1, 2, 2, 1280, 128, torch.bfloat16, 4, 2, "C=320: the window edge cuts through tiles"),
    (2, 2, 1, 1024, 128, torch.bfloat16, 8, 3, "C=128, three chunks, batch 2"),
    (1, 2, 2, 768, 64, torch.bfloat16, 3, 2, "D=64"),
    (1, 2, 1, 300, 64, torch.float32, 3, 2, "fp32 on CUDA cores"),
    (1, 4, 2, 1000, 128, torch.bfloat16, 3, 2, "ragged last chunk: 334, 334, 332"),
    (1, 2, 1, 2301, 128, torch.bfloat16, 5, 2, "ragged last chunk: four of 461, one of 457"),
    (1, 2, 2, 700, 64, torch.bfloat16, 3, 1, "ragged last chunk, D=64: 234, 234, 232"),
    (1, 2, 1, 301, 64, torch.float32, 4, 2, "ragged last chunk, fp32: 76, 76, 76, 73"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[-1] for c in CASES])
def test_local_window_matches_oracle(case):
    B, H, Hkv, S, D, dtype, P, w, what = case
    q, k, v, do = make(B, H, Hkv, S, D, dtype, device=DEV, seed=21)
    O, lse = dfa.dfa_attn_fwd_local(q, k, v, n_chunks=P, window=w)
    grads = dfa.dfa_attn_bwd_local(q, k, v, O, lse, do, n_chunks=P, window=w)
    dfa.dfa_check_errors()
    C = -(-S // P)   # every chunk but the last holds ceil(S / P) tokens
    Or, lr = oracle.attn_fwd_local(np64(q), np64(k), np64(v), chunk=C, window=w)
    refs = oracle.attn_bwd_local(np64(q), np64(k), np64(v), np64(do), chunk=C, window=w)
    check(O, lse, grads, Or, lr, refs, dtype, what)


def test_window_covering_all_chunks_gives_the_causal_bits():
    q, k, v, do = make(1, 2, 2, 1024, 128, torch.bfloat16, device=DEV, seed=22)
    O1, l1 = dfa.dfa_attn_fwd_local(q, k, v, n_chunks=4, window=4)
    O2, l2 = dfa.dfa_attn_fwd(q, k, v, n_chunks=4)
    assert torch.equal(O1, O2) and torch.equal(l1, l2)
    g1 = dfa.dfa_attn_bwd_local(q, k, v, O1, l1, do, n_chunks=4, window=4)
    g2 = dfa.dfa_attn_bwd(q, k, v, O2, l2, do, n_chunks=4)
    for a, b in zip(g1, g2):
        torch.testing.assert_close(a, b, rtol=0, atol=2e-3)   # dQ adds in a different order (atomics)


def test_bad_window_is_rejected():
    q, k, v, do = make(1, 2, 2, 256, 128, torch.bfloat16, device=DEV, seed=23)
    with pytest.raises(dfa.DfaError):
        dfa.dfa_attn_fwd_local(q, k, v, n_chunks=2, window=0)


def test_the_benchmark_local_window_at_full_size():
    """The configuration the benchmark times: the 128K workload (32 heads,
    D = 128) in 16 chunks of 8192 tokens with a window of two chunks.  A query
    row of chunk c sees exactly chunks c - 1 and c, and a key of chunk c - 1
    is seen by the queries of chunks c - 1 and c; so the oracle's local window
    on the slice of chunks [c - 2, c] (positions kept global through the
    offsets) gives chunk c's O, lse and dQ and chunk c - 1's dK and dV as in
    the whole sequence.  Checked for chunk 1 on head 0 and chunk 15 on the
    last head (a different key/value head)."""
    from long_context_causal_gb300.inputs import WORKLOADS, make_workload
    w = WORKLOADS["llama7b_s128k"]
    q, k, v, do = make_workload(w, DEV)
    P, W = w.n_chunks, 2
    C = w.S // P
    O, lse = dfa.dfa_attn_fwd_local(q, k, v, n_chunks=P, window=W, scale=w.scale)
    dQ, dK, dV = dfa.dfa_attn_bwd_local(q, k, v, O, lse, do, n_chunks=P, window=W, scale=w.scale)
    dfa.dfa_check_errors()
    for c, h in ((1, 0), (P - 1, w.H - 1)):
        g = h // (w.H // w.H_kv)
        a, m, b = max(c - 2, 0) * C, c * C, (c + 1) * C
        prev = m - C - a                                  # chunk c - 1 within the slice
        sl = lambda t, j: np64(t[:, a:b, j:j + 1])
        Or, lr = oracle.attn_fwd_local(sl(q, h), sl(k, g), sl(v, g), chunk=C, window=W, scale=w.scale,
                                       q_offset=a, kv_offset=a)
        dqr, dkr, dvr = oracle.attn_bwd_local(sl(q, h), sl(k, g), sl(v, g), sl(do, h), chunk=C, window=W,
                                              scale=w.scale, q_offset=a, kv_offset=a)
        what = f"chunk {c} head {h}"
        assert np.max(np.abs(np64(O[:, m:b, h]) - Or[:, m - a:, 0])) <= 2e-2, f"{what}: O"
        assert np.max(np.abs(np64(lse[:, h, m:b]) - lr[:, 0, m - a:])) <= 1e-3, f"{what}: lse"
        for name, gpu, ref in (("dQ", dQ[:, m:b, h], dqr[:, m - a:, 0]),
                               ("dK", dK[:, m - C:m, g], dkr[:, prev:prev + C, 0]),
                               ("dV", dV[:, m - C:m, g], dvr[:, prev:prev + C, 0])):
            rel = np.max(np.abs(np64(gpu) - ref)) / max(np.max(np.abs(ref)), 1e-2)
            assert rel <= 3e-2, f"{what}: {name} rel err {rel}"
