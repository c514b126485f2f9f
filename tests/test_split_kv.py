"""Split-kv helper items (DISTFLASHATTN §3.2: idle workers compute part of a busy
worker's attention and return a partial output with its log-sum-exp, which the
owner merges) against the fp64 oracle and against the unsplit forward.

Tolerances as in test_parity.py (bf16 I/O: O 2e-2, lse 1e-3 max abs; each
gradient 3e-2 x max|reference gradient|).  The split forward and the plain
balanced forward agree to the same bounds: both are the exact softmax, the
split one only rounds the pieces' partials through fp32 before the merge.
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


def n_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def check_fwd(O, lse, Or, lr, what):
    eo = np.max(np.abs(np64(O) - Or))
    lg = np64(lse)
    fin = np.isfinite(lr)
    assert np.array_equal(np.isfinite(lg), fin), f"{what}: -inf pattern of lse differs"
    el = np.max(np.abs(lg[fin] - lr[fin]))
    assert eo <= 2e-2, f"{what}: O err {eo}"
    assert el <= 1e-3, f"{what}: lse err {el}"


CASES = [
    # (B, H, Hkv, S, D, causal, k_scale)
    (1, 1, 1, 4096, 128, True, 1.0),
    (1, 2, 1, 8192, 64, True, 1.0),      # GQA, D = 64, ragged last piece
    (1, 1, 1, 1000, 128, True, 1.0),     # ragged last tile
    (1, 2, 2, 2048, 128, False, 1.0),    # non-causal: every block sees every piece
    (2, 3, 3, 1536, 128, True, 1.0),     # batch
    (1, 4, 1, 2048, 128, True, 4.0),     # sharp softmax: pieces with very different maxima
    (1, 8, 1, 4096, 128, True, 1.0),     # GQA 8:1
    (2, 2, 2, 1280, 64, False, 1.0),     # D = 64, non-causal, batch, ragged
]


@pytest.mark.parametrize("case", CASES)
def test_split_kv_forward_matches_oracle_and_backward_uses_it(case):
    B, H, Hkv, S, D, causal, ks = case
    assert dfa.dfa_split_piece_tiles(B, H, S, causal, n_sms()) > 0, "case must be split"
    q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=29, device=DEV, k_scale=ks)
    merges = dfa.dfa_launch_count("merge")
    O, lse = dfa.dfa_attn_fwd(q, k, v, causal=causal, sched="split_kv")
    dfa.dfa_check_errors()
    assert dfa.dfa_launch_count("merge") == merges + 1, "the split path merges its pieces"
    Or, lr = oracle.attn_fwd(np64(q), np64(k), np64(v), causal=causal)
    check_fwd(O, lse, Or, lr, str(case))
    Ob, lb = dfa.dfa_attn_fwd(q, k, v, causal=causal, sched="balanced")
    torch.cuda.synchronize()
    assert torch.max(torch.abs(O.float() - Ob.float())).item() <= 2e-2
    assert torch.max(torch.abs(lse - lb)).item() <= 1e-3
    grads = dfa.dfa_attn_bwd(q, k, v, O, lse, do, causal=causal, sched="split_kv")
    dfa.dfa_check_errors()
    ref = oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do), causal=causal)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        rel = np.max(np.abs(np64(g) - r)) / max(np.max(np.abs(r)), 1e-2)
        assert rel <= 3e-2, f"{case}: {name} rel err {rel}"


def test_split_kv_on_a_problem_too_small_to_split_is_the_balanced_forward():
    q, k, v, _ = make(1, 1, 1, 256, 128, torch.bfloat16, seed=31, device=DEV)
    assert dfa.dfa_split_piece_tiles(1, 1, 256, True, n_sms()) == 0
    O, lse = dfa.dfa_attn_fwd(q, k, v, sched="split_kv")
    Ob, lb = dfa.dfa_attn_fwd(q, k, v, sched="balanced")
    torch.cuda.synchronize()
    assert torch.equal(O, Ob) and torch.equal(lse, lb)


def test_split_kv_on_a_large_problem_is_the_balanced_forward():
    q, k, v, _ = make(1, 32, 32, 8192, 128, torch.bfloat16, seed=37, device=DEV)
    assert dfa.dfa_split_piece_tiles(1, 32, 8192, True, n_sms()) == 0
    merges = dfa.dfa_launch_count("merge")
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=8, sched="split_kv")
    Ob, lb = dfa.dfa_attn_fwd(q, k, v, n_chunks=8, sched="balanced")
    torch.cuda.synchronize()
    assert dfa.dfa_launch_count("merge") == merges
    assert torch.equal(O, Ob) and torch.equal(lse, lb)


def test_split_kv_long_single_head_agrees_with_sampled_oracle_rows():
    """One head of 32K tokens: 128 query blocks on a GPU of more SMs, the case
    split-kv is for.  Sampled rows (first, last, piece and tile boundaries,
    random) are checked against the oracle, the rest against the unsplit run."""
    S, D = 32768, 128
    q, k, v, _ = make(1, 1, 1, S, D, torch.bfloat16, seed=41, device=DEV)
    piece = dfa.dfa_split_piece_tiles(1, 1, S, True, n_sms())
    assert piece > 0
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=8, sched="split_kv")
    Ob, lb = dfa.dfa_attn_fwd(q, k, v, n_chunks=8, sched="balanced")
    torch.cuda.synchronize()
    assert torch.max(torch.abs(O.float() - Ob.float())).item() <= 2e-2
    assert torch.max(torch.abs(lse - lb)).item() <= 1e-3
    rng = np.random.default_rng(5)
    edge = [piece * 128 * m + d for m in range(1, S // (piece * 128) + 1) for d in (-1, 0)]
    rows = sorted({0, 1, 255, 256, S - 1, *[r for r in edge if 0 <= r < S], *rng.integers(0, S, 24).tolist()})
    idx = np.array([(0, 0, r) for r in rows], dtype=np.int64)
    Or, lr = oracle.attn_fwd_rows(np64(q), np64(k), np64(v), idx)
    eo = np.max(np.abs(np64(O[0, rows, 0]) - Or))
    el = np.max(np.abs(np64(lse[0, 0, rows]) - lr))
    assert eo <= 2e-2, f"32K sampled rows: O err {eo}"
    assert el <= 1e-3, f"32K sampled rows: lse err {el}"


BWD_CASES = [
    # (B, H, Hkv, S, causal): few key-tile pairs, so the backward splits every key tile's query range
    (1, 1, 1, 4096, True),
    (1, 1, 1, 8192, True),
    (1, 2, 1, 16384, True),     # GQA: the pieces of one key tile cover both heads of the group
    (1, 1, 1, 4096, False),
]


@pytest.mark.parametrize("case", BWD_CASES)
def test_split_kv_backward_pieces_match_oracle(case):
    B, H, Hkv, S, causal = case
    D = 128
    assert dfa.dfa_split_bwd_piece_tiles(B, Hkv, S, causal, n_sms()) > 0, "case must be split"
    q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=43, device=DEV)
    O, lse = dfa.dfa_attn_fwd(q, k, v, causal=causal)
    conv = dfa.dfa_launch_count("convert")
    grads = dfa.dfa_attn_bwd(q, k, v, O, lse, do, causal=causal, sched="split_kv")
    dfa.dfa_check_errors()
    assert dfa.dfa_launch_count("convert") == conv + 3, "dQ convert and the dK, dV casts"
    ref_grads = dfa.dfa_attn_bwd(q, k, v, O, lse, do, causal=causal, sched="balanced")
    dfa.dfa_check_errors()
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref_grads):
        scale = torch.max(torch.abs(r.float())).item()
        assert torch.max(torch.abs(g.float() - r.float())).item() <= 2e-2 * scale, f"{case}: {name} vs balanced"
    if S <= 8192:
        ref = oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do), causal=causal)
        for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
            rel = np.max(np.abs(np64(g) - r)) / max(np.max(np.abs(r)), 1e-2)
            assert rel <= 3e-2, f"{case}: {name} rel err {rel}"
