"""Variable-length (packed) batches through the C ABI against the fp64 oracle.

Every sequence of a packed batch is plain attention on its own (no token
attends across a sequence boundary).  Tolerances as in test_parity.py (bf16
I/O: O 2e-2, lse 1e-3 max abs; each gradient 3e-2 x max|reference gradient|).
A packed batch holding one sequence, or sequences of one length, computes
each query block exactly as the dense entry points do, so the forward bits
and dK/dV bits agree with them; dQ adds its partials with unordered atomics
and agrees to 2e-2.
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


def packed(lens, H, Hkv, D, seed, k_scale=1.0):
    T = int(sum(lens))
    q, k, v, do = make(1, H, Hkv, T, D, torch.bfloat16, seed=seed, device=DEV, k_scale=k_scale)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q[0], k[0], v[0], do[0], cu


CASES = [
    # (lens, H, Hkv, D, causal)
    ([300, 0, 1000, 1, 129, 2048], 4, 2, 128, True),    # ragged tails, an empty and a one-token sequence
    ([17, 256, 255, 513], 2, 1, 64, True),               # D = 64 kernels, GQA 2:1
    ([200, 700], 2, 2, 128, False),                      # non-causal inside each sequence
    ([128, 128, 384, 4096], 8, 8, 128, True),            # tile-aligned lengths, one long sequence
    ([4096, 100, 2000], 8, 1, 128, True),                # GQA 8:1
    ([333, 777], 4, 4, 64, False),                       # D = 64, non-causal
]


@pytest.mark.parametrize("case", CASES)
def test_varlen_matches_oracle(case):
    lens, H, Hkv, D, causal = case
    q, k, v, do, cu = packed(lens, H, Hkv, D, seed=43)
    O, lse = dfa.dfa_attn_fwd_varlen(q, k, v, cu, causal=causal)
    dQ, dK, dV = dfa.dfa_attn_bwd_varlen(q, k, v, O, lse, do, cu, causal=causal)
    dfa.dfa_check_errors()
    Or, lr = oracle.attn_fwd_varlen(np64(q), np64(k), np64(v), cu, causal=causal)
    assert np.max(np.abs(np64(O) - Or)) <= 2e-2, f"{case}: O"
    assert np.max(np.abs(np64(lse) - lr)) <= 1e-3, f"{case}: lse"
    ref = oracle.attn_bwd_varlen(np64(q), np64(k), np64(v), np64(do), cu, causal=causal)
    for name, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref):
        rel = np.max(np.abs(np64(g) - r)) / max(np.max(np.abs(r)), 1e-2)
        assert rel <= 3e-2, f"{case}: {name} rel err {rel}"


def test_one_sequence_is_the_dense_entry_point():
    q, k, v, do, cu = packed([1536], 4, 2, 128, seed=47)
    O, lse = dfa.dfa_attn_fwd_varlen(q, k, v, cu)
    g = dfa.dfa_attn_bwd_varlen(q, k, v, O, lse, do, cu)
    Od, ld = dfa.dfa_attn_fwd(q[None], k[None], v[None])
    gd = dfa.dfa_attn_bwd(q[None], k[None], v[None], Od, ld, do[None])
    dfa.dfa_check_errors()
    assert torch.equal(O, Od[0]) and torch.equal(lse, ld[0])
    assert torch.equal(g[1], gd[1][0]) and torch.equal(g[2], gd[2][0])
    assert torch.max(torch.abs(g[0].float() - gd[0][0].float())).item() <= 2e-2


def test_equal_lengths_are_the_dense_batch():
    n, L, H, Hkv, D = 3, 640, 2, 2, 64
    q, k, v, do, cu = packed([L] * n, H, Hkv, D, seed=53)
    O, lse = dfa.dfa_attn_fwd_varlen(q, k, v, cu)
    Od, ld = dfa.dfa_attn_fwd(q.view(n, L, H, D), k.view(n, L, Hkv, D), v.view(n, L, Hkv, D))
    torch.cuda.synchronize()
    assert torch.equal(O.view(n, L, H, D), Od)
    assert torch.equal(lse.view(H, n, L).transpose(0, 1), ld)


def test_many_short_sequences_in_one_launch():
    rng = np.random.default_rng(59)
    lens = rng.integers(1, 700, 40).tolist()
    q, k, v, do, cu = packed(lens, 4, 1, 128, seed=61, k_scale=2.0)
    launches = dfa.dfa_launch_count("fwd")
    O, lse = dfa.dfa_attn_fwd_varlen(q, k, v, cu)
    dQ, dK, dV = dfa.dfa_attn_bwd_varlen(q, k, v, O, lse, do, cu)
    dfa.dfa_check_errors()
    assert dfa.dfa_launch_count("fwd") == launches + 1
    Or, lr = oracle.attn_fwd_varlen(np64(q), np64(k), np64(v), cu)
    assert np.max(np.abs(np64(O) - Or)) <= 2e-2
    assert np.max(np.abs(np64(lse) - lr)) <= 1e-3
    ref = oracle.attn_bwd_varlen(np64(q), np64(k), np64(v), np64(do), cu)
    for name, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref):
        rel = np.max(np.abs(np64(g) - r)) / max(np.max(np.abs(r)), 1e-2)
        assert rel <= 3e-2, f"{name} rel err {rel}"


def test_empty_batch_and_bad_offsets():
    q, k, v, do, cu = packed([64], 2, 2, 128, seed=67)
    O, lse = dfa.dfa_attn_fwd_varlen(q[:0], k[:0], v[:0], [0])
    assert O.shape == (0, 2, 128)
    with pytest.raises(dfa.DfaError) as e:
        dfa.dfa_attn_fwd_varlen(q, k, v, cu, workspace_buf=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert e.value.status == dfa.DFA_ERR_WORKSPACE
    with pytest.raises(dfa.DfaError) as e:   # offsets that end past the packed tensor
        dfa.dfa_attn_fwd_varlen(q, k, v, [0, 100])
    assert e.value.status == dfa.DFA_ERR_INVALID_ARG
    with pytest.raises(dfa.DfaError) as e:
        dfa.dfa_attn_fwd_varlen(q, k, v, [0, 40, 20])
    assert e.value.status == dfa.DFA_ERR_INVALID_ARG
    with pytest.raises(dfa.DfaError) as e:
        dfa.dfa_attn_fwd_varlen(q.float(), k.float(), v.float(), cu)
    assert e.value.status == dfa.DFA_ERR_UNSUPPORTED


def test_shutdown_releases_caches_and_later_calls_rebuild_them():
    q, k, v, do, cu = packed([700, 300], 2, 2, 128, seed=71)
    O1, l1 = dfa.dfa_attn_fwd_varlen(q, k, v, cu)
    g1 = dfa.dfa_attn_bwd_varlen(q, k, v, O1, l1, do, cu)
    Od1, ld1 = dfa.dfa_attn_fwd(q[None], k[None], v[None], sched="split_kv")
    torch.cuda.synchronize()
    dfa.dfa_shutdown()
    O2, l2 = dfa.dfa_attn_fwd_varlen(q, k, v, cu)
    g2 = dfa.dfa_attn_bwd_varlen(q, k, v, O2, l2, do, cu)
    Od2, ld2 = dfa.dfa_attn_fwd(q[None], k[None], v[None], sched="split_kv")
    dfa.dfa_check_errors()
    assert torch.equal(O1, O2) and torch.equal(l1, l2) and torch.equal(Od1, Od2) and torch.equal(ld1, ld2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])


def test_batches_of_empty_and_of_one_token_sequences():
    q, k, v, do, cu = packed([64], 2, 2, 128, seed=97)
    O, lse = dfa.dfa_attn_fwd_varlen(q[:0], k[:0], v[:0], [0, 0, 0])      # three empty sequences
    g = dfa.dfa_attn_bwd_varlen(q[:0], k[:0], v[:0], O, lse, do[:0], [0, 0, 0])
    dfa.dfa_check_errors()
    assert O.shape[0] == 0 and all(t.shape[0] == 0 for t in g)
    q, k, v, do, cu = packed([1] * 7, 4, 2, 128, seed=101)                 # seven one-token sequences
    O, lse = dfa.dfa_attn_fwd_varlen(q, k, v, cu)
    dQ, dK, dV = dfa.dfa_attn_bwd_varlen(q, k, v, O, lse, do, cu)
    dfa.dfa_check_errors()
    # One token sees only itself: O = v of its group, P = 1 so dS = 0 (dQ = dK = 0) and dV = sum of dO over the group.
    G = 2
    vg = v.float().repeat_interleave(G, dim=1)
    assert torch.max(torch.abs(O.float() - vg)).item() <= 1e-2
    Or, lr = oracle.attn_fwd_varlen(np64(q), np64(k), np64(v), cu)
    assert np.max(np.abs(np64(lse) - lr)) <= 1e-3
    assert torch.max(torch.abs(dQ.float())).item() <= 1e-2 and torch.max(torch.abs(dK.float())).item() <= 1e-2
    dv_ref = do.float().view(7, 2, G, 128).sum(dim=2)
    assert torch.max(torch.abs(dV.float() - dv_ref)).item() <= 2e-2 * max(torch.max(torch.abs(dv_ref)).item(), 1.0)


def test_the_benchmark_packed_batch_equals_one_dense_call_per_sequence():
    """The packed batch the benchmark times (ten sequences, 57344 down to 512
    tokens, 131072 in all, 32 heads, D = 128, same seed): one packed call each
    way gives every sequence the bits of a dense call on that sequence alone
    (O, lse, dK, dV), and its dQ within rounding."""
    lens = [57344, 28672, 16384, 12288, 8192, 4096, 2048, 1024, 512, 512]
    q, k, v, do, cu = packed(lens, 32, 32, 128, seed=5)
    O, lse = dfa.dfa_attn_fwd_varlen(q, k, v, cu)
    dQ, dK, dV = dfa.dfa_attn_bwd_varlen(q, k, v, O, lse, do, cu)
    for a, b in zip(cu[:-1].tolist(), cu[1:].tolist()):
        Od, ld = dfa.dfa_attn_fwd(q[None, a:b], k[None, a:b], v[None, a:b])
        assert torch.equal(O[a:b], Od[0]) and torch.equal(lse[:, a:b], ld[0]), (a, b)
        gq, gk, gv = dfa.dfa_attn_bwd(q[None, a:b], k[None, a:b], v[None, a:b], Od, ld, do[None, a:b])
        assert torch.equal(dK[a:b], gk[0]) and torch.equal(dV[a:b], gv[0]), (a, b)
        scale = gq.float().abs().max().item()
        assert (dQ[a:b].float() - gq[0].float()).abs().max().item() <= 1e-2 * scale, (a, b)
        del Od, ld, gq, gk, gv
    dfa.dfa_check_errors()
