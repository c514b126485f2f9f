"""Parity of the chunk-pair backward step (DISTFLASHATTN §3.3: a worker's
backward for one (query chunk, key chunk) pair, from the owner's saved output
and log-sum-exp) against the fp64 oracle, through the C ABI.

Every case takes a query chunk and a key chunk out of one longer sequence
whose final O and lse come from the oracle's full forward, so the pair sees
the global row statistics exactly as a worker would.  Tolerances as in the
other parity tests: fp32 I/O 1e-3 absolute on each partial gradient; bf16
I/O 3e-2 x max|reference partial| (floor 1e-2).
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


def check(got, ref, dtype, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        err = np.max(np.abs(np64(g) - r)) if r.size else 0.0
        if dtype == torch.float32:
            assert err <= 1e-3, f"{what}: {name} abs err {err}"
        else:
            rel = err / max(np.max(np.abs(r)), 1e-2)
            assert rel <= 3e-2, f"{what}: {name} rel err {rel}"


def sequence(B, H, Hkv, S, D, dtype, seed):
    q, k, v, do = make(B, H, Hkv, S, D, dtype, device=DEV, seed=seed)
    O, lse = oracle.attn_fwd(np64(q), np64(k), np64(v), causal=True)
    dlt = oracle.delta(np64(q), np64(k), np64(v), np64(do), causal=True)
    return q, k, v, do, O, lse, dlt


def pair(seq, qa, qb, ka, kb, dtype, causal=True):
    q, k, v, do, O, lse, dlt = seq
    sl = lambda t, a, b: t[:, a:b].contiguous()
    Og = torch.from_numpy(O[:, qa:qb]).to(dtype=dtype, device=DEV).contiguous()
    lg = torch.from_numpy(lse[:, :, qa:qb]).to(dtype=torch.float32, device=DEV).contiguous()
    got = dfa.dfa_chunk_attn_bwd(sl(q, qa, qb), sl(k, ka, kb), sl(v, ka, kb), Og, lg, sl(do, qa, qb),
                                 q_offset=qa, kv_offset=ka, causal=causal)
    dfa.dfa_check_errors()
    ref = oracle.chunk_bwd(np64(q[:, qa:qb]), np64(k[:, ka:kb]), np64(v[:, ka:kb]), np64(do[:, qa:qb]),
                           lse[:, :, qa:qb], dlt[:, :, qa:qb], q_offset=qa, kv_offset=ka, causal=causal)
    return got, ref


# (B, H, Hkv, S, D, dtype, q chunk [qa, qb), key chunk [ka, kb), path)
CASES = [
    (1, 4, 2, 768, 128, torch.bfloat16, (512, 768), (0, 256), "tensor cores: below the diagonal"),
    (1, 4, 2, 768, 128, torch.bfloat16, (384, 768), (384, 768), "tensor cores: diagonal pair"),
    (1, 2, 1, 900, 128, torch.bfloat16, (512, 812), (128, 328), "tensor cores: ragged chunks"),
    (2, 2, 2, 640, 128, torch.bfloat16, (256, 384), (128, 640), "tensor cores: keys straddle the queries"),
    (1, 2, 1, 300, 64, torch.bfloat16, (137, 300), (11, 170), "CUDA cores: D = 64, unaligned offsets"),
    (1, 3, 1, 200, 128, torch.float32, (64, 200), (37, 120), "CUDA cores: fp32"),
    (1, 2, 2, 384, 128, torch.bfloat16, (128, 256), (130, 300), "CUDA cores: offsets not 128 apart"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[-1] for c in CASES])
def test_chunk_pair_backward_matches_oracle(case):
    B, H, Hkv, S, D, dtype, (qa, qb), (ka, kb), what = case
    seq = sequence(B, H, Hkv, S, D, dtype, seed=11)
    got, ref = pair(seq, qa, qb, ka, kb, dtype)
    check(got, ref, dtype, what)


def test_pair_above_the_diagonal_adds_nothing():
    seq = sequence(1, 2, 2, 512, 128, torch.bfloat16, seed=12)
    got, _ = pair(seq, 0, 256, 256, 512, torch.bfloat16)
    for t in got:
        assert torch.count_nonzero(t) == 0


def test_non_causal_pair():
    dtype = torch.bfloat16
    q, k, v, do = make(1, 2, 1, 384, 128, dtype, device=DEV, seed=13)
    O, lse = oracle.attn_fwd(np64(q), np64(k), np64(v), causal=False)
    dlt = oracle.delta(np64(q), np64(k), np64(v), np64(do), causal=False)
    got, ref = pair((q, k, v, do, O, lse, dlt), 0, 128, 256, 384, dtype, causal=False)
    check(got, ref, dtype, "non-causal")


def test_accumulators_are_added_to():
    seq = sequence(1, 2, 1, 512, 128, torch.bfloat16, seed=14)
    (q, k, v, do, O, lse, _) = seq
    Og = torch.from_numpy(O[:, 256:]).to(dtype=torch.bfloat16, device=DEV).contiguous()
    lg = torch.from_numpy(lse[:, :, 256:]).to(dtype=torch.float32, device=DEV).contiguous()
    args = (q[:, 256:].contiguous(), k[:, :256].contiguous(), v[:, :256].contiguous(), Og, lg, do[:, 256:].contiguous())
    once = dfa.dfa_chunk_attn_bwd(*args, q_offset=256, kv_offset=0)
    twice = dfa.dfa_chunk_attn_bwd(*args, q_offset=256, kv_offset=0)
    dfa.dfa_chunk_attn_bwd(*args, q_offset=256, kv_offset=0, dQ_acc=twice[0], dK_acc=twice[1], dV_acc=twice[2])
    dfa.dfa_check_errors()
    for a, b in zip(once, twice):
        torch.testing.assert_close(b, 2 * a, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("P", [2, 4])
def test_pairs_sum_to_the_whole_sequence_backward(P):
    # The distributed backward: every worker adds its pairs' shares; the totals
    # are the whole-sequence gradients (compared with the oracle and with the
    # library's own whole-sequence backward).
    B, H, Hkv, S, D, dtype = 1, 4, 2, 1024, 128, torch.bfloat16
    q, k, v, do = make(B, H, Hkv, S, D, dtype, device=DEV, seed=15)
    O, lse = dfa.dfa_attn_fwd(q, k, v)
    C = S // P
    f32 = dict(dtype=torch.float32, device=DEV)
    dQ, dK, dV = (torch.zeros((B, S, H, D), **f32), torch.zeros((B, S, Hkv, D), **f32),
                  torch.zeros((B, S, Hkv, D), **f32))
    launches = dfa.dfa_launch_count("fwd")
    for p in range(P):
        qs = slice(p * C, (p + 1) * C)
        for r in range(p + 1):
            ks = slice(r * C, (r + 1) * C)
            dfa.dfa_chunk_attn_bwd(q[:, qs], k[:, ks], v[:, ks], O[:, qs], lse[:, :, qs].contiguous(), do[:, qs],
                                   q_offset=p * C, kv_offset=r * C, dQ_acc=dQ[:, qs], dK_acc=dK[:, ks],
                                   dV_acc=dV[:, ks])
    dfa.dfa_check_errors()
    assert dfa.dfa_launch_count("fwd") == launches, "the backward step must not run a forward"
    ref = oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do))
    check((dQ, dK, dV), ref, dtype, f"sum over {P} chunks")
    whole = dfa.dfa_attn_bwd(q, k, v, O, lse, do)
    for a, b in zip((dQ, dK, dV), whole):
        err = (a - b.float()).abs().max().item() / max(b.float().abs().max().item(), 1e-2)
        assert err <= 2e-2, err


def test_bad_arguments_are_rejected():
    q, k, v, do = make(1, 2, 1, 256, 128, torch.bfloat16, device=DEV, seed=16)
    O = torch.zeros_like(q)
    lse = torch.zeros((1, 2, 256), dtype=torch.float32, device=DEV)
    with pytest.raises(dfa.DfaError):
        dfa.dfa_chunk_attn_bwd(q, k, v, O, lse, do, q_offset=-1)
    with pytest.raises(dfa.DfaError):
        dfa.dfa_chunk_attn_bwd(q, k, v, O, lse, do, workspace_buf=torch.empty(16, dtype=torch.uint8, device=DEV))


def test_the_benchmark_chunk_steps_at_full_size():
    """The chunk steps the benchmark times, on the 128K workload (16 chunks of
    8192 tokens, 32 heads).  Forward: the last query chunk against key chunk 0
    (no mask) and against itself (the diagonal) matches the oracle on sampled
    rows of two heads, with the chunks' global offsets.  Backward: the chunk
    steps of the last query chunk over all 16 key chunks add up to the
    whole-sequence dQ of its rows, and those of key chunk 0 over all 16 query
    chunks to the whole-sequence dK and dV of its keys (the whole-sequence
    gradients are checked against the oracle at this size in
    test_parity_large.py)."""
    from long_context_causal_gb300.inputs import WORKLOADS, make_workload
    w = WORKLOADS["llama7b_s128k"]
    q, k, v, do = make_workload(w, DEV)
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=w.n_chunks, scale=w.scale)
    dQ, dK, dV = dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=w.n_chunks, scale=w.scale)
    P = w.n_chunks
    C = w.S // P
    last = (P - 1) * C
    G = w.H // w.H_kv
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, C - 1], rng.integers(0, C, 64)])).astype(np.int64)
    idx = np.stack([np.zeros_like(rows), np.zeros_like(rows), rows], 1)
    for ka in (0, last):
        Op, lp = dfa.dfa_chunk_attn_fwd(q[:, last:], k[:, ka:ka + C], v[:, ka:ka + C], q_offset=last, kv_offset=ka,
                                        scale=w.scale)
        for h in (0, w.H - 1):
            g = h // G
            Or, lr = oracle.attn_fwd_rows(np64(q[:, last:, h:h + 1]), np64(k[:, ka:ka + C, g:g + 1]),
                                          np64(v[:, ka:ka + C, g:g + 1]), idx, scale=w.scale, q_offset=last,
                                          kv_offset=ka)
            t = torch.as_tensor(rows, device=DEV)
            assert np.max(np.abs(np64(Op[0, t, h]) - Or)) <= 2e-2, (ka, h, "O")
            assert np.max(np.abs(np64(lp[0, h, t]) - lr)) <= 1e-3, (ka, h, "lse")
        del Op, lp
    f32 = dict(dtype=torch.float32, device=DEV)

    def step(i, j, dq, dk, dv):
        qs, ks = slice(i * C, (i + 1) * C), slice(j * C, (j + 1) * C)
        dfa.dfa_chunk_attn_bwd(q[:, qs], k[:, ks], v[:, ks], O[:, qs], lse[:, :, qs].contiguous(), do[:, qs],
                               q_offset=i * C, kv_offset=j * C, scale=w.scale, dQ_acc=dq, dK_acc=dk, dV_acc=dv)
    dq = torch.zeros((1, C, w.H, w.D), **f32)
    scratch_k, scratch_v = torch.zeros((1, C, w.H_kv, w.D), **f32), torch.zeros((1, C, w.H_kv, w.D), **f32)
    for j in range(P):
        step(P - 1, j, dq, scratch_k, scratch_v)
    dk, dv = torch.zeros((1, C, w.H_kv, w.D), **f32), torch.zeros((1, C, w.H_kv, w.D), **f32)
    scratch_q = torch.zeros((1, C, w.H, w.D), **f32)
    for i in range(P):
        step(i, 0, scratch_q, dk, dv)
    dfa.dfa_check_errors()
    for name, got, whole in (("dQ", dq, dQ[:, last:]), ("dK", dk, dK[:, :C]), ("dV", dv, dV[:, :C])):
        ref = whole.float()
        err = (got - ref).abs().max().item()
        assert err <= 1e-2 * ref.abs().max().item(), f"{name}: {err}"
