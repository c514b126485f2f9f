"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (max abs error unless stated):
  fp32 I/O:  O 1e-4, lse 1e-5, dQ/dK/dV 1e-3; chunked vs unchunked 1e-5
  bf16 I/O:  O 2e-2, lse 1e-3, each gradient 3e-2 x max|reference gradient|
A gradient that is analytically zero (a single token: dS = P (dP - Delta) = 0)
has no scale of its own; its relative error is taken against a floor of 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import WORKLOADS, make, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda"

TOL = {
    torch.float32: dict(O=1e-4, lse=1e-5, grad_abs=1e-3),
    torch.bfloat16: dict(O=2e-2, lse=1e-3, grad_rel=3e-2),
}


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_fwd(O, lse, Or, lr, dtype, what=""):
    tol = TOL[dtype]
    eo = np.max(np.abs(np64(O) - Or)) if Or.size else 0.0
    fin = np.isfinite(lr)
    lg = np64(lse)
    assert np.array_equal(np.isfinite(lg), fin), f"{what}: -inf pattern of lse differs"
    el = np.max(np.abs(lg[fin] - lr[fin])) if fin.any() else 0.0
    assert eo <= tol["O"], f"{what}: O err {eo}"
    assert el <= tol["lse"], f"{what}: lse err {el}"


def check_grads(got, ref, dtype, what=""):
    tol = TOL[dtype]
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        err = np.max(np.abs(np64(g) - r))
        if dtype == torch.float32:
            assert err <= tol["grad_abs"], f"{what}: {name} abs err {err}"
        else:
            rel = err / max(np.max(np.abs(r)), 1e-2)
            assert rel <= tol["grad_rel"], f"{what}: {name} rel err {rel}"


def run_fwd_bwd(q, k, v, do, n_chunks=1, sched="balanced", causal=True):
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=n_chunks, causal=causal, sched=sched)
    dQ, dK, dV = dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=n_chunks, causal=causal, sched=sched)
    dfa.dfa_check_errors()
    return O, lse, (dQ, dK, dV)


# ---------------------------------------------------------------- workload 1, in full
def test_single_head_fp32_workload_full_oracle():
    w = WORKLOADS["single_head_s1k_fp32"]
    q, k, v, do = make_workload(w, DEV)
    O, lse, grads = run_fwd_bwd(q, k, v, do, n_chunks=w.n_chunks)
    Or, lr = oracle.attn_fwd(np64(q), np64(k), np64(v), scale=w.scale)
    check_fwd(O, lse, Or, lr, torch.float32, "fwd")
    ref = oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do), scale=w.scale)
    check_grads(grads, ref, torch.float32, "bwd")


def test_chunked_equals_unchunked_fp32():
    """Chunk steps merged with the rescale rule equal the whole-sequence forward."""
    w = WORKLOADS["single_head_s1k_fp32"]
    q, k, v, _ = make_workload(w, DEV)
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=w.n_chunks)
    C, P = w.chunk, w.n_chunks
    for p in range(P):
        qs = q[:, p * C:(p + 1) * C]
        acc = None
        for t in range(p + 1):
            part = dfa.dfa_chunk_attn_fwd(qs, k[:, t * C:(t + 1) * C], v[:, t * C:(t + 1) * C],
                                          q_offset=p * C, kv_offset=t * C)
            acc = part if acc is None else dfa.dfa_merge_partials(*acc, *part)
        dfa.dfa_check_errors()
        assert torch.max(torch.abs(acc[0] - O[:, p * C:(p + 1) * C])).item() <= 1e-5
        assert torch.max(torch.abs(acc[1] - lse[:, :, p * C:(p + 1) * C])).item() <= 1e-5


# ---------------------------------------------------------------- chunk step and merge
CHUNK_CASES = [
    # (dtype, B, H, Hkv, Lq, Lkv, D, q_off, kv_off, causal)
    (torch.float32, 1, 2, 1, 256, 256, 64, 256, 0, True),       # off-diagonal block: all visible
    (torch.float32, 2, 2, 2, 200, 300, 128, 100, 0, True),      # diagonal cuts the block, ragged
    (torch.bfloat16, 1, 4, 2, 256, 256, 128, 0, 0, True),       # diagonal block
    (torch.bfloat16, 2, 2, 1, 130, 250, 64, 300, 170, True),    # odd offsets, ragged tails
    (torch.bfloat16, 1, 2, 2, 128, 128, 128, 0, 64, True),      # first 64 rows see nothing
    (torch.bfloat16, 1, 2, 2, 96, 384, 128, 0, 0, False),       # non-causal
]


@pytest.mark.parametrize("case", CHUNK_CASES)
def test_chunk_fwd_matches_oracle(case):
    dt, B, H, Hkv, Lq, Lkv, D, qo, ko, causal = case
    q, k, v, _ = make(B, H, Hkv, Lq, D, dt, seed=3, device=DEV, S_kv=Lkv)
    Op, lp = dfa.dfa_chunk_attn_fwd(q, k, v, q_offset=qo, kv_offset=ko, causal=causal)
    dfa.dfa_check_errors()
    Or, lr = oracle.attn_fwd(np64(q), np64(k), np64(v), causal=causal, q_offset=qo, kv_offset=ko)
    check_fwd(Op, lp, Or, lr, dt, str(case))


def test_chunk_fwd_on_strided_views():
    """Chunks given as views into a larger [B, S, H, D] tensor (batch stride != chunk size)."""
    B, H, Hkv, S, D = 2, 4, 2, 512, 128
    for dt in (torch.float32, torch.bfloat16):
        q, k, v, _ = make(B, H, Hkv, S, D, dt, seed=5, device=DEV)
        qs, ks, vs = q[:, 256:384], k[:, 128:256], v[:, 128:256]
        Op, lp = dfa.dfa_chunk_attn_fwd(qs, ks, vs, q_offset=256, kv_offset=128)
        dfa.dfa_check_errors()
        Or, lr = oracle.attn_fwd(np64(qs), np64(ks), np64(vs), q_offset=256, kv_offset=128)
        check_fwd(Op, lp, Or, lr, dt, f"strided {dt}")


def test_merge_matches_oracle_including_empty_rows():
    g = torch.Generator(device=DEV).manual_seed(11)
    B, L, H, D = 2, 37, 3, 128
    Oa = torch.randn((B, L, H, D), generator=g, device=DEV)
    Ob = torch.randn((B, L, H, D), generator=g, device=DEV)
    la = torch.randn((B, H, L), generator=g, device=DEV) * 5
    lb = torch.randn((B, H, L), generator=g, device=DEV) * 5
    la[0, 0, :5] = -float("inf")
    lb[0, 0, 3:8] = -float("inf")
    Oa[0, :5, 0] = 0
    Ob[0, 3:8, 0] = 0
    Om, lm = dfa.dfa_merge_partials(Oa, la, Ob, lb)
    Or, lr = oracle.merge(np64(Oa), np64(la), np64(Ob), np64(lb))
    fin = np.isfinite(lr)
    assert np.array_equal(np.isfinite(np64(lm)), fin)
    assert np.max(np.abs(np64(lm)[fin] - lr[fin])) <= 1e-5
    assert np.max(np.abs(np64(Om) - Or)) <= 1e-5
    # In-place (O_out aliases O_a).
    Oa2, la2 = Oa.clone(), la.clone()
    dfa.dfa_merge_partials(Oa2, la2, Ob, lb, O_out=Oa2, lse_out=la2)
    torch.cuda.synchronize()
    assert torch.equal(Oa2, Om) and torch.equal(la2, lm)


@pytest.mark.parametrize("shape", [(1, 5, 3, 64), (1, 7, 2, 12), (2, 3, 1, 1032), (3, 333, 5, 128)])
def test_merge_row_groups_ragged_and_in_place(shape):
    # Rows shorter and longer than a warp's 128 floats, odd row counts, and
    # the output aliasing either input.
    B, L, H, D = shape
    g = torch.Generator(device=DEV).manual_seed(13)
    Oa = torch.randn((B, L, H, D), generator=g, device=DEV)
    Ob = torch.randn((B, L, H, D), generator=g, device=DEV)
    la = torch.randn((B, H, L), generator=g, device=DEV) * 3
    lb = torch.randn((B, H, L), generator=g, device=DEV) * 3
    lb[-1, -1, -1] = -float("inf")
    Or, lr = oracle.merge(np64(Oa), np64(la), np64(Ob), np64(lb))
    Om, lm = dfa.dfa_merge_partials(Oa, la, Ob, lb)
    torch.cuda.synchronize()
    assert np.max(np.abs(np64(lm) - lr)) <= 1e-5 and np.max(np.abs(np64(Om) - Or)) <= 1e-5
    for side in ("a", "b"):
        Oa2, la2, Ob2, lb2 = Oa.clone(), la.clone(), Ob.clone(), lb.clone()
        Od, ld = (Oa2, la2) if side == "a" else (Ob2, lb2)
        dfa.dfa_merge_partials(Oa2, la2, Ob2, lb2, O_out=Od, lse_out=ld)
        torch.cuda.synchronize()
        assert torch.equal(Od, Om) and torch.equal(ld, lm), f"in place on {side}"


# ---------------------------------------------------------------- whole-sequence, small shapes
SMALL = [
    # (dtype, B, H, Hkv, S, D, n_chunks)
    (torch.bfloat16, 1, 2, 2, 128, 128, 1),
    (torch.bfloat16, 1, 4, 2, 512, 128, 4),
    (torch.bfloat16, 2, 4, 1, 384, 64, 3),
    (torch.bfloat16, 1, 2, 2, 1000, 128, 8),    # ragged last tile
    (torch.bfloat16, 1, 3, 3, 1, 128, 1),       # single token
    (torch.bfloat16, 1, 8, 2, 1536, 128, 6),
    (torch.float32, 1, 2, 1, 640, 128, 5),
    (torch.float32, 2, 2, 2, 129, 64, 1),
]


@pytest.mark.parametrize("case", SMALL)
def test_whole_sequence_matches_oracle(case):
    dt, B, H, Hkv, S, D, P = case
    q, k, v, do = make(B, H, Hkv, S, D, dt, seed=7, device=DEV)
    O, lse, grads = run_fwd_bwd(q, k, v, do, n_chunks=P)
    Or, lr = oracle.attn_fwd(np64(q), np64(k), np64(v))
    check_fwd(O, lse, Or, lr, dt, str(case))
    ref = oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do))
    check_grads(grads, ref, dt, str(case))


@pytest.mark.parametrize("k_scale", [2.0, 4.0])
def test_sharp_softmax_exercises_the_lazy_rescale(k_scale):
    """Large score ranges make the running max jump late in a row, so some rows
    of a warp rescale their output accumulator while others do not."""
    q, k, v, do = make(1, 4, 1, 2048, 128, torch.bfloat16, seed=23, device=DEV, k_scale=k_scale)
    O, lse, grads = run_fwd_bwd(q, k, v, do, n_chunks=4)
    Or, lr = oracle.attn_fwd(np64(q), np64(k), np64(v))
    check_fwd(O, lse, Or, lr, torch.bfloat16, f"k x{k_scale}")
    check_grads(grads, oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do)), torch.bfloat16, f"k x{k_scale}")


def test_non_causal_whole_sequence():
    q, k, v, do = make(1, 2, 1, 384, 128, torch.bfloat16, seed=9, device=DEV)
    O, lse, grads = run_fwd_bwd(q, k, v, do, causal=False)
    Or, lr = oracle.attn_fwd(np64(q), np64(k), np64(v), causal=False)
    check_fwd(O, lse, Or, lr, torch.bfloat16, "non-causal")
    check_grads(grads, oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do), causal=False),
                torch.bfloat16, "non-causal")


# ---------------------------------------------------------------- contract properties
def test_backward_reuses_saved_outputs_and_never_runs_the_forward():
    """Rematerialization-aware checkpointing (DISTFLASHATTN §3.3): the backward reads the
    saved O/lse; a repeated forward gives the same bits, so results do not depend on it."""
    q, k, v, do = make(1, 4, 2, 768, 128, torch.bfloat16, seed=13, device=DEV)
    O1, l1 = dfa.dfa_attn_fwd(q, k, v, n_chunks=3)
    O2, l2 = dfa.dfa_attn_fwd(q, k, v, n_chunks=3)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(l1, l2)
    before = dfa.dfa_launch_count("fwd")
    dfa.dfa_attn_bwd(q, k, v, O1, l1, do, n_chunks=3)
    dfa.dfa_check_errors()
    assert dfa.dfa_launch_count("fwd") == before


def test_ragged_last_chunk_changes_only_the_decomposition():
    # S = 1000 in 3 chunks (334, 334, 332) and in 7 (143 x 6, 142): n_chunks
    # never changes the result, so the bits equal those of one chunk.
    q, k, v, do = make(1, 4, 2, 1000, 128, torch.bfloat16, seed=19, device=DEV)
    O1, l1 = dfa.dfa_attn_fwd(q, k, v, n_chunks=1)
    g1 = dfa.dfa_attn_bwd(q, k, v, O1, l1, do, n_chunks=1)
    for P in (3, 7):
        O, l = dfa.dfa_attn_fwd(q, k, v, n_chunks=P)
        g = dfa.dfa_attn_bwd(q, k, v, O, l, do, n_chunks=P)
        dfa.dfa_check_errors()
        assert torch.equal(O, O1) and torch.equal(l, l1), P
        assert torch.equal(g[1], g1[1]) and torch.equal(g[2], g1[2]), P
    with pytest.raises(dfa.DfaError) as e:   # S = 9 in 4 chunks of 3 leaves the last one empty
        dfa.dfa_attn_fwd(q[:, :9].contiguous(), k[:, :9].contiguous(), v[:, :9].contiguous(), n_chunks=4)
    assert e.value.status == dfa.DFA_ERR_INVALID_ARG


def test_schedules_give_the_same_forward_bits():
    q, k, v, do = make(1, 8, 2, 2048, 128, torch.bfloat16, seed=17, device=DEV)
    Ob, lb = dfa.dfa_attn_fwd(q, k, v, n_chunks=4, sched="balanced")
    Ou, lu = dfa.dfa_attn_fwd(q, k, v, n_chunks=4, sched="unbalanced")
    torch.cuda.synchronize()
    assert torch.equal(Ob, Ou) and torch.equal(lb, lu)
    gb = dfa.dfa_attn_bwd(q, k, v, Ob, lb, do, n_chunks=4, sched="balanced")
    gu = dfa.dfa_attn_bwd(q, k, v, Ob, lb, do, n_chunks=4, sched="unbalanced")
    dfa.dfa_check_errors()
    assert torch.equal(gb[1], gu[1]) and torch.equal(gb[2], gu[2])   # dK, dV: one CTA per key tile
    assert torch.max(torch.abs(gb[0].float() - gu[0].float())).item() <= 2e-2


def test_n_chunks_does_not_change_the_result():
    q, k, v, _ = make(1, 4, 4, 1024, 128, torch.bfloat16, seed=19, device=DEV)
    outs = [dfa.dfa_attn_fwd(q, k, v, n_chunks=P) for P in (1, 2, 4, 8)]
    torch.cuda.synchronize()
    for O, l in outs[1:]:
        assert torch.equal(O, outs[0][0]) and torch.equal(l, outs[0][1])
