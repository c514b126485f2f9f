"""Parity at the full workload sizes, in the launch configuration bench.py times.

The workloads are the DISTFLASHATTN evaluation lengths on the Llama-7B head
shape (abstract and §4.1: 32K to 512K tokens, and a GQA variant).  The oracle
cannot run them in full, so it checks what it can compute row by row:

* every head: 64 seeded random query rows plus rows 0, S-1 and the rows either
  side of every chunk boundary, for O, lse and dQ (a query row needs only the
  keys at or before it, and its own lse and Delta);
* the 32K and GQA 64K workloads: every query row of two heads (the first and
  the last, in different GQA groups) for O and lse, the full oracle;
* two key/value heads: sampled key rows in the last 512 positions for dK and
  dV (a key row needs only the query rows at or after it, passed to the oracle
  as a tail slice with its query offset);
* every head: properties that hold at any size,
    sum_j dV_j = sum_i dO_i,  sum_j dK_j = 0,  <Q, dQ> = <K, dK>,  <V, dV> = <O, dO>
  (per GQA group; they follow from sum_j P_ij = 1 and sum_j dS_ij = 0).

Each head is copied to the host on its own.  Query and dO rows that the
sampled checks do not read are left zero, so only the sampled rows are moved.
Tolerances: O 2e-2 abs, lse 1e-3 abs, gradients 3e-2 x max|reference| (bf16
I/O); the invariants to 2e-2 of the magnitude of their terms.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import WORKLOADS, make_workload

RANDOM_ROWS = 64
FULL_ROW_WORKLOADS = ("llama7b_s32k", "llama7b_gqa8_s64k")
KEY_TAIL = 512


def head64(t, h):
    """Head h of a [1, S, heads, D] device tensor as fp64 numpy [1, S, 1, D]."""
    return t[:, :, h:h + 1].double().cpu().numpy()


def rows64(t, h, rows, S):
    """fp64 [1, S, 1, D] holding head h of t at `rows` and zeros elsewhere."""
    a = np.zeros((1, S, 1, t.shape[-1]))
    idx = torch.as_tensor(rows, device=t.device)
    a[0, rows, 0] = t[0, idx, h].double().cpu().numpy()
    return a


def sample_rows(w, rng):
    C = -(-w.S // w.n_chunks)
    rows = {0, w.S - 1}
    for p in range(1, w.n_chunks):
        rows.update({p * C - 1, p * C})
    rows.update(rng.integers(0, w.S, RANDOM_ROWS).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def gathered(t, rows, h):
    return t[0, torch.as_tensor(rows, device=t.device), h].double().cpu().numpy()


def check_workload(w, full_rows, q, k, v, do, O, lse, dQ, dK, dV):
    """Every check above on one workload's inputs and results (any device)."""
    name = w.name
    dev = q.device
    G = w.H // w.H_kv
    S = w.S
    rng = np.random.default_rng(1)

    for g in range(w.H_kv):
        kh, vh = head64(k, g), head64(v, g)
        for h in range(g * G, (g + 1) * G):
            # ---- O, lse, dQ on sampled rows of this head
            rows = sample_rows(w, rng)
            idx = np.stack([np.zeros_like(rows), np.zeros_like(rows), rows], 1)
            qh, doh = rows64(q, h, rows, S), rows64(do, h, rows, S)
            Or, lr = oracle.attn_fwd_rows(qh, kh, vh, idx, scale=w.scale)
            dqr = oracle.attn_dq_rows(qh, kh, vh, doh, idx, scale=w.scale)
            Og, dqg = gathered(O, rows, h), gathered(dQ, rows, h)
            lg = lse[0, h, torch.as_tensor(rows, device=dev)].double().cpu().numpy()
            assert np.max(np.abs(Og - Or)) <= 2e-2, f"{name} h{h}: O"
            assert np.max(np.abs(lg - lr)) <= 1e-3, f"{name} h{h}: lse"
            assert np.max(np.abs(dqg - dqr)) <= 3e-2 * np.max(np.abs(dqr)), f"{name} h{h}: dQ"

            # ---- every row of two heads: the full oracle for O and lse
            if full_rows and h in (0, w.H - 1):
                allr = np.arange(S, dtype=np.int64)
                aidx = np.stack([np.zeros_like(allr), np.zeros_like(allr), allr], 1)
                Of, lf = oracle.attn_fwd_rows(head64(q, h), kh, vh, aidx, scale=w.scale)
                assert np.max(np.abs(O[0, :, h].double().cpu().numpy() - Of)) <= 2e-2, f"{name} h{h}: O all rows"
                assert np.max(np.abs(lse[0, h].double().cpu().numpy() - lf)) <= 1e-3, f"{name} h{h}: lse all rows"

        # ---- dK, dV on sampled key rows near the end, for two key/value heads
        if g in (0, w.H_kv - 1):
            T = KEY_TAIL
            keys = np.unique(np.concatenate([[S - 1, S - 128, S - 129], rng.integers(S - T, S, 5)]))
            kidx = np.stack([np.zeros_like(keys), np.zeros_like(keys), keys], 1)
            heads = slice(g * G, (g + 1) * G)
            q_tail = q[:, S - T:, heads].double().cpu().numpy()
            do_tail = do[:, S - T:, heads].double().cpu().numpy()
            dkr, dvr = oracle.attn_dkv_rows(q_tail, kh, vh, do_tail, kidx, scale=w.scale, q_offset=S - T)
            kt = torch.as_tensor(keys, device=dev)
            dkg, dvg = dK[0, kt, g].double().cpu().numpy(), dV[0, kt, g].double().cpu().numpy()
            assert np.max(np.abs(dkg - dkr)) <= 3e-2 * np.max(np.abs(dkr)), f"{name} g{g}: dK"
            assert np.max(np.abs(dvg - dvr)) <= 3e-2 * np.max(np.abs(dvr)), f"{name} g{g}: dV"
        del kh, vh

    # ---- invariants on every head / group (fp64 reductions of the GPU results)
    d = lambda t: t.double()
    for g in range(w.H_kv):
        hs = slice(g * G, (g + 1) * G)
        sdv, sdo = d(dV[0, :, g]).sum(0), d(do[0, :, hs]).sum((0, 1))
        assert (sdv - sdo).abs().max() <= 2e-2 * d(do[0, :, hs]).abs().sum((0, 1)).max() / np.sqrt(S)
        sdk = d(dK[0, :, g]).sum(0)
        assert sdk.abs().max() <= 2e-2 * d(dK[0, :, g]).abs().sum(0).max()
        qdq = (d(q[0, :, hs]) * d(dQ[0, :, hs])).sum()
        kdk = (d(k[0, :, g]) * d(dK[0, :, g])).sum()
        mag = (d(q[0, :, hs]) * d(dQ[0, :, hs])).abs().sum()
        assert (qdq - kdk).abs() <= 2e-2 * mag
        vdv = (d(v[0, :, g]) * d(dV[0, :, g])).sum()
        odo = (d(O[0, :, hs]) * d(do[0, :, hs])).sum()
        mag = (d(O[0, :, hs]) * d(do[0, :, hs])).abs().sum()
        assert (vdv - odo).abs() <= 2e-2 * mag


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["llama7b_s32k", "llama7b_gqa8_s64k", "llama7b_s128k", "llama7b_s512k"])
def test_workload_rows_of_every_head_and_invariants(name):
    w = WORKLOADS[name]
    q, k, v, do = make_workload(w, "cuda")
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=w.n_chunks, scale=w.scale, sched="balanced")
    dQ, dK, dV = dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=w.n_chunks, scale=w.scale, sched="balanced")
    dfa.dfa_check_errors()
    check_workload(w, name in FULL_ROW_WORKLOADS, q, k, v, do, O, lse, dQ, dK, dV)


def test_the_full_size_checks_pass_exact_results_and_catch_a_wrong_head():
    """The checking code itself, on the CPU: with the oracle's own full
    results standing in for the kernels' (a small GQA workload with the
    production recipe), every check passes; with one head's dQ rows taken from
    another head, the per-head row check fails."""
    from long_context_causal_gb300.inputs import Workload
    w = Workload("small_gqa", 1, 4, 2, 1280, 64, 5, torch.float32, k_scale=2.0)
    q, k, v, do = make_workload(w, "cpu")
    f = lambda t: t.double().numpy()
    Or, lr = oracle.attn_fwd(f(q), f(k), f(v), scale=w.scale)
    dqr, dkr, dvr = oracle.attn_bwd(f(q), f(k), f(v), f(do), scale=w.scale)
    t = torch.from_numpy
    outs = [t(Or), t(lr), t(dqr), t(dkr), t(dvr)]
    check_workload(w, True, q, k, v, do, *outs)
    bad = outs[2].clone()
    bad[:, :, 3] = outs[2][:, :, 2]
    with pytest.raises(AssertionError, match="h3: dQ"):
        check_workload(w, True, q, k, v, do, outs[0], outs[1], bad, outs[3], outs[4])


@pytest.mark.gpu
def test_at_full_size_the_schedule_and_chunk_count_change_only_the_decomposition():
    """The 128K workload as the benchmark runs it (balanced list, 16 chunks)
    against the unbalanced list and against one chunk: the work decomposition
    changes, the result does not.  O, lse, dK and dV are the same bits (every
    output row is computed by one CTA in a fixed order); dQ adds fp32 partials
    with atomics in no fixed order and may differ in its last bits."""
    w = WORKLOADS["llama7b_s128k"]
    q, k, v, do = make_workload(w, "cuda")
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=w.n_chunks, scale=w.scale, sched="balanced")
    dQ, dK, dV = dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=w.n_chunks, scale=w.scale, sched="balanced")
    dq_max = dQ.float().abs().max().item()
    for sched, P in (("unbalanced", w.n_chunks), ("balanced", 1)):
        O2, l2 = dfa.dfa_attn_fwd(q, k, v, n_chunks=P, scale=w.scale, sched=sched)
        assert torch.equal(O2, O) and torch.equal(l2, lse), (sched, P)
        del O2, l2
        g = dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=P, scale=w.scale, sched=sched)
        assert torch.equal(g[1], dK) and torch.equal(g[2], dV), (sched, P)
        assert (g[0].float() - dQ.float()).abs().max().item() <= 1e-2 * dq_max, (sched, P)
        del g
    dfa.dfa_check_errors()
