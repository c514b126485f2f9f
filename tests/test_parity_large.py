"""Parity at the full workload sizes, in the launch configuration bench.py times.

The oracle cannot run these sizes in full, so for two heads per workload it
checks sampled query rows (O, lse and dQ; a row needs only the keys at or
before it) and sampled key rows near the end of the sequence (dK, dV; a key
needs only the query rows at or after it), including rows 0, S-1 and the rows
either side of every chunk boundary.  On every head, properties that hold at
any size are checked too:
  sum_j dV_j = sum_i dO_i,   sum_j dK_j = 0,   <Q, dQ> = <K, dK>,   <V, dV> = <O, dO>
(per GQA group; they follow from sum_j P_ij = 1 and sum_j dS_ij = 0).
Tolerances: O 2e-2 abs, lse 1e-3 abs, gradients 3e-2 x max|reference| (bf16 I/O);
the invariants to 2e-2 of the magnitude of their terms.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import WORKLOADS, make_workload

pytestmark = pytest.mark.gpu


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def sample_rows(w, rng, n=24):
    C = w.chunk
    rows = {0, w.S - 1}
    for p in range(1, w.n_chunks):
        rows.update({p * C - 1, p * C})
    rows.update(rng.integers(0, w.S, n).tolist())
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["llama7b_s32k", "llama7b_gqa8_s64k", "llama7b_s128k", "llama7b_s512k"])
def test_workload_sampled_rows_and_invariants(name):
    w = WORKLOADS[name]
    q, k, v, do = make_workload(w, "cuda")
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=w.n_chunks, scale=w.scale, sched="balanced")
    dQ, dK, dV = dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=w.n_chunks, scale=w.scale, sched="balanced")
    dfa.dfa_check_errors()
    G = w.H // w.H_kv
    rng = np.random.default_rng(1)

    # ---- sampled rows of two heads (the second one in another GQA group)
    for h in (0, w.H - 1):
        g = h // G
        heads = list(range(g * G, (g + 1) * G))
        hq = heads.index(h)
        qh = np64(q[:, :, heads])
        kh, vh = np64(k[:, :, g:g + 1]), np64(v[:, :, g:g + 1])
        doh = np64(do[:, :, heads])
        rows = sample_rows(w, rng)
        idx = np.stack([np.zeros_like(rows), np.full_like(rows, hq), rows], 1)
        Or, lr = oracle.attn_fwd_rows(qh, kh, vh, idx, scale=w.scale)
        dqr = oracle.attn_dq_rows(qh, kh, vh, doh, idx, scale=w.scale)
        Og = np64(O[0, rows, h])
        lg = np64(lse[0, h, rows])
        dqg = np64(dQ[0, rows, h])
        assert np.max(np.abs(Og - Or)) <= 2e-2, f"{name} h{h}: O"
        assert np.max(np.abs(lg - lr)) <= 1e-3, f"{name} h{h}: lse"
        assert np.max(np.abs(dqg - dqr)) <= 3e-2 * np.max(np.abs(dqr)), f"{name} h{h}: dQ"
        keys = np.unique(np.concatenate([[w.S - 1, w.S - 128, w.S - 129],
                                         rng.integers(w.S - 512, w.S, 5)]))
        kidx = np.stack([np.zeros_like(keys), np.zeros_like(keys), keys], 1)
        dkr, dvr = oracle.attn_dkv_rows(qh, kh, vh, doh, kidx, scale=w.scale)
        dkg, dvg = np64(dK[0, keys, g]), np64(dV[0, keys, g])
        assert np.max(np.abs(dkg - dkr)) <= 3e-2 * np.max(np.abs(dkr)), f"{name} g{g}: dK"
        assert np.max(np.abs(dvg - dvr)) <= 3e-2 * np.max(np.abs(dvr)), f"{name} g{g}: dV"

    # ---- invariants on every head / group (fp64 reductions of the GPU results)
    d = lambda t: t.double()
    for g in range(w.H_kv):
        hs = slice(g * G, (g + 1) * G)
        sdv, sdo = d(dV[0, :, g]).sum(0), d(do[0, :, hs]).sum((0, 1))
        assert (sdv - sdo).abs().max() <= 2e-2 * d(do[0, :, hs]).abs().sum((0, 1)).max() / np.sqrt(w.S)
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
