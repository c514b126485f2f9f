"""Repeated calls give the same bits where one CTA owns each output row.

O and lse of every forward, and dK, dV of the BALANCED, local-window and
packed-batch backwards, are written by the CTA that owns the row, so repeated
calls on the same inputs return identical bits; a difference would point at
a race (a stale tile in the K/V ring, a P/dS buffer reused too early).  dQ,
and dK, dV of a SPLIT_KV backward, add fp32 partials with atomics in no fixed
order: they must stay finite and agree to within a few bf16 ulps.
"""
import numpy as np
import pytest
import torch

from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import make

pytestmark = pytest.mark.gpu
REPS = 25


def run(kind, q, k, v, do, **kw):
    if kind == "varlen":
        O, lse = dfa.dfa_attn_fwd_varlen(q, k, v, kw["cu"])
        return (O, lse, *dfa.dfa_attn_bwd_varlen(q, k, v, O, lse, do, kw["cu"]))
    if kind == "local":
        O, lse = dfa.dfa_attn_fwd_local(q, k, v, n_chunks=kw["P"], window=kw["w"])
        return (O, lse, *dfa.dfa_attn_bwd_local(q, k, v, O, lse, do, n_chunks=kw["P"], window=kw["w"]))
    O, lse = dfa.dfa_attn_fwd(q, k, v, sched=kind)
    return (O, lse, *dfa.dfa_attn_bwd(q, k, v, O, lse, do, sched=kind))


CASES = [
    ("balanced", (1, 4, 2, 2000, 128), {}),
    ("balanced", (2, 4, 1, 1100, 64), {}),
    ("unbalanced", (1, 2, 2, 1500, 128), {}),
    ("split_kv", (1, 1, 1, 16384, 128), {}),
    ("local", (1, 2, 1, 2300, 128), {"P": 5, "w": 2}),
    ("varlen", [300, 1, 0, 1500, 129], {"H": 4, "Hkv": 2, "D": 128}),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{i}" for i, c in enumerate(CASES)])
def test_repeated_calls_are_reproducible(case):
    kind, shp, kw = case
    if kind == "varlen":
        q, k, v, do = (t[0] for t in make(1, kw["H"], kw["Hkv"], sum(shp), kw["D"], torch.bfloat16,
                                          seed=107, device="cuda"))
        kw = dict(kw, cu=np.concatenate([[0], np.cumsum(shp)]).astype(np.int32))
    else:
        q, k, v, do = make(*shp, torch.bfloat16, seed=107, device="cuda")
    first = [t.clone() for t in run(kind, q, k, v, do, **kw)]
    atomic = {2} | ({3, 4} if kind == "split_kv" else set())
    for _ in range(REPS):
        out = run(kind, q, k, v, do, **kw)
        dfa.dfa_check_errors()
        for i, (a, b) in enumerate(zip(out, first)):
            assert bool(torch.isfinite(a.float()).all()), f"{kind}: output {i} not finite"
            if i in atomic:
                scale = max(torch.max(torch.abs(b.float())).item(), 1e-3)
                assert torch.max(torch.abs(a.float() - b.float())).item() <= 1e-2 * scale
            else:
                assert torch.equal(a, b), f"{kind}: output {i} differs between repeated calls"
