"""The pages' distributed method executed step by step on one GPU.

DISTFLASHATTN (§3.2, App. B): P workers own one token chunk each; at every
step a worker computes one (query chunk, key/value chunk) block of the causal
triangle, and under the balanced schedule an early worker helps a late one and
hands back a partial output with its log-sum-exp, which the owner merges.  The
backward (§3.3) runs the same blocks from the owners' final O and lse, and
each block's share of dQ goes to the query chunk's owner, of dK and dV to the
key/value chunk's owner.  Here the schedule comes from the host scheduler
(dfa_chunk_schedule), the blocks run through dfa_chunk_attn_fwd /
dfa_chunk_attn_bwd and the hand-backs through dfa_merge_partials; the result
must equal the whole-sequence calls and the fp64 oracle (bf16 tolerances of
test_parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import make

pytestmark = pytest.mark.gpu


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("sched", ["balanced", "unbalanced"])
def test_schedule_driven_chunk_steps_equal_the_whole_sequence(sched):
    B, H, Hkv, S, D, P = 1, 4, 2, 4096, 128, 8
    C = S // P
    q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=89, device="cuda")
    steps = dfa.dfa_chunk_schedule(P, sched)
    owner = {}                                   # query chunk -> merged (O_partial, lse) so far
    for s in range(steps.shape[0]):
        for w in range(P):
            blk = int(steps[s, w])
            if blk < 0:
                continue
            qc, kc = divmod(blk, P)
            assert w in (qc, P - 1 - qc)         # the owner or its mirror helper
            part = dfa.dfa_chunk_attn_fwd(q[:, qc * C:(qc + 1) * C].contiguous(),
                                          k[:, kc * C:(kc + 1) * C].contiguous(),
                                          v[:, kc * C:(kc + 1) * C].contiguous(),
                                          q_offset=qc * C, kv_offset=kc * C)
            owner[qc] = part if qc not in owner else dfa.dfa_merge_partials(*owner[qc], *part)
    dfa.dfa_check_errors()
    assert sorted(owner) == list(range(P))
    O_chunks = torch.cat([owner[c][0] for c in range(P)], dim=1)
    lse_chunks = torch.cat([owner[c][1] for c in range(P)], dim=2)
    O, lse = dfa.dfa_attn_fwd(q, k, v, n_chunks=P)
    dfa.dfa_check_errors()
    assert torch.max(torch.abs(O_chunks - O.float())).item() <= 2e-2
    assert torch.max(torch.abs(lse_chunks - lse)).item() <= 1e-3
    Or, lr = oracle.attn_fwd(np64(q), np64(k), np64(v))
    assert np.max(np.abs(np64(O_chunks) - Or)) <= 2e-2
    assert np.max(np.abs(np64(lse_chunks) - lr)) <= 1e-3

    # Backward over the same blocks, from the owners' final O (bf16, as saved) and lse.
    O_saved = O_chunks.to(torch.bfloat16)
    f32 = dict(dtype=torch.float32, device="cuda")
    dQ = torch.zeros((B, S, H, D), **f32)
    dK = torch.zeros((B, S, Hkv, D), **f32)
    dV = torch.zeros((B, S, Hkv, D), **f32)
    for s in range(steps.shape[0]):
        for w in range(P):
            blk = int(steps[s, w])
            if blk < 0:
                continue
            qc, kc = divmod(blk, P)
            qs, ks = slice(qc * C, (qc + 1) * C), slice(kc * C, (kc + 1) * C)
            dq_c, dk_c, dv_c = dQ[:, qs], dK[:, ks], dV[:, ks]
            gq, gk, gv = dq_c.contiguous(), dk_c.contiguous(), dv_c.contiguous()
            dfa.dfa_chunk_attn_bwd(q[:, qs].contiguous(), k[:, ks].contiguous(), v[:, ks].contiguous(),
                                   O_saved[:, qs].contiguous(), lse_chunks[:, :, qs].contiguous(),
                                   do[:, qs].contiguous(), q_offset=qc * C, kv_offset=kc * C,
                                   dQ_acc=gq, dK_acc=gk, dV_acc=gv)
            dq_c.copy_(gq)
            dk_c.copy_(gk)
            dv_c.copy_(gv)
    dfa.dfa_check_errors()
    ref = oracle.attn_bwd(np64(q), np64(k), np64(v), np64(do))
    for name, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref):
        rel = np.max(np.abs(np64(g) - r)) / max(np.max(np.abs(r)), 1e-2)
        assert rel <= 3e-2, f"{sched}: {name} rel err {rel}"
