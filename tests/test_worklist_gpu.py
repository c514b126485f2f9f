"""The persistent kernels process exactly the work list the host scheduler
built: per CTA, the tiles counted by the MMA issuer, the softmax / compute
warpgroup and the TMA producer equal the host's cost model for that worker's
items (read back through the per-CTA trace of include/dfa_debug.h)."""
import numpy as np
import pytest
import torch

from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import make

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sched", ["balanced", "unbalanced"])
@pytest.mark.parametrize("shape", [(1, 8, 2, 4096, 128), (2, 4, 4, 1536, 64)])
def test_kernels_follow_the_work_list(shape, sched):
    B, H, Hkv, S, D = shape
    q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=3, device="cuda")
    O, lse = dfa.dfa_attn_fwd(q, k, v, sched=sched)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(16 * 1024, dtype=torch.int64, device="cuda")
    for which in ("fwd", "bwd"):
        buf.zero_()
        dfa.dfa_debug_cta_trace(buf)
        try:
            if which == "fwd":
                dfa.dfa_attn_fwd(q, k, v, sched=sched, O=O, lse=lse)
            else:
                dfa.dfa_attn_bwd(q, k, v, O, lse, do, sched=sched)
            dfa.dfa_check_errors()
        finally:
            dfa.dfa_debug_cta_trace(None)
        r = buf.view(-1, 8).cpu().numpy()
        if which == "fwd":
            rows, units = B * H, (S + 255) // 256
            tiles = lambda u: 2 * u + 2                      # 256 query rows vs 128-key tiles
        else:
            rows, units = B * Hkv, (S + 127) // 128
            tiles = lambda u: (H // Hkv) * (u + 1)           # query tiles per key tile, all heads
        W = min(sms, rows * units)
        off, items, _ = dfa.dfa_build_worklist(rows, units, W, sched)
        cost = np.array([sum(tiles(int(i) % units) for i in items[off[w]:off[w + 1]]) for w in range(W)])
        assert np.array_equal(r[:W, 3], np.diff(off)), which
        for slot in (4, 5, 6):
            assert np.array_equal(r[:W, slot], cost), (which, slot)
