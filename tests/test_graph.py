"""The whole-sequence forward and backward run inside a CUDA graph.

After one eager call has built and cached the work lists (pinned host memory),
a call enqueues only stream work: the work-list copy from pinned memory, the
accumulator clears and the kernel launches, all of which can be captured.  A
captured fwd + bwd step replayed on new inputs gives the results of the eager
calls: the same bits for O, lse, dK and dV (one CTA owns each output row), and
dQ within the bf16 gradient tolerance (its fp32 partials are added by atomics
in no fixed order).
"""
import pytest
import torch

from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import make

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(1, 4, 2, 2048, 128), (2, 2, 2, 768, 64)])
def test_captured_fwd_bwd_replays_match_eager_calls(shape):
    B, H, Hkv, S, D = shape
    q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=73, device="cuda")
    O, lse = torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    dQ, dK, dV = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsf = dfa.workspace(B, H, Hkv, S, D, 2, False)
    wsb = dfa.workspace(B, H, Hkv, S, D, 2, True)

    def step():
        dfa.dfa_attn_fwd(q, k, v, n_chunks=2, O=O, lse=lse, workspace_buf=wsf)
        dfa.dfa_attn_bwd(q, k, v, O, lse, do, n_chunks=2, dQ=dQ, dK=dK, dV=dV, workspace_buf=wsb)

    step()                                   # eager: builds and caches the work lists
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                               # warm-up on the side stream, as capture requires
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (79, 83):
        nq, nk, nv, ndo = make(B, H, Hkv, S, D, torch.bfloat16, seed=seed, device="cuda")
        for dst, src in ((q, nq), (k, nk), (v, nv), (do, ndo)):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (O, lse, dQ, dK, dV)]
        step()
        dfa.dfa_check_errors()
        for name, a, b in zip(("O", "lse", "dK", "dV"), (got[0], got[1], got[3], got[4]), (O, lse, dK, dV)):
            assert torch.equal(a, b), f"{name} differs between the replay and the eager call"
        scale = torch.max(torch.abs(dQ.float())).item()
        assert torch.max(torch.abs(got[2].float() - dQ.float())).item() <= 2e-2 * scale
