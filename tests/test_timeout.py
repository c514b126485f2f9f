"""Failure detection on the GPU without a fault: a kernel whose bounded
mbarrier waits run out (nothing ever arrives) gives up after the limit, raises
the device error flag and returns; the host reads DFA_ERR_TIMEOUT from
dfa_check_errors(), the flag is cleared, and the context keeps working."""
import time

import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gb300 import dfa
from long_context_causal_gb300.inputs import make

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    out = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    t0 = time.time()
    dfa.dfa_debug_wait_timeout(out)
    with pytest.raises(dfa.DfaError) as e:
        dfa.dfa_check_errors()
    elapsed = time.time() - t0
    assert e.value.status == dfa.DFA_ERR_TIMEOUT
    assert out.tolist() == [0, 0], "both waits gave up"
    assert 3.0 < elapsed < 30.0, elapsed   # the 4 s limit, not an endless spin
    dfa.dfa_check_errors()                 # the flag was cleared
    q, k, v, do = make(1, 2, 2, 256, 128, torch.bfloat16, seed=3, device="cuda")
    O, lse = dfa.dfa_attn_fwd(q, k, v)
    dfa.dfa_check_errors()
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    Or, lr = oracle.attn_fwd(f(q), f(k), f(v))
    assert np.max(np.abs(f(O) - Or)) <= 2e-2
    assert np.max(np.abs(f(lse) - lr)) <= 1e-3
