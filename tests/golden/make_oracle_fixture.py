"""Writes oracle_tiny_causal.json: a small seeded case and the oracle's outputs.

Calls only the fp64 oracle (no CUDA code).  The fixture guards the oracle
against accidental change; its correctness is pinned separately by the finite
difference, closed-form and library checks in tests/test_oracle.py.
Run from the repository root:  python tests/golden/make_oracle_fixture.py
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402

rng = np.random.default_rng(2310)
B, S, H, Hkv, D = 1, 5, 2, 1, 3
scale = 0.5
q = np.round(rng.standard_normal((B, S, H, D)), 3)
k = np.round(rng.standard_normal((B, S, Hkv, D)), 3)
v = np.round(rng.standard_normal((B, S, Hkv, D)), 3)
dO = np.round(rng.standard_normal((B, S, H, D)), 3)
O, lse = oracle.attn_fwd(q, k, v, scale=scale)
dQ, dK, dV = oracle.attn_bwd(q, k, v, dO, scale=scale)
out = {"what": "causal GQA attention, B=1 S=5 H=2 H_kv=1 D=3, scale 0.5; outputs from the fp64 oracle",
       "scale": scale}
for name, a in (("q", q), ("k", k), ("v", v), ("dO", dO), ("O", O), ("lse", lse), ("dQ", dQ), ("dK", dK), ("dV", dV)):
    out[name] = a.tolist()
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_causal.json"), "w") as f:
    json.dump(out, f, indent=1)
