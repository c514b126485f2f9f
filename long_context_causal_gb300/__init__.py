"""GB300-native causal chunk attention (DISTFLASHATTN hot path).

``long_context_causal_gb300.dfa`` is the Python binding of the C-ABI library
``libdfa.so`` (built from ``csrc/`` by ``__graft_entry__.build()``);
``long_context_causal_gb300.inputs`` draws the seeded synthetic workloads.
Importing the package itself loads nothing.
"""
