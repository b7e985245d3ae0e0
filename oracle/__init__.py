"""CPU oracle for the causal depthwise conv1d forward pass (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg import this package; the CUDA library and its binding never do.
"""
