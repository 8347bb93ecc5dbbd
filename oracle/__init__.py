"""CPU oracle of the MoE SwiGLU layer (Mixture-of-Kittens articles), in NumPy float64.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it. The library's own path never does: it
shares no code with the CUDA kernels, and the CUDA kernels never call back into it.

Modules:
* ``numerics``: bf16 rounding, E4M3 encode/decode, MXFP8 block quantisation, SwiGLU.
* ``moe``: router, schedule table, forward, backward, router backward, shared expert,
  a per-token brute-force evaluator and a finite-difference loss.
* ``sampled``: single-output evaluators (one token's y or dX row, one dW element) for
  full-size workloads the dense oracle cannot hold.

Every function is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py``
(brute force, closed forms, library routines, finite differences, invariants). The pages
print no per-element values, so no pin comes from them directly; the one number they do
print for this path (the two-wave minibatch of 2368 tokens) pins the host planner.
"""
from . import numerics, moe  # noqa: F401
