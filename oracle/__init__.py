"""fp64 CPU oracle for chunked causal linear attention (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

It also holds the causal softmax attention of a query segment over its
gathered key/value prefix (``softmax_segment_fwd`` and its gradients
``softmax_segment_bwd``: the standard-attention layers of the hybrid variant).

Every linear-attention function takes numpy arrays shaped ``[B, H, T, d]`` (any float dtype; they
are widened to float64) and per-head decays ``lam`` shaped ``[H]`` or
``[B, H]`` (``None`` means lambda = 1), and returns float64 arrays.

Parity pins: every function here is pinned in ``tests/test_oracle_pins.py``
(exact rational examples, brute force, autograd, closed forms and invariants).
"""
from .oracle import (  # noqa: F401
    build,
    fwd_recurrent,
    bwd_recurrent,
    fwd_chunked,
    bwd_chunked,
    fwd_quadratic,
    bwd_quadratic,
    segment_states,
    segment_grad_states,
    fwd_gated,
    bwd_gated,
    fwd_gated_vec,
    bwd_gated_vec,
    state_scan,
    threads_used,
)
from .softmax_oracle import softmax_segment_bwd, softmax_segment_fwd  # noqa: F401
