"""fp64 CPU oracle of the selective-scan (S6) hot path and of the multi-head SSM with one decay
per head (the state-space-duality layer).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline may import this package; the library in ``selective_state_space_145_b300``
never does, and this package never imports it.
"""

from .oracle import (  # noqa: F401
    causal_conv1d,
    causal_conv1d_bwd,
    chunk_aggregates,
    compose,
    selective_scan,
    selective_scan_bwd,
    silu,
    softplus,
    ssd,
    state_update,
)
