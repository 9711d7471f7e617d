"""Seeded synthetic inputs for the Flint MoE decode/prefill path.

This package is the only code shared by the CUDA path's tests/benchmark and the
CPU oracle.  It draws random tensors with the distributions of the workloads
(shapes, value distributions, seeds) and holds none of the method's arithmetic:
no dequantisation, no GEMV, no routing, no rounding.
"""

from .flint_synth import (  # noqa: F401
    CONFIGS,
    H,
    E,
    N_SHARED,
    INTER,
    TOP_K,
    N_LAYERS,
    config_seed,
    gen_dense,
    gen_dense_x,
    gen_layer,
    gen_x,
)
