"""Seeded synthetic inputs for the BitLinear W1.58A8 forward.

This package is shared by the oracle's tests, the GPU parity tests and the
benchmark. It draws random tensors and names workloads; it performs none of
the method's arithmetic (no scale, no rounding, no quantisation, no packing).
"""

from .synth import (  # noqa: F401
    WORKLOADS,
    Projection,
    Workload,
    gaussian_weights,
    student_t_weights,
    gaussian_activations,
    outlier_activations,
    make_projection_inputs,
)
