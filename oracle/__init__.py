"""CPU oracle for the BitLinear W1.58A8 forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline arm may import
this package. The product path (the CUDA library and its Python binding) never
imports, links or executes anything here, and this package shares no code with
it: the only module both sides use is the seeded input generator package
``workloads``, which performs none of the method's arithmetic.
"""

from .bitlinear_oracle import (  # noqa: F401
    EPS_ABSMAX,
    EPS_GAMMA,
    absmean_gamma,
    bf16_bits_to_f32,
    bitlinear_forward,
    exact_abs_sum,
    pack_codes,
    quant_act,
    rescale,
    round_ratio_to_f32,
    ternary_codes,
    ternary_int8_matmul,
    unpack_codes,
)
from .quantizer_variants import (  # noqa: F401,E402
    DEFAULT_FACTOR,
    alpha_round_quantize,
    scaled_mean,
    threshold_quantize,
)
from .grouped import (  # noqa: F401,E402
    GROUP,
    bitlinear_forward_grouped,
    group_accumulators,
    group_codes,
    group_gammas,
    grouped_rescale,
    grouped_y_bound,
)
