"""Seeded synthetic inputs shared by the CPU oracle and the GPU harness.

This package holds no step of ResidualQuant itself: it only draws the looped
K/V states, queries and rotation signs that both sides consume.  Every value is
a function of (seed, field, coordinates) through the counter-based Philox4x32-10
generator followed by IEEE-754 fp32 operations that are correctly rounded on any
conforming machine (add, multiply, divide, square root), so the numpy version
here and the CUDA version inside the native library produce bit-identical
tensors.  The CUDA twin lives in the library's synthetic-input kernel; the two
are compared element by element in the test suite.
"""

from .philox import philox4x32_10  # noqa: F401
from .recipe import (  # noqa: F401
    Config,
    CONFIGS,
    config_by_name,
    outlier_channels,
    outlier_table,
    round_bf16_f32,
    rotation_signs,
    gen_states,
    gen_queries,
    FIELD_BASE,
    FIELD_NOISE,
    FIELD_U,
    FIELD_QUERY,
    FIELD_SIGN,
    FIELD_OUTLIER,
)
