"""CPU oracle (float64, NumPy).  Test infrastructure only: never imported by the
library, and never imports it."""
from .epilogue import (  # noqa: F401
    DEFAULT_ALPHA, DEFAULT_AXIS, DEFAULT_EPSILON,
    skip_layer_norm, skip_bias_sum,
    bias_softmax, bias_softmax_dims, bias_row_of,
    bias_add, quick_gelu,
)
