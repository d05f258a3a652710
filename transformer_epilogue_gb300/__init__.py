"""GB300-native fused transformer-block epilogue ops (SkipLayerNormalization,
BiasSoftmax, BiasAdd, QuickGelu): hand-written sm_103a CUDA kernels behind a C
ABI (``include/ep.h``), with a thin ctypes binding."""
from ._binding import (  # noqa: F401
    DEFAULT_ALPHA, DEFAULT_AXIS, DEFAULT_EPSILON,
    EP_F16, EP_F32, EP_BF16, EP_OK, EP_ERR_CUDA, EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED, EP_ERR_WORKSPACE,
    EpError, LIB_PATH, ep_bias_add, ep_bias_softmax, ep_bias_softmax_noalloc, ep_bias_softmax_workspace_size, ep_quick_gelu,
    ep_pipeline_timeouts, ep_selftest_bounded_wait, ep_skip_layer_norm, ep_skip_layer_norm_ex, kernel_launch_count, load_library, raw,
)
