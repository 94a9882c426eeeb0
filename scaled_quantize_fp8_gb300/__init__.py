"""GB300-native FP8 linear layer: quantize-cast kernels (delayed, tensorwise, MXFP8,
blockwise) and scaled FP8 GEMMs on the sm_103a tensor core, behind a C ABI
(include/fp8lin.h). This package is the build step plus a thin Python binding."""
from . import _lib  # noqa: F401
from .binding import (  # noqa: F401
    DelayedState, QTensor, Recipe, amax_update, dgelu_quantize, empty_qtensor, gelu_quantize,
    linear_bwd, linear_dgrad_dgelu, linear_fwd, linear_fwd_gelu, quantize, quantize_group,
    quantize_master, quantize_static_scratch, workspace_bytes,
)
