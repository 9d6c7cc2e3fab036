"""GB300-native sparse 3-D convolution: indice maps, strided output sets and
implicit-GEMM conv forward / dinput / dfilter, behind the C ABI of libspc.so.

``binding`` holds the Python functions, named after the C entry points; the
library is built in-tree by ``build.build()``.
"""

from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    SPC_MAP_SUBM_MIRROR,
    SPC_MAP_TRANSPOSED,
    SPC_PREC_EXACT,
    SPC_PREC_TF32,
    SpcError,
    SpcLibraryMissing,
    check_status,
    new_status,
    spc_build_indice_map,
    spc_conv_dgrad,
    spc_conv_fwd,
    spc_conv_fwd_fused,
    spc_conv_fwd_int8,
    spc_get_wait_limit_ns,
    spc_set_wait_limit_ns,
    SPC_ACT_NONE,
    SPC_ACT_RELU,
    spc_conv_inverse,
    spc_map_row_order,
    spc_maxpool_fwd,
    spc_maxpool_dgrad,
    spc_conv_wgrad,
    spc_out_shape,
    spc_strided_out_coords,
)
