"""GB300 (sm_103a) fused tiled attention: forward and 5-/7-GEMM backward.

``binding`` exposes the C ABI of ``include/fa.h`` under the same names;
``api`` wraps it for torch tensors.  The CUDA library is loaded on first use
and its absence is an error (there is no CPU path).
"""

from .binding import (  # noqa: F401
    FA_BWD_5GEMM, FA_BWD_7GEMM, FA_BWD_AUTO, FaError,
    fa_bwd, fa_bwd_choose, fa_bwd_launches, fa_bwd_workspace_size, fa_fwd,
    fa_fwd_launches, fa_get_device_error, fa_strerror,
)
from .api import attention_backward, attention_forward, check_device_error  # noqa: F401
