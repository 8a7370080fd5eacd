"""GB300 (sm_103a) query-aware block-sparse paged decode attention.

The compute lives in the CUDA library ``_lib/libhs.so`` (C ABI: ``include/hs.h``);
this package is its ctypes binding plus a small decode-step driver.
"""

from . import hs  # noqa: F401  (fails loudly when the library is not built)
from .hs import (  # noqa: F401
    HSError,
    attn_params,
    attn_shape,
    hot_buffer,
    hs_build_block_summaries,
    hs_get_device_error,
    hs_quantize_e4m3_g32,
    hs_score_select_topk,
    hs_sparse_paged_decode_attn,
    hs_status_string,
    hs_swapin_misses,
    hs_version,
    hs_workspace_bytes,
    paged_kv,
    select_params,
)
