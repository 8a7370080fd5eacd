"""GB300 (sm_103a) query-aware block-sparse paged decode attention.

The compute lives in the CUDA library ``_lib/libhs.so`` (C ABI: ``include/hs.h``);
``query_aware_sparse_hs_gb300.hs`` is its ctypes binding (importing it fails
loudly when the library has not been built) and ``.decode`` a small decode-step
driver.  ``python -m query_aware_sparse_hs_gb300.build`` compiles the library.
"""

_BINDING = ("HSError", "attn_params", "attn_shape", "hot_buffer", "hs_build_block_summaries",
            "hs_get_device_error", "hs_quantize_e4m3_g32", "hs_score_select_topk",
            "hs_sparse_paged_decode_attn", "hs_status_string", "hs_swapin_misses", "hs_version",
            "hs_workspace_bytes", "paged_kv", "select_params")


def __getattr__(name):
    if name in _BINDING:
        from . import hs
        return getattr(hs, name)
    raise AttributeError(name)
