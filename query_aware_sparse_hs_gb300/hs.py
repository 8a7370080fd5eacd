"""ctypes binding of ``libhs.so`` (the C ABI declared in ``include/hs.h``).

Argument marshalling only: tensors become device pointers and sizes, the call
goes to the CUDA library, a non-OK status raises :class:`HSError`.  Every step
of the computation runs in the library's kernels; there is no fallback.  The
library is built by ``python -m query_aware_sparse_hs_gb300.build`` (or
``__graft_entry__.build()``); importing this module without it fails loudly.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_uint32, c_ulonglong, c_void_p

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libhs.so")

HS_OK, HS_ERR_INVALID_ARG, HS_ERR_UNSUPPORTED, HS_ERR_CUDA = 0, 1, 2, 3
HS_ERR_OUT_OF_RANGE, HS_ERR_CAPACITY, HS_ERR_TIMEOUT, HS_ERR_WORKSPACE = 4, 5, 6, 7
HS_ERR_SCRATCH_LIMIT = 8
HS_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024
HS_ATTN_EARLY_SUMMARIES = 1
HS_ATTN_RANGES = 2
HS_ATTN_NO_RANGES = 4
HS_EBIT_PAGE_RANGE, HS_EBIT_CAPACITY, HS_EBIT_TIMEOUT, HS_EBIT_BLOCK_RANGE = 0x1, 0x2, 0x4, 0x8
KV_DTYPES = {"f32": 0, "bf16": 1, "fp8": 2}
ALGO = {"auto": 0, "simt": 1, "tcgen05": 2}


class HSError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {hs_status_string(status)} (status {status})")


class AttnShape(ctypes.Structure):
    _fields_ = [("num_q_heads", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("block_size", c_int32), ("kv_dtype", c_int32)]


class PagedKV(ctypes.Structure):
    _fields_ = [("k_pages", c_void_p), ("v_pages", c_void_p), ("k_scales", c_void_p),
                ("v_scales", c_void_p), ("page_table", c_void_p), ("seq_lens", c_void_p),
                ("batch", c_int32), ("max_blocks", c_int32), ("num_pages", c_int64)]


class SelectParams(ctypes.Structure):
    _fields_ = [("sink_tokens", c_int32), ("window_tokens", c_int32), ("k_scored", c_int32),
                ("capacity", c_int32), ("history_weight", c_float), ("score_history", c_void_p)]


class AttnParams(ctypes.Structure):
    _fields_ = [("scale", c_float), ("out_is_fp32", c_int32), ("blocks_per_split", c_int32),
                ("algo", c_int32), ("max_ctas", c_int32), ("split_counters", c_void_p),
                ("wait_limit_ns", c_uint32), ("flags", c_uint32)]


class HotBuffer(ctypes.Structure):
    _fields_ = [("page_table", c_void_p), ("slot_owner", c_void_p), ("last_used", c_void_p),
                ("k_slots", c_void_p), ("v_slots", c_void_p), ("k_slot_scales", c_void_p),
                ("v_slot_scales", c_void_p), ("host_k", c_void_p), ("host_v", c_void_p),
                ("host_k_scales", c_void_p), ("host_v_scales", c_void_p), ("batch", c_int32),
                ("max_blocks", c_int32), ("slots_per_stream", c_int32)]


class SwapStats(ctypes.Structure):
    _fields_ = [("hits", c_ulonglong), ("misses", c_ulonglong), ("evictions", c_ulonglong),
                ("bytes_in", c_ulonglong)]


SYMBOLS = {
    "hs_status_string": (ctypes.c_char_p, [c_int32]),
    "hs_version": (c_int32, []),
    "hs_workspace_bytes": (c_size_t, [POINTER(AttnShape), c_int32, c_int32, POINTER(AttnParams)]),
    "hs_attn_geometry": (c_int32, [POINTER(AttnShape), c_int32, c_int32, POINTER(AttnParams),
                                   POINTER(c_int32), POINTER(c_int32)]),
    "hs_select_workspace_bytes": (c_size_t, [POINTER(AttnShape), c_int32, c_int32]),
    "hs_build_block_summaries": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_int32, c_void_p,
                                           c_void_p, c_void_p]),
    "hs_append_token": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p]),
    "hs_score_select_topk": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p, c_void_p,
                                       c_void_p, POINTER(SelectParams), c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_size_t, c_void_p]),
    "hs_sparse_paged_decode_attn": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p, c_void_p,
                                              c_void_p, c_int32, POINTER(AttnParams), c_void_p, c_void_p,
                                              c_void_p, c_size_t, c_void_p]),
    "hs_score_select_attend_workspace_bytes": (c_size_t, [POINTER(AttnShape), c_int32, c_int32, c_int32,
                                                          POINTER(AttnParams)]),
    "hs_score_select_attend_fused": (c_int32, [POINTER(AttnShape), c_int32, c_int32, c_int32,
                                               POINTER(AttnParams)]),
    "hs_score_select_attend": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p, c_void_p, c_void_p,
                                         POINTER(SelectParams), c_void_p, c_void_p, c_void_p, POINTER(AttnParams),
                                         c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "hs_decode_step": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, POINTER(SelectParams), c_void_p, c_void_p, c_void_p, POINTER(AttnParams),
                                 c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "hs_decode_step_reuse": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_int32, POINTER(AttnParams),
                                       c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "hs_sparse_paged_decode_attn_noalloc": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p,
                                                      c_void_p, c_void_p, c_int32, POINTER(AttnParams),
                                                      c_void_p, c_void_p, c_void_p]),
    "hs_swapin_misses": (c_int32, [POINTER(AttnShape), POINTER(HotBuffer), c_void_p, c_void_p, c_int32,
                                   c_int32, c_void_p, c_void_p]),
    "hs_swapin_plan": (c_int32, [POINTER(AttnShape), POINTER(HotBuffer), c_void_p, c_void_p, c_int32, c_int32,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "hs_score_select_swapin_plan": (c_int32, [POINTER(AttnShape), POINTER(PagedKV), c_void_p, c_void_p, c_void_p,
                                              POINTER(SelectParams), c_void_p, c_void_p, c_void_p, c_void_p,
                                              c_size_t, POINTER(HotBuffer), c_int32, c_void_p, c_void_p, c_void_p,
                                              c_void_p, c_void_p, c_void_p]),
    "hs_swapin_copy": (c_int32, [POINTER(AttnShape), POINTER(HotBuffer), c_void_p, c_void_p, c_int32, c_int32,
                                 c_void_p, c_void_p]),
    "hs_swapin_copy_attend": (c_int32, [POINTER(AttnShape), POINTER(HotBuffer), c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_int32, c_float, c_int32, c_void_p, c_void_p, c_void_p,
                                        c_void_p]),
    "hs_merge_attn_partials": (c_int32, [POINTER(AttnShape), c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                         c_int32, c_void_p, c_void_p]),
    "hs_quantize_e4m3_g32": (c_int32, [c_void_p, c_int32, c_int64, c_int32, c_void_p, c_void_p,
                                       c_void_p]),
    "hs_get_device_error": (c_int32, [c_void_p, POINTER(c_uint32)]),
    "hs_get_device_error_detail": (c_int32, [c_void_p, POINTER(c_uint32), POINTER(c_uint32)]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m query_aware_sparse_hs_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SYMBOLS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library():
    return _lib


def hs_status_string(status: int) -> str:
    return _lib.hs_status_string(int(status)).decode()


def hs_version() -> int:
    return int(_lib.hs_version())


def _check(status: int, where: str):
    if status != HS_OK:
        raise HSError(status, where)


def _ptr(t) -> int | None:
    if t is None or isinstance(t, int):  # None, or an address already
        return t
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_shape(num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype) -> AttnShape:
    return AttnShape(num_q_heads, num_kv_heads, head_dim, block_size,
                     KV_DTYPES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype))


def paged_kv(k_pages, v_pages, page_table, seq_lens, k_scales=None, v_scales=None) -> PagedKV:
    """Describe a paged cache: pages [num_pages][B][D], page_table [batch][Hkv][max_blocks]."""
    kv = PagedKV(_ptr(k_pages), _ptr(v_pages), _ptr(k_scales), _ptr(v_scales), _ptr(page_table),
                 _ptr(seq_lens), int(page_table.shape[0]), int(page_table.shape[-1]),
                 int(k_pages.shape[0]))
    kv._keep = (k_pages, v_pages, page_table, seq_lens, k_scales, v_scales)
    return kv


def select_params(sink_tokens, window_tokens, k_scored, capacity, history_weight=0.0,
                  score_history=None) -> SelectParams:
    p = SelectParams(sink_tokens, window_tokens, k_scored, capacity, float(history_weight), _ptr(score_history))
    p._keep = score_history
    return p


def attn_params(scale, out_is_fp32=False, blocks_per_split=0, algo="auto", max_ctas=0,
                split_counters=None, wait_limit_ns=0, early_summaries=False, ranges=None) -> AttnParams:
    """wait_limit_ns: bound of the tensor-core kernels' waits (0 = 2 s).
    early_summaries: HS_ATTN_EARLY_SUMMARIES (smin/smax are not written by the
    kernel launched just before the call on its stream).  ranges: True =
    HS_ATTN_RANGES, False = HS_ATTN_NO_RANGES, None = the library's choice."""
    flags = (HS_ATTN_EARLY_SUMMARIES if early_summaries else 0) | \
        {None: 0, True: HS_ATTN_RANGES, False: HS_ATTN_NO_RANGES}[ranges]
    p = AttnParams(float(scale), 1 if out_is_fp32 else 0, int(blocks_per_split),
                   ALGO[algo] if isinstance(algo, str) else int(algo), int(max_ctas), _ptr(split_counters),
                   int(wait_limit_ns), flags)
    p._keep = split_counters
    return p


def hs_workspace_bytes(shape: AttnShape, batch: int, capacity: int, params: AttnParams) -> int:
    return int(_lib.hs_workspace_bytes(ctypes.byref(shape), batch, capacity, ctypes.byref(params)))


def hs_attn_geometry(shape: AttnShape, batch: int, capacity: int, params: AttnParams):
    """(splits, chunks_per_cta) of the tensor-core attention; chunks_per_cta 0 = equal splits."""
    sp, per = c_int32(0), c_int32(0)
    if _lib.hs_attn_geometry(ctypes.byref(shape), batch, capacity, ctypes.byref(params), ctypes.byref(sp),
                             ctypes.byref(per)) != 0:
        raise HSError(HS_ERR_INVALID_ARG, "hs_attn_geometry")
    return sp.value, per.value


def hs_select_workspace_bytes(shape: AttnShape, batch: int, max_blocks: int) -> int:
    return int(_lib.hs_select_workspace_bytes(ctypes.byref(shape), batch, max_blocks))


def hs_build_block_summaries(shape, kv, first_block, smin, smax, stream=None):
    _check(_lib.hs_build_block_summaries(ctypes.byref(shape), ctypes.byref(kv), int(first_block),
                                         _ptr(smin), _ptr(smax), _stream(stream)),
           "hs_build_block_summaries")


def hs_append_token(shape, kv, new_k, new_v, smin, smax, stream=None):
    _check(_lib.hs_append_token(ctypes.byref(shape), ctypes.byref(kv), _ptr(new_k), _ptr(new_v), _ptr(smin),
                                _ptr(smax), _stream(stream)),
           "hs_append_token")


def hs_score_select_topk(shape, kv, q, smin, smax, params, sel, sel_count, scores=None,
                         workspace=None, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.hs_score_select_topk(ctypes.byref(shape), ctypes.byref(kv), _ptr(q), _ptr(smin),
                                     _ptr(smax), ctypes.byref(params), _ptr(sel), _ptr(sel_count),
                                     _ptr(scores), _ptr(workspace), ws_bytes, _stream(stream)),
           "hs_score_select_topk")


def hs_sparse_paged_decode_attn(shape, kv, q, sel, sel_count, capacity, params, out, lse=None,
                                workspace=None, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.hs_sparse_paged_decode_attn(ctypes.byref(shape), ctypes.byref(kv), _ptr(q), _ptr(sel),
                                            _ptr(sel_count), int(capacity), ctypes.byref(params),
                                            _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                            _stream(stream)),
           "hs_sparse_paged_decode_attn")


def hs_score_select_attend_workspace_bytes(shape: AttnShape, batch: int, max_blocks: int, capacity: int,
                                           params: AttnParams) -> int:
    return int(_lib.hs_score_select_attend_workspace_bytes(ctypes.byref(shape), batch, max_blocks, capacity,
                                                           ctypes.byref(params)))


def hs_score_select_attend_fused(shape: AttnShape, batch: int, max_blocks: int, capacity: int,
                                 params: AttnParams) -> int:
    """1: the combined call is one launch for this geometry on the current device; 0: separate launches."""
    return int(_lib.hs_score_select_attend_fused(ctypes.byref(shape), batch, max_blocks, capacity,
                                                 ctypes.byref(params)))


def hs_decode_step(shape, kv, q, new_k, new_v, smin, smax, sel_params, sel, sel_count, scores, attn_params, out,
                   lse=None, workspace=None, stream=None):
    """Append of the newest token, selection and attention of one decode step
    in one call (one launch where the library can fuse them)."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.hs_decode_step(ctypes.byref(shape), ctypes.byref(kv), _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(smin),
                               _ptr(smax), ctypes.byref(sel_params), _ptr(sel), _ptr(sel_count), _ptr(scores),
                               ctypes.byref(attn_params), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                               _stream(stream)),
           "hs_decode_step")


def hs_decode_step_reuse(shape, kv, q, new_k, new_v, smin, smax, sel, sel_count, capacity, attn_params, out,
                         lse=None, workspace=None, stream=None):
    """Append of the newest token and attention over another layer's selection
    (sel / sel_count, read only) in one call (one launch where the library can
    fuse them)."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.hs_decode_step_reuse(ctypes.byref(shape), ctypes.byref(kv), _ptr(q), _ptr(new_k), _ptr(new_v),
                                     _ptr(smin), _ptr(smax), _ptr(sel), _ptr(sel_count), int(capacity),
                                     ctypes.byref(attn_params), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                     _stream(stream)),
           "hs_decode_step_reuse")


def hs_score_select_attend(shape, kv, q, smin, smax, sel_params, sel, sel_count, scores, attn_params, out,
                           lse=None, workspace=None, stream=None):
    """Selection and attention of one decode step in one call (one launch where
    the library can fuse them)."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.hs_score_select_attend(ctypes.byref(shape), ctypes.byref(kv), _ptr(q), _ptr(smin), _ptr(smax),
                                       ctypes.byref(sel_params), _ptr(sel), _ptr(sel_count), _ptr(scores),
                                       ctypes.byref(attn_params), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                       _stream(stream)),
           "hs_score_select_attend")


def hs_sparse_paged_decode_attn_noalloc(shape, kv, q, sel, sel_count, capacity, params, out, lse=None,
                                        stream=None):
    """hs_sparse_paged_decode_attn without a workspace argument, for callers that
    cannot allocate device memory: the library's own fixed scratch array
    (HS_NOALLOC_SCRATCH_BYTES per GPU) holds the split partials."""
    _check(_lib.hs_sparse_paged_decode_attn_noalloc(ctypes.byref(shape), ctypes.byref(kv), _ptr(q), _ptr(sel),
                                                    _ptr(sel_count), int(capacity), ctypes.byref(params),
                                                    _ptr(out), _ptr(lse), _stream(stream)),
           "hs_sparse_paged_decode_attn_noalloc")


def hot_buffer(page_table, slot_owner, last_used, k_slots, v_slots, host_k, host_v,
               slots_per_stream, k_slot_scales=None, v_slot_scales=None, host_k_scales=None,
               host_v_scales=None) -> HotBuffer:
    hb = HotBuffer(_ptr(page_table), _ptr(slot_owner), _ptr(last_used), _ptr(k_slots), _ptr(v_slots),
                   _ptr(k_slot_scales), _ptr(v_slot_scales), _ptr(host_k), _ptr(host_v),
                   _ptr(host_k_scales), _ptr(host_v_scales), int(page_table.shape[0]),
                   int(page_table.shape[-1]), int(slots_per_stream))
    hb._keep = (page_table, slot_owner, last_used, k_slots, v_slots, host_k, host_v, k_slot_scales,
                v_slot_scales, host_k_scales, host_v_scales)
    return hb


def hs_swapin_misses(shape, hb, sel, sel_count, capacity, step, stats=None, stream=None):
    _check(_lib.hs_swapin_misses(ctypes.byref(shape), ctypes.byref(hb), _ptr(sel), _ptr(sel_count),
                                 int(capacity), int(step), _ptr(stats), _stream(stream)),
           "hs_swapin_misses")


def hs_swapin_plan(shape, hb, sel, sel_count, capacity, step, hit_sel, hit_count, miss_sel, miss_count,
                   stats=None, stream=None):
    _check(_lib.hs_swapin_plan(ctypes.byref(shape), ctypes.byref(hb), _ptr(sel), _ptr(sel_count), int(capacity),
                               int(step), _ptr(hit_sel), _ptr(hit_count), _ptr(miss_sel), _ptr(miss_count),
                               _ptr(stats), _stream(stream)),
           "hs_swapin_plan")


def hs_score_select_swapin_plan(shape, kv, q, smin, smax, params, sel, sel_count, hb, step, hit_sel, hit_count,
                                miss_sel, miss_count, scores=None, workspace=None, stats=None, stream=None):
    """hs_score_select_topk then hs_swapin_plan, each stream's plan in the selection's launch where it fits."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.hs_score_select_swapin_plan(ctypes.byref(shape), ctypes.byref(kv), _ptr(q), _ptr(smin), _ptr(smax),
                                            ctypes.byref(params), _ptr(sel), _ptr(sel_count), _ptr(scores),
                                            _ptr(workspace), ws_bytes, ctypes.byref(hb), int(step), _ptr(hit_sel),
                                            _ptr(hit_count), _ptr(miss_sel), _ptr(miss_count), _ptr(stats),
                                            _stream(stream)),
           "hs_score_select_swapin_plan")


def hs_swapin_copy(shape, hb, miss_sel, miss_count, capacity, max_ctas=0, stats=None, stream=None):
    _check(_lib.hs_swapin_copy(ctypes.byref(shape), ctypes.byref(hb), _ptr(miss_sel), _ptr(miss_count),
                               int(capacity), int(max_ctas), _ptr(stats), _stream(stream)),
           "hs_swapin_copy")


def hs_swapin_copy_attend(shape, hb, seq_lens, q, miss_sel, miss_count, capacity, scale, out, lse, max_ctas=0,
                          stats=None, stream=None):
    _check(_lib.hs_swapin_copy_attend(ctypes.byref(shape), ctypes.byref(hb), _ptr(seq_lens), _ptr(q), _ptr(miss_sel),
                                      _ptr(miss_count), int(capacity), float(scale), int(max_ctas), _ptr(out),
                                      _ptr(lse), _ptr(stats), _stream(stream)),
           "hs_swapin_copy_attend")


def hs_merge_attn_partials(shape, outs, lses, out, lse=None, stream=None):
    """outs [parts][batch][Hq][D] f32, lses [parts][batch][Hq] f32 -> out (bf16 or f32), lse."""
    parts, batch = outs.shape[0], outs.shape[1]
    _check(_lib.hs_merge_attn_partials(ctypes.byref(shape), int(batch), int(parts), _ptr(outs), _ptr(lses),
                                       _ptr(out), 1 if out.dtype == torch.float32 else 0, _ptr(lse),
                                       _stream(stream)),
           "hs_merge_attn_partials")


def hs_quantize_e4m3_g32(src, codes, scales, stream=None):
    """src [rows][D] f32 or bf16 -> codes [rows][D] uint8, scales [rows][D/32] f32."""
    D = src.shape[-1]
    rows = src.numel() // D
    _check(_lib.hs_quantize_e4m3_g32(_ptr(src), 1 if src.dtype == torch.float32 else 0, rows, D,
                                     _ptr(codes), _ptr(scales), _stream(stream)),
           "hs_quantize_e4m3_g32")


def hs_get_device_error(stream=None) -> tuple[int, int]:
    """Synchronise, read and clear the device error word: (status, bits)."""
    bits = c_uint32(0)
    st = _lib.hs_get_device_error(_stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


TIMEOUT_KERNELS = {1: "tensor-core attention", 2: "single-launch step", 3: "e4m3 attention",
                   4: "tensor-core bound scoring"}


def hs_get_device_error_detail(stream=None) -> tuple[int, int, dict | None]:
    """(status, bits, where) - where describes the first bounded wait that ran
    out since the last read (None if none): kernel, CTA, barrier address,
    parity, warp."""
    bits = c_uint32(0)
    rec = (c_uint32 * 11)()
    st = _lib.hs_get_device_error_detail(_stream(stream), ctypes.byref(bits), rec)
    where = None
    if rec[0]:
        w = rec[2]
        names = ("issued", "mma_s", "mma_o", "softmax0", "softmax1", "producer_item", "softmax_item", "item_chunks")
        where = {"kernel": TIMEOUT_KERNELS.get(rec[0], rec[0]), "cta": int(rec[1]), "barrier": w & 0x3FFFF,
                 "parity": (w >> 18) & 1, "warp": (w >> 19) & 31,
                 "progress": {n: int(ctypes.c_int32(rec[3 + i]).value) for i, n in enumerate(names)}}
    return int(st), int(bits.value), where
