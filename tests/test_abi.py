"""The C-ABI library loads and exports every function that include/hs.h
declares; host-side argument checks answer without a GPU.  CPU only (no
compute call is made)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "hs.h")).read()
    return re.findall(r"HS_API\s+[\w\s\*]+?\b(hs_\w+)\s*\(", src)


def test_header_declares_the_four_entry_points():
    names = set(_declared())
    for n in ("hs_build_block_summaries", "hs_score_select_topk", "hs_sparse_paged_decode_attn",
              "hs_swapin_misses"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from query_aware_sparse_hs_gb300 import hs
    lib = hs.library()
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in hs.SYMBOLS, name
    out = subprocess.run(["nm", "-D", "--defined-only", hs.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    assert exported == set(_declared())


def test_status_strings_and_version():
    from query_aware_sparse_hs_gb300 import hs
    assert hs.hs_version() >= 1
    assert hs.hs_status_string(0) == "ok"
    assert "capacity" in hs.hs_status_string(hs.HS_ERR_CAPACITY)
    assert hs.hs_status_string(99) == "unknown status"


def test_host_checks_reject_bad_arguments_without_a_gpu():
    from query_aware_sparse_hs_gb300 import hs
    lib = hs.library()
    shape = hs.attn_shape(32, 4, 128, 64, "bf16")
    assert lib.hs_build_block_summaries(ctypes.byref(shape), None, 0, None, None, None) == hs.HS_ERR_INVALID_ARG
    bad = hs.attn_shape(32, 5, 128, 64, "bf16")
    assert lib.hs_build_block_summaries(ctypes.byref(bad), None, 0, None, None, None) == hs.HS_ERR_INVALID_ARG
    odd_dim = hs.attn_shape(32, 4, 80, 64, "bf16")
    assert lib.hs_build_block_summaries(ctypes.byref(odd_dim), None, 0, None, None, None) == hs.HS_ERR_UNSUPPORTED
    g3 = hs.attn_shape(12, 4, 128, 64, "bf16")
    assert lib.hs_build_block_summaries(ctypes.byref(g3), None, 0, None, None, None) == hs.HS_ERR_UNSUPPORTED
    # a selection capacity below the largest possible selection is refused before launch
    kv = hs.PagedKV()
    kv.seq_lens = 0x1000
    kv.batch, kv.max_blocks = 1, 512
    params = hs.select_params(4, 256, 27, 31)  # needs 1 + 5 + 27 = 33
    st = lib.hs_score_select_topk(ctypes.byref(shape), ctypes.byref(kv), 0x1000, 0x1000, 0x1000,
                                  ctypes.byref(params), 0x1000, 0x1000, None, None, 0, None)
    assert st == hs.HS_ERR_CAPACITY
    # score smoothing: the weight must be in [0, 1) and needs a history buffer
    for weight, hist in ((1.0, 0x1000), (-0.1, 0x1000), (0.3, None)):
        p = hs.select_params(4, 256, 27, 33)
        p.history_weight, p.score_history = weight, hist
        st = lib.hs_score_select_topk(ctypes.byref(shape), ctypes.byref(kv), 0x1000, 0x1000, 0x1000,
                                      ctypes.byref(p), 0x1000, 0x1000, None, None, 0, None)
        assert st == hs.HS_ERR_INVALID_ARG, (weight, hist)
    assert lib.hs_quantize_e4m3_g32(0x1000, 0, 10, 96, 0x1000, 0x1000, None) == hs.HS_ERR_UNSUPPORTED
    # the append call: a missing new token, or an e4m3 cache without scales
    full = hs.PagedKV()
    full.k_pages = full.v_pages = full.page_table = full.seq_lens = 0x1000
    full.batch, full.max_blocks, full.num_pages = 1, 4, 4
    assert lib.hs_append_token(ctypes.byref(shape), ctypes.byref(full), None, 0x1000, 0x1000, 0x1000,
                               None) == hs.HS_ERR_INVALID_ARG
    fp8 = hs.attn_shape(32, 4, 128, 64, "fp8")
    assert lib.hs_append_token(ctypes.byref(fp8), ctypes.byref(full), 0x1000, 0x1000, 0x1000, 0x1000,
                               None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_workspace_bytes(ctypes.byref(bad), 8, 33, None) == 0


def test_workspace_size_formula():
    from query_aware_sparse_hs_gb300 import hs
    shape = hs.attn_shape(32, 4, 128, 64, "bf16")
    p = hs.attn_params(0.1, blocks_per_split=4)
    # 9 splits of 4 blocks cover 33; (D + 1) floats per (request, q head, split)
    assert hs.hs_workspace_bytes(shape, 8, 33, p) == ((8 * 32 * 9 * 129 * 4 + 255) // 256) * 256


def test_kv_bytes_per_token_of_an_8b_gqa_model():
    """64 KB per token and 2 GiB at 32K context for 32 layers x 4 kv heads x 128 x fp16
    (SparDA article, §1.1) from the bench's layout arithmetic."""
    import bench
    assert bench.kv_bytes_per_token(32, 4, 128, 2) == 65536
    assert bench.kv_bytes_per_token(32, 4, 128, 2) * 32768 == 2 * 1024 ** 3
    assert bench.kv_bytes_per_token(32, 4, 128, 2) * 131072 == 8 * 1024 ** 3



def test_host_checks_of_the_overlap_and_merge_calls():
    """The overlapped swap-in calls and the partial merge refuse missing or
    aliased buffers before launching anything (no GPU needed)."""
    from query_aware_sparse_hs_gb300 import hs
    lib = hs.library()
    shape = hs.attn_shape(32, 4, 128, 64, "bf16")
    hb = hs.HotBuffer()
    P = 0x1000
    # plan: the hit and miss lists may not alias the selection or each other
    assert lib.hs_swapin_plan(ctypes.byref(shape), ctypes.byref(hb), P, P, 32, 0, P, P, P + 64, P, None,
                              None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_swapin_plan(ctypes.byref(shape), ctypes.byref(hb), P, P, 32, 0, None, P, P + 64, P, None,
                              None) == hs.HS_ERR_INVALID_ARG
    # copy: a negative CTA count; copy+attend: missing query or outputs
    assert lib.hs_swapin_copy(ctypes.byref(shape), ctypes.byref(hb), P, P, 32, -1, None,
                              None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_swapin_copy_attend(ctypes.byref(shape), ctypes.byref(hb), P, None, P, P, 32, 0.088, 0, P, P,
                                     None, None) == hs.HS_ERR_INVALID_ARG
    # an empty hot buffer description is refused
    assert lib.hs_swapin_copy(ctypes.byref(shape), ctypes.byref(hb), P, P, 32, 0, None,
                              None) == hs.HS_ERR_INVALID_ARG
    # merge of partials: no parts, or a misaligned output
    assert lib.hs_merge_attn_partials(ctypes.byref(shape), 2, 0, P, P, P, 1, None, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_merge_attn_partials(ctypes.byref(shape), 2, 2, P, P, P + 2, 1, None,
                                      None) == hs.HS_ERR_INVALID_ARG
    # attention: a negative CTA cap is refused
    kv = hs.PagedKV()
    kv.k_pages = kv.v_pages = kv.page_table = kv.seq_lens = P
    kv.batch, kv.max_blocks, kv.num_pages = 1, 4, 4
    params = hs.attn_params(0.088, max_ctas=-1)
    st = lib.hs_sparse_paged_decode_attn(ctypes.byref(shape), ctypes.byref(kv), P, P, P, 8, ctypes.byref(params),
                                         P, None, None, 0, None)
    assert st == hs.HS_ERR_INVALID_ARG


def test_host_checks_of_the_combined_call():
    from query_aware_sparse_hs_gb300 import hs
    lib = hs.library()
    shape = hs.attn_shape(32, 4, 128, 64, "bf16")
    params = hs.attn_params(0.088)
    sp = hs.select_params(4, 256, 27, 33)
    kv = hs.PagedKV()
    P = 0x10000
    kv.k_pages = kv.v_pages = kv.page_table = kv.seq_lens = P
    kv.batch, kv.max_blocks, kv.num_pages = 8, 512, 4096
    need = hs.hs_score_select_attend_workspace_bytes(shape, 8, 512, 32, params)
    sel_ws = hs.hs_select_workspace_bytes(shape, 8, 512)
    assert sel_ws == 8 * 4 * 512 * 4 and need > sel_ws
    # no workspace for the selection's score buffer: refused before any device work
    st = lib.hs_score_select_attend(ctypes.byref(shape), ctypes.byref(kv), P, P, P, ctypes.byref(sp), P, P, None,
                                    ctypes.byref(params), P, None, None, 0, None)
    assert st == hs.HS_ERR_WORKSPACE
    # the selection's own checks come first: a capacity below the largest selection
    small = hs.select_params(4, 256, 27, 8)
    st = lib.hs_score_select_attend(ctypes.byref(shape), ctypes.byref(kv), P, P, P, ctypes.byref(small), P, P,
                                    None, ctypes.byref(params), P, None, P, need, None)
    assert st == hs.HS_ERR_CAPACITY
    # the geometry query answers -1 for an invalid shape or CTA cap
    bad = hs.attn_shape(32, 5, 128, 64, "bf16")
    assert hs.hs_score_select_attend_fused(bad, 8, 512, 32, params) == -1
    assert hs.hs_score_select_attend_fused(shape, 8, 512, 32, hs.attn_params(0.088, max_ctas=-1)) == -1
    assert hs.hs_score_select_attend_workspace_bytes(bad, 8, 512, 32, params) == 0
