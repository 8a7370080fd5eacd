"""Bound scoring, selection and attention of one decode step through the one
combined call (hs_score_select_attend).  Where the library runs it as a single
cluster launch (bf16, head_dim 128, g <= 8, every (request, kv head) in one
cluster of at most 8 CTAs, all in one wave) its scores, selection, output and
lse must equal, bit for bit, those of the separate calls (the same arithmetic
in the same order), and the output must follow the oracle's attention over the
selection ("KV 稀疏化" wiki §5 and §2; "分块稀疏注意力与KV Cache量化" §2.2).
GPU only."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import WORKLOADS, drift_queries, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3  # fp32 output of bf16 K/V, as in the parity tests

# name -> (workload, single launch expected)
CASES = {
    # one 128-block tile, eight attention splits per (request, kv head)
    "llama_1tile_8splits": (WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=3000, ctx_max=5000, k_scored=9), 1),
    # 16-token blocks: eight tiles, six splits, ragged lengths
    "b16_8tiles": (WORKLOADS["ragged_bf16"].scaled(batch=4, ctx_min=1000, ctx_max=16384, k_scored=64), 1),
    # requests shorter than one tile next to long ones: CTAs without a tile
    "b16_short_and_long": (WORKLOADS["ragged_bf16"].scaled(batch=4, ctx_min=40, ctx_max=9000, k_scored=16), 1),
    # more than 8 tiles per request: the separate launches
    "b16_too_many_tiles": (WORKLOADS["ragged_bf16"].scaled(batch=2, ctx_min=17000, ctx_max=20000, k_scored=32), 0),
    # e4m3 K/V: the separate launches
    "fp8": (WORKLOADS["fp8_g32"].scaled(batch=2, ctx_min=3000, ctx_max=4133, k_scored=20), 0),
}


@pytest.fixture(scope="module")
def cases():
    from _parity import Case
    return {name: Case(w, make_inputs(w)) for name, (w, _) in CASES.items()}


def _err_clear():
    from query_aware_sparse_hs_gb300 import hs
    st, bits = hs.hs_get_device_error()
    assert st == 0 and bits == 0, (st, bits)


def _pair(c, **kw):
    """Two decoders on the same inputs: one combined call, and the separate calls."""
    fused = c.decoder(out_is_fp32=True, **kw)
    split = c.decoder(out_is_fp32=True, fuse_step=False, **kw)
    for d in (fused, split):
        d.build_summaries(c.kv)
    return fused, split


def _assert_same(c, fused, split):
    w = c.w
    assert torch.equal(fused.sel_count, split.sel_count)
    assert torch.equal(fused.sel, split.sel)
    for b, L in enumerate(c.lens):
        nb = O.num_blocks(L, w.block_size)
        assert torch.equal(fused.scores[b, :, :nb], split.scores[b, :, :nb]), b
    assert torch.equal(fused.out, split.out)
    assert torch.equal(fused.lse, split.lse)


def _assert_oracle(c, dec, pairs):
    from _parity import tie_window_ok
    w = c.w
    g, B = w.group, w.block_size
    scale = 1.0 / math.sqrt(w.head_dim)
    sel, cnt = dec.sel.cpu().numpy(), dec.sel_count.cpu().numpy()
    out, lse = dec.out.cpu().numpy(), dec.lse.cpu().numpy()
    for b, kvh in pairs:
        r = c.oracle_pair(b, kvh)
        got = sel[b, kvh, :cnt[b, kvh]].tolist()
        assert tie_window_ok(r["score"], r["forced"], got, r["sel"], w.k_scored), (b, kvh)
        K, V = c.logical(b, kvh, "k"), c.logical(b, kvh, "v")
        ref, ref_lse = O.sparse_attention(c.q_group(b, kvh), K, V, got, B, scale)
        assert np.abs(out[b, kvh * g:(kvh + 1) * g] - ref).max() <= TOL, (b, kvh)
        assert np.abs(lse[b, kvh * g:(kvh + 1) * g] - ref_lse).max() <= TOL, (b, kvh)


@pytest.mark.parametrize("name", list(CASES))
def test_combined_call_equals_separate_calls_and_oracle(cases, name):
    from query_aware_sparse_hs_gb300 import hs
    c = cases[name]
    w = c.w
    fused, split = _pair(c)
    want = CASES[name][1]
    assert hs.hs_score_select_attend_fused(fused.shape, w.batch, fused.max_blocks, fused.capacity,
                                           fused.attn_params) == want
    fused.step(c.kv, c.q)
    split.step(c.kv, c.q)
    _err_clear()
    _assert_same(c, fused, split)
    pairs = [(b, kvh) for b in range(w.batch) for kvh in range(w.num_kv_heads)]
    _assert_oracle(c, fused, pairs[:: max(1, len(pairs) // 6)])


def test_full_size_llama_layer_single_launch():
    """The Llama-8B-like layer (8 x 32768 tokens, 4 tiles and 4 splits per
    (request, kv head)): bit-identical to the separate calls, the oracle on
    sampled pairs, and repeated calls give the same bits."""
    from _parity import Case
    from query_aware_sparse_hs_gb300 import hs
    w = WORKLOADS["llama8b_bf16"]
    c = Case(w, make_inputs(w))
    fused, split = _pair(c)
    assert hs.hs_score_select_attend_fused(fused.shape, w.batch, fused.max_blocks, fused.capacity,
                                           fused.attn_params) == 1
    fused.step(c.kv, c.q)
    split.step(c.kv, c.q)
    _err_clear()
    _assert_same(c, fused, split)
    first = fused.out.clone()
    for _ in range(3):
        fused.step(c.kv, c.q)
    _err_clear()
    assert torch.equal(fused.out, first)
    _assert_oracle(c, fused, [(0, 0), (3, 2), (7, 3)])


def test_empty_and_tiny_requests():
    from _parity import Case
    w = WORKLOADS["ragged_bf16"].scaled(batch=4, ctx_min=40, ctx_max=40, k_scored=2)
    x = make_inputs(w)
    x["seq_lens"] = torch.tensor([0, 1, 17, 40], dtype=torch.int32)
    c = Case(w, x)
    fused, split = _pair(c)
    fused.step(c.kv, c.q)
    split.step(c.kv, c.q)
    _err_clear()
    _assert_same(c, fused, split)
    cnt = fused.sel_count.cpu().numpy()
    assert np.all(cnt[0] == 0) and np.all(cnt[1] == 1)
    out, lse = fused.out.cpu().numpy(), fused.lse.cpu().numpy()
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    _assert_oracle(c, fused, [(b, kvh) for b in (1, 2, 3) for kvh in range(w.num_kv_heads)])


def test_smoothed_steps_match_separate_calls():
    """Score smoothing across steps (SparDA article §6.1) inside the single launch."""
    from _parity import Case
    w = CASES["llama_1tile_8splits"][0]
    c = Case(w, make_inputs(w))
    fused, split = _pair(c, score_smoothing=0.3)
    for q in drift_queries(w, c.x["q"], 4):
        q = q.to(c.q.device).contiguous()
        fused.step(c.kv, q)
        split.step(c.kv, q)
        _err_clear()
        assert torch.equal(fused.score_history.nan_to_num(7.0), split.score_history.nan_to_num(7.0))
        assert torch.equal(fused.sel, split.sel) and torch.equal(fused.out, split.out)


def test_bad_page_id_is_reported_and_skipped():
    """A selected block whose page id is out of range: HS_EBIT_PAGE_RANGE, the
    block is left out, exactly as in the separate attention call."""
    from _parity import Case
    from query_aware_sparse_hs_gb300 import hs
    w = CASES["llama_1tile_8splits"][0]
    c = Case(w, make_inputs(w))
    fused, split = _pair(c)
    _err_clear()
    c.page_table[1, 2, 0] = 1 << 30  # block 0 is a sink block: always selected
    fused.step(c.kv, c.q)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_ERR_OUT_OF_RANGE and bits == hs.HS_EBIT_PAGE_RANGE
    split.step(c.kv, c.q)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_ERR_OUT_OF_RANGE and bits == hs.HS_EBIT_PAGE_RANGE
    assert torch.equal(fused.out, split.out) and torch.equal(fused.sel, split.sel)


def test_workspace_is_checked():
    from _parity import Case
    from query_aware_sparse_hs_gb300 import hs
    w = CASES["llama_1tile_8splits"][0]
    c = Case(w, make_inputs(w))
    d = c.decoder()
    need = hs.hs_score_select_attend_workspace_bytes(d.shape, w.batch, d.max_blocks, d.capacity, d.attn_params)
    assert need > 0 and d.workspace.numel() >= need
    small = d.workspace[:need - 256]
    with pytest.raises(hs.HSError) as e:
        hs.hs_score_select_attend(d.shape, c.kv, c.q, d.smin, d.smax, d.sel_params, d.sel, d.sel_count, None,
                                  d.attn_params, d.out, d.lse, small)
    assert e.value.status == hs.HS_ERR_WORKSPACE
