"""One whole decode step through hs_decode_step: the append of the newest
token ("KV 稀疏化" wiki §5: the summary of its block covers it), bound scoring,
selection and attention.  Where the step is a single launch the append runs
inside it; its pages, summaries, scores, selection, output and lse must equal,
bit for bit, those of hs_append_token followed by the separate calls, and the
output must follow the oracle run on the seeded cache with the new token in
place.  GPU only."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3  # fp32 output of bf16 K/V, as in the parity tests

# name -> (workload, single launch expected)
CASES = {
    # newest token inside its block
    "llama_mid_block": (WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=3000, ctx_max=5000, k_scored=9), 1),
    # newest token in row 0 of a new block: the box starts afresh
    "llama_block_start": (WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=4097, ctx_max=4097, k_scored=9), 1),
    # 16-token blocks, eight tiles, ragged lengths
    "b16_8tiles": (WORKLOADS["ragged_bf16"].scaled(batch=4, ctx_min=1000, ctx_max=16384, k_scored=64), 1),
    # more than 8 tiles per request: the append kernel, then the separate launches
    "b16_separate": (WORKLOADS["ragged_bf16"].scaled(batch=2, ctx_min=17000, ctx_max=20000, k_scored=32), 0),
}


def _new_token(w, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (w.batch, w.num_kv_heads, w.head_dim)
    k = (torch.randn(shape, generator=g) * 3).to(torch.bfloat16)
    v = torch.randn(shape, generator=g).to(torch.bfloat16)
    return k, v


@pytest.mark.parametrize("name", list(CASES))
def test_decode_step_equals_append_then_separate_calls_and_oracle(name):
    from _parity import Case, tie_window_ok
    from query_aware_sparse_hs_gb300 import hs
    w, want = CASES[name]
    x = make_inputs(w)
    c = Case(w, x, tail_nan=False)
    new_k, new_v = _new_token(w, 7 + len(name))
    dk, dv = new_k.cuda(), new_v.cuda()
    # two copies of the cache: the single call and the reference sequence each append into their own
    pages_a = (c.k_pages.clone(), c.v_pages.clone())
    pages_b = (c.k_pages.clone(), c.v_pages.clone())
    kv_a = hs.paged_kv(*pages_a, c.page_table, c.seq_lens)
    kv_b = hs.paged_kv(*pages_b, c.page_table, c.seq_lens)
    one = c.decoder(out_is_fp32=True)
    ref = c.decoder(out_is_fp32=True, fuse_step=False)
    # the summaries of the cache before the newest token existed (L - 1 tokens)
    before = (c.seq_lens - 1).clamp(min=0).contiguous()
    one.build_summaries(hs.paged_kv(*pages_a, c.page_table, before))
    ref.build_summaries(hs.paged_kv(*pages_b, c.page_table, before))
    assert hs.hs_score_select_attend_fused(one.shape, w.batch, one.max_blocks, one.capacity, one.attn_params) == want
    one.decode_step(kv_a, c.q, dk, dv)
    ref.append(kv_b, dk, dv)
    ref.select(kv_b, c.q)
    ref.attend(kv_b, c.q)
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)
    assert torch.equal(one.sel_count, ref.sel_count) and torch.equal(one.sel, ref.sel)
    for b, L in enumerate(c.lens):  # rows of blocks past a request's end are never written
        nb = O.num_blocks(L, w.block_size)
        assert torch.equal(one.smin[b, :, :nb], ref.smin[b, :, :nb]), b
        assert torch.equal(one.smax[b, :, :nb], ref.smax[b, :, :nb]), b
        assert torch.equal(one.scores[b, :, :nb], ref.scores[b, :, :nb]), b
    assert torch.equal(one.out, ref.out) and torch.equal(one.lse, ref.lse)
    assert torch.equal(pages_a[0], pages_b[0]) and torch.equal(pages_a[1], pages_b[1])

    # the oracle on the seeded cache with the new token written at L - 1
    g, B = w.group, w.block_size
    scale = 1.0 / math.sqrt(w.head_dim)
    sel, cnt = one.sel.cpu().numpy(), one.sel_count.cpu().numpy()
    out, lse = one.out.cpu().numpy(), one.lse.cpu().numpy()
    smin, smax = one.smin.float().cpu().numpy(), one.smax.float().cpu().numpy()
    pairs = [(b, kvh) for b in range(w.batch) for kvh in range(w.num_kv_heads)]
    for b, kvh in pairs[:: max(1, len(pairs) // 6)]:
        L = c.lens[b]
        K, V = c.logical(b, kvh, "k"), c.logical(b, kvh, "v")
        K[L - 1] = new_k[b, kvh].double().numpy()
        V[L - 1] = new_v[b, kvh].double().numpy()
        lo, hi = O.stored_summaries(*O.block_summaries(K, B), "bf16")
        nb = O.num_blocks(L, B)
        assert np.array_equal(smin[b, kvh, :nb], lo) and np.array_equal(smax[b, kvh, :nb], hi), (b, kvh)
        r = O.decode_pair(c.q_group(b, kvh), K, V, B, "bf16", w.sink_tokens, w.window_tokens, w.k_scored, scale)
        got = sel[b, kvh, :cnt[b, kvh]].tolist()
        assert tie_window_ok(r["score"], r["forced"], got, r["sel"], w.k_scored), (b, kvh)
        ref_out, ref_lse = O.sparse_attention(c.q_group(b, kvh), K, V, got, B, scale)
        assert np.abs(out[b, kvh * g:(kvh + 1) * g] - ref_out).max() <= TOL, (b, kvh)
        assert np.abs(lse[b, kvh * g:(kvh + 1) * g] - ref_lse).max() <= TOL, (b, kvh)


def test_decode_step_checks_its_arguments():
    from _parity import Case
    from query_aware_sparse_hs_gb300 import hs
    w = CASES["llama_mid_block"][0]
    c = Case(w, make_inputs(w), tail_nan=False)
    d = c.decoder()
    with pytest.raises(hs.HSError) as e:
        hs.hs_decode_step(d.shape, c.kv, c.q, None, None, d.smin, d.smax, d.sel_params, d.sel, d.sel_count, None,
                          d.attn_params, d.out, d.lse, d.workspace)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)


def test_decode_step_with_early_summaries_equals_without():
    """HS_ATTN_EARLY_SUMMARIES (the step may copy its summary tiles before the
    previous kernel completes; the caller guarantees that kernel does not write
    them): two layers stepped in turn, so the kernel before each step is the
    other layer's.  Every output equals, bit for bit, that of the same steps
    without the flag."""
    from _parity import Case
    from query_aware_sparse_hs_gb300 import hs
    w = CASES["llama_mid_block"][0]
    results = []
    for early in (False, True):
        runs = []
        for layer in range(2):
            x = make_inputs(w)
            if layer:
                x["q"] = x["q"].flip(-1).contiguous()
            c = Case(w, x, tail_nan=False)
            d = c.decoder(out_is_fp32=True, early_summaries=early)
            d.build_summaries(hs.paged_kv(c.k_pages, c.v_pages, c.page_table, (c.seq_lens - 1).clamp(min=0)))
            runs.append((c, d))
        new_k, new_v = _new_token(w, 99)
        dk, dv = new_k.cuda(), new_v.cuda()
        for _ in range(3):  # layer 0, layer 1, layer 0, ...
            for c, d in runs:
                d.decode_step(c.kv, c.q, dk, dv)
        torch.cuda.synchronize()
        assert hs.hs_get_device_error() == (hs.HS_OK, 0)
        results.append([(d.out.clone(), d.lse.clone(), d.sel.clone(), d.sel_count.clone(), d.smin.clone(), d.smax.clone())
                        for _, d in runs])
    lens = runs[0][0].lens
    for a, b in zip(*results):
        for x, y in zip(a[:4], b[:4]):
            assert torch.equal(x, y)
        for bi, L in enumerate(lens):  # summary rows of blocks past a request's end are never written
            nb = O.num_blocks(L, w.block_size)
            for x, y in zip(a[4:], b[4:]):
                assert torch.equal(x[bi, :, :nb], y[bi, :, :nb]), bi


@pytest.mark.parametrize("name", list(CASES))
def test_decode_step_reuse_equals_append_then_attention(name):
    """A layer that reuses another layer's selection: hs_decode_step_reuse
    (one launch where the step fuses) must equal, bit for bit, the append
    followed by the attention over that selection - pages, summaries, output
    and lse - and leave the reused selection untouched."""
    from _parity import Case
    from query_aware_sparse_hs_gb300 import hs
    w, _ = CASES[name]
    x = make_inputs(w)
    c = Case(w, x, tail_nan=False)
    lead = c.decoder(out_is_fp32=True)
    lead.build_summaries(c.kv)
    lead.select(c.kv, c.q)  # the selection the deeper layer reuses
    sel0, cnt0 = lead.sel.clone(), lead.sel_count.clone()
    new_k, new_v = _new_token(w, 31 + len(name))
    dk, dv = new_k.cuda(), new_v.cuda()
    q2 = c.q.flip(-1).contiguous()  # the reusing layer's own query
    pages_a = (c.k_pages.clone(), c.v_pages.clone())
    pages_b = (c.k_pages.clone(), c.v_pages.clone())
    kv_a = hs.paged_kv(*pages_a, c.page_table, c.seq_lens)
    kv_b = hs.paged_kv(*pages_b, c.page_table, c.seq_lens)
    one, ref = c.decoder(out_is_fp32=True), c.decoder(out_is_fp32=True)
    before = (c.seq_lens - 1).clamp(min=0).contiguous()
    one.build_summaries(hs.paged_kv(*pages_a, c.page_table, before))
    ref.build_summaries(hs.paged_kv(*pages_b, c.page_table, before))
    one.decode_step_reuse(kv_a, q2, dk, dv, lead)
    ref.append(kv_b, dk, dv)
    ref.attend(kv_b, q2, selection=lead)
    torch.cuda.synchronize()
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)
    assert torch.equal(one.out, ref.out) and torch.equal(one.lse, ref.lse)
    assert torch.equal(pages_a[0], pages_b[0]) and torch.equal(pages_a[1], pages_b[1])
    for b, L in enumerate(c.lens):  # rows of blocks past a request's end are never written
        nb = O.num_blocks(L, w.block_size)
        assert torch.equal(one.smin[b, :, :nb], ref.smin[b, :, :nb]), b
        assert torch.equal(one.smax[b, :, :nb], ref.smax[b, :, :nb]), b
    assert torch.equal(lead.sel, sel0) and torch.equal(lead.sel_count, cnt0)
