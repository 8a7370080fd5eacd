"""Error reporting: host-side argument checks return a status and launch
nothing; device-detected problems set bits of the error word and the kernels
skip the offending item.  No test here faults the GPU: every planted error is
a value the kernels check before using it.  GPU only."""

import numpy as np
import pytest
import torch

from synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _case():
    from _parity import Case
    w = WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=1024, ctx_max=1024, k_scored=4)
    return Case(w, make_inputs(w))


def test_bad_page_id_sets_page_range_bit():
    from query_aware_sparse_hs_gb300 import hs
    c = _case()
    dec = c.decoder(out_is_fp32=True)
    dec.build_summaries(c.kv)
    dec.select(c.kv, c.q)
    assert hs.hs_get_device_error()[0] == hs.HS_OK
    bad_table = c.page_table.clone()
    j = int(dec.sel[0, 1, 2])
    bad_table[0, 1, j] = 1 << 30  # outside the pool: checked before any read
    kv_bad = hs.paged_kv(c.k_pages, c.v_pages, bad_table, c.seq_lens)
    dec.attend(kv_bad, c.q)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_ERR_OUT_OF_RANGE and bits & hs.HS_EBIT_PAGE_RANGE
    assert np.isfinite(dec.out.cpu().numpy()).all()
    # the error word is cleared by the read
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)


def test_selected_block_past_the_request_sets_block_range_bit():
    from query_aware_sparse_hs_gb300 import hs
    c = _case()
    dec = c.decoder(out_is_fp32=True)
    dec.build_summaries(c.kv)
    dec.select(c.kv, c.q)
    dec.sel[1, 0, 0] = 10_000
    dec.attend(c.kv, c.q)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_ERR_OUT_OF_RANGE and bits & hs.HS_EBIT_BLOCK_RANGE


def test_host_side_checks():
    from query_aware_sparse_hs_gb300 import hs
    c = _case()
    dec = c.decoder()
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(hs.HSError) as e:
        hs.hs_sparse_paged_decode_attn(dec.shape, c.kv, c.q, dec.sel, dec.sel_count, dec.capacity,
                                       dec.attn_params, dec.out, dec.lse, small)
    assert e.value.status == hs.HS_ERR_WORKSPACE
    tight = hs.select_params(4, 256, 4, 5)  # 5 < 1 + 4 + 1 + 4
    with pytest.raises(hs.HSError) as e:
        hs.hs_score_select_topk(dec.shape, c.kv, c.q, dec.smin, dec.smax, tight, dec.sel, dec.sel_count)
    assert e.value.status == hs.HS_ERR_CAPACITY
    odd = hs.attn_shape(32, 4, 96, 64, "bf16")
    with pytest.raises(hs.HSError) as e:
        hs.hs_build_block_summaries(odd, c.kv, 0, dec.smin, dec.smax)
    assert e.value.status == hs.HS_ERR_UNSUPPORTED
    f32shape = hs.attn_shape(32, 4, 128, 64, "f32")
    with pytest.raises(hs.HSError) as e:
        hs.hs_sparse_paged_decode_attn(f32shape, c.kv, c.q, dec.sel, dec.sel_count, dec.capacity,
                                       hs.attn_params(0.1, algo="tcgen05"), dec.out, dec.lse, dec.workspace)
    assert e.value.status == hs.HS_ERR_UNSUPPORTED
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)


def test_select_workspace_when_no_score_buffer():
    """Tensor-core scoring needs a score buffer: scores_opt or the workspace."""
    from query_aware_sparse_hs_gb300 import hs
    c = _case()
    dec = c.decoder()
    dec.build_summaries(c.kv)
    dec.select(c.kv, c.q)
    ref = dec.sel.clone()
    with pytest.raises(hs.HSError) as e:
        hs.hs_score_select_topk(dec.shape, c.kv, c.q, dec.smin, dec.smax, dec.sel_params, dec.sel, dec.sel_count)
    assert e.value.status == hs.HS_ERR_WORKSPACE
    ws = torch.empty(hs.hs_select_workspace_bytes(dec.shape, c.w.batch, c.page_table.shape[-1]),
                     dtype=torch.uint8, device="cuda")
    dec.sel.fill_(-7)
    hs.hs_score_select_topk(dec.shape, c.kv, c.q, dec.smin, dec.smax, dec.sel_params, dec.sel, dec.sel_count,
                            None, ws)
    assert torch.equal(dec.sel, ref)
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)


def _oracle_close(c, dec, tol=2e-3):
    """Every (request, kv head) of the decoder's fp32 output against the oracle."""
    from _parity import np32
    out = np32(dec.out)
    for b in range(c.w.batch):
        for kvh in range(c.w.num_kv_heads):
            r = c.oracle_pair(b, kvh)
            g = c.w.group
            assert dec.sel[b, kvh, :int(dec.sel_count[b, kvh])].tolist() == r["sel"]
            assert np.abs(out[b, kvh * g:(kvh + 1) * g] - r["out"]).max() <= tol


@pytest.mark.parametrize("mode", ["separate", "single_launch", "ranges"])
def test_wait_that_runs_out_reports_timeout_then_the_next_call_is_exact(mode):
    """The bounded waits of the tensor-core kernels: with a wait limit of 1 ns
    (far below the time any copy or product takes) a wait runs out, the CTA
    stops every role, lets the copies and products it issued land, frees its
    tensor memory and returns; the host reads HS_ERR_TIMEOUT and the context
    stays usable.  After the split counters are zeroed again (as the header
    asks after a time-out) the next call with the default limit matches the
    oracle.  "ranges": balanced chunk ranges on 3 CTAs, so each CTA runs
    several items and their hand-overs between the softmax groups."""
    single_launch = mode == "single_launch"
    from query_aware_sparse_hs_gb300 import hs
    c = _case()
    dec = c.decoder(out_is_fp32=True)
    dec.build_summaries(c.kv)
    fused = hs.hs_score_select_attend_fused(dec.shape, c.w.batch, dec.max_blocks, dec.capacity, dec.attn_params)
    assert fused == 1  # this geometry takes the single launch when asked to
    ranges = dict(max_ctas=3, ranges=True) if mode == "ranges" else {}
    short = hs.attn_params(dec.attn_params.scale, True, algo="tcgen05", split_counters=dec.split_counters,
                           wait_limit_ns=1, **ranges)
    if ranges:
        dec.attn_params = hs.attn_params(dec.attn_params.scale, True, algo="tcgen05",
                                         split_counters=dec.split_counters, **ranges)
        assert hs.hs_attn_geometry(dec.shape, c.w.batch, dec.capacity, dec.attn_params)[1] > 0
        dec.workspace = torch.empty((hs.hs_workspace_bytes(dec.shape, c.w.batch, dec.capacity, dec.attn_params),),
                                    dtype=torch.uint8, device="cuda")
    for _ in range(2):
        if single_launch:
            hs.hs_score_select_attend(dec.shape, c.kv, c.q, dec.smin, dec.smax, dec.sel_params, dec.sel,
                                      dec.sel_count, None, short, dec.out, dec.lse, dec.workspace)
        else:
            dec.select(c.kv, c.q)
            assert hs.hs_get_device_error() == (hs.HS_OK, 0)
            hs.hs_sparse_paged_decode_attn(dec.shape, c.kv, c.q, dec.sel, dec.sel_count, dec.capacity, short,
                                           dec.out, dec.lse, dec.workspace)
        st, bits, where = hs.hs_get_device_error_detail()
        assert st == hs.HS_ERR_TIMEOUT and bits & hs.HS_EBIT_TIMEOUT, (st, bits)
        # the record of the first wait that ran out names the kernel and a warp of a CTA of it
        assert where is not None, where
        assert where["kernel"] == ("single-launch step" if single_launch else "tensor-core attention"), where
        assert 0 <= where["warp"] < 12 and 0 <= where["cta"] < 1024, where
        dec.split_counters.zero_()
    dec.out.fill_(float("nan"))
    if single_launch:
        dec.select_attend(c.kv, c.q)
    else:
        dec.select(c.kv, c.q)
        dec.attend(c.kv, c.q)
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)
    _oracle_close(c, dec)
    assert int(dec.split_counters.abs().sum()) == 0
