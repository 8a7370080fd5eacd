"""The append step through the C ABI (hs_append_token): token by token, the
cache rows and block summaries it leaves must equal the oracle's quantisation
of the same rows and its plain per-block min/max over everything appended so
far.  GPU only.

Each request starts from a prefix (one from an empty cache) whose summaries are
built by the library; the rest of its tokens are appended one call per token,
crossing block boundaries.  A request that has reached its length keeps its
length, so later calls re-append its last token: that must change nothing.
Rows not yet appended hold NaN, summaries of blocks not yet begun hold NaN.
"""

import numpy as np
import pytest
import torch

import oracle as O
from synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, prefix lengths are L - tail, tail)
    "f32_b16_d64": (WORKLOADS["tiny_f32"].scaled(batch=3, ctx_min=40, ctx_max=140), 50),
    "bf16_b64_d128": (WORKLOADS["llama8b_bf16"].scaled(batch=3, ctx_min=90, ctx_max=260), 80),
    "fp8_b64_d128": (WORKLOADS["fp8_g32"].scaled(batch=3, ctx_min=90, ctx_max=260), 80),
}


def _np(t):
    return t.float().cpu().numpy() if t.dtype != torch.uint8 else t.cpu().numpy()


@pytest.mark.parametrize("name", list(CASES))
def test_append_matches_the_oracle_token_by_token(name):
    from query_aware_sparse_hs_gb300 import hs
    w, tail = CASES[name]
    x = make_inputs(w)
    dev = torch.device("cuda")
    B, D, hkv = w.block_size, w.head_dim, w.num_kv_heads
    lens = x["seq_lens"].tolist()
    start = [0] + [max(0, L - tail) for L in lens[1:]]  # request 0 starts empty
    table = x["page_table"].to(dev)
    src_k, src_v = x["k_pages"].to(dev), x["v_pages"].to(dev)  # f32 or bf16 source rows
    P = src_k.shape[0]
    fp8 = w.kv_dtype == "fp8"

    # the cache before the appends: the prefix as stored, NaN everywhere else
    if fp8:
        k_pages = torch.full((P, B, D), 0x7F, dtype=torch.uint8, device=dev)  # e4m3 NaN
        v_pages = torch.full_like(k_pages, 0x7F)
        k_scales = torch.full((P, B, D // 32), float("nan"), device=dev)
        v_scales = torch.full_like(k_scales, float("nan"))
    else:
        k_pages = torch.full_like(src_k, float("nan"))
        v_pages = torch.full_like(src_v, float("nan"))
        k_scales = v_scales = None
    tb = x["page_table"].numpy()
    prefix = torch.zeros((P, B), dtype=torch.bool)
    for b, s0 in enumerate(start):
        for kvh in range(hkv):
            for t in range(s0):
                prefix[int(tb[b, kvh, t // B]), t % B] = True
    prefix = prefix.to(dev)
    if fp8:  # the prefix as the library's quantiser stores it
        kc, vc = torch.empty_like(k_pages), torch.empty_like(v_pages)
        ks, vs = torch.empty_like(k_scales), torch.empty_like(v_scales)
        hs.hs_quantize_e4m3_g32(src_k, kc, ks)
        hs.hs_quantize_e4m3_g32(src_v, vc, vs)
        k_pages[prefix], v_pages[prefix] = kc[prefix], vc[prefix]
        k_scales[prefix], v_scales[prefix] = ks[prefix], vs[prefix]
    else:
        k_pages[prefix], v_pages[prefix] = src_k[prefix], src_v[prefix]
    seq = torch.tensor(start, dtype=torch.int32, device=dev)
    kv = hs.paged_kv(k_pages, v_pages, table, seq, k_scales, v_scales)
    shape = hs.attn_shape(w.num_q_heads, hkv, D, B, w.kv_dtype)
    sdt = torch.float32 if w.kv_dtype == "f32" else torch.bfloat16
    smin = torch.full((w.batch, hkv, w.max_blocks, D), float("nan"), dtype=sdt, device=dev)
    smax = torch.full_like(smin, float("nan"))
    hs.hs_build_block_summaries(shape, kv, 0, smin, smax)

    # one append per step; each request advances until it reaches its length
    b_idx = torch.arange(w.batch, device=dev)[:, None].expand(w.batch, hkv)
    h_idx = torch.arange(hkv, device=dev)[None, :].expand(w.batch, hkv)
    steps = max(L - s for L, s in zip(lens, start))
    for i in range(steps):
        cur = [min(L, s + i + 1) for L, s in zip(lens, start)]
        seq.copy_(torch.tensor(cur, dtype=torch.int32))
        t = torch.tensor(cur, device=dev)[:, None].expand(w.batch, hkv) - 1
        pages = table[b_idx, h_idx, t // B].long()
        new_k = src_k[pages, t % B].contiguous()  # [batch][Hkv][D]
        new_v = src_v[pages, t % B].contiguous()
        hs.hs_append_token(shape, kv, new_k, new_v, smin, smax)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_OK, bits

    # compare with the oracle over every request's full length
    sk, sv = _np(src_k), _np(src_v)
    gk, gv = _np(k_pages), _np(v_pages)
    gks = _np(k_scales) if fp8 else None
    gvs = _np(v_scales) if fp8 else None
    gmin, gmax = _np(smin), _np(smax)
    for b, L in enumerate(lens):
        nb = O.num_blocks(L, B)
        for kvh in range(hkv):
            row = tb[b, kvh]
            rk, rv = O.gather_rows(sk, row, L, B), O.gather_rows(sv, row, L, B)
            if fp8:
                kc, ks = O.quantize_e4m3_g32(rk)
                vc, vs = O.quantize_e4m3_g32(rv)
                assert np.array_equal(O.gather_rows(gk, row, L, B), kc), (b, kvh)
                assert np.array_equal(O.gather_rows(gv, row, L, B), vc), (b, kvh)
                assert np.array_equal(O.gather_rows(gks, row, L, B), ks), (b, kvh)
                assert np.array_equal(O.gather_rows(gvs, row, L, B), vs), (b, kvh)
                K = O.kv_values("fp8", kc, ks)
            else:
                assert np.array_equal(O.gather_rows(gk, row, L, B), rk), (b, kvh)
                assert np.array_equal(O.gather_rows(gv, row, L, B), rv), (b, kvh)
                K = O.kv_values(w.kv_dtype, rk)
            emin, emax = O.stored_summaries(*O.block_summaries(K, B), w.kv_dtype)
            assert np.array_equal(gmin[b, kvh, :nb].astype(np.float64), emin), (b, kvh)
            assert np.array_equal(gmax[b, kvh, :nb].astype(np.float64), emax), (b, kvh)


def test_append_reports_a_missing_page_and_an_overlong_request():
    """A block without a page, or a length past max_blocks * B, sets its error
    bit; that stream's cache and summaries stay as they were, the others are
    appended."""
    from query_aware_sparse_hs_gb300 import hs
    w = WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=128, ctx_max=256)
    x = make_inputs(w, device="cuda")
    B, D, hkv, mb = w.block_size, w.head_dim, w.num_kv_heads, w.max_blocks
    shape = hs.attn_shape(w.num_q_heads, hkv, D, B, "bf16")
    table = x["page_table"].clone()
    table[0, :, 2:] = -1  # request 0: blocks from 2 on have no page
    seq = x["seq_lens"].clone()
    seq[0] = 2 * B
    kv = hs.paged_kv(x["k_pages"], x["v_pages"], table, seq)
    smin = torch.zeros((w.batch, hkv, mb, D), dtype=torch.bfloat16, device="cuda")
    smax = torch.zeros_like(smin)
    hs.hs_build_block_summaries(shape, kv, 0, smin, smax)
    new_k = torch.randn((w.batch, hkv, D), device="cuda").to(torch.bfloat16)
    new_v = torch.randn_like(new_k)

    # request 0 grows into block 2, which has no page yet
    seq[0] = 2 * B + 1
    before = (x["k_pages"].clone(), smin.clone(), smax.clone())
    hs.hs_append_token(shape, kv, new_k, new_v, smin, smax)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_ERR_OUT_OF_RANGE and bits == hs.HS_EBIT_PAGE_RANGE
    assert torch.equal(smin[0], before[1][0]) and torch.equal(smax[0], before[2][0])
    # request 1 re-appended its last row with the new values
    t1 = int(seq[1]) - 1
    for kvh in range(hkv):
        page = int(table[1, kvh, t1 // B])
        assert torch.equal(x["k_pages"][page, t1 % B], new_k[1, kvh])
        assert torch.equal(x["v_pages"][page, t1 % B], new_v[1, kvh])

    # a length past max_blocks * B
    seq[0] = mb * B + 1
    hs.hs_append_token(shape, kv, new_k, new_v, smin, smax)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_ERR_OUT_OF_RANGE and bits == hs.HS_EBIT_BLOCK_RANGE
    assert torch.equal(smin[0], before[1][0])
