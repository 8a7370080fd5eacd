"""Full-size workloads in the launch configuration bench.py times (automatic
split geometry and kernel choice), checked against the oracle on sampled
(request, kv head) pairs, plus properties that hold for every pair.  GPU only;
each test needs a few GB of device memory (the offload test also ~17 GB of
pinned host memory).
"""

import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import WORKLOADS, drift_queries, make_inputs

pytestmark = pytest.mark.gpu


def _dev_inputs(w):
    """Inputs generated on the GPU as bench.py does; fp8 K/V quantised by the library."""
    from query_aware_sparse_hs_gb300 import hs
    x = make_inputs(w, device="cuda")
    if w.kv_dtype == "fp8":
        D = w.head_dim
        for name in ("k", "v"):
            src = x[f"{name}_pages"]
            codes = torch.empty(src.shape, dtype=torch.uint8, device="cuda")
            scales = torch.empty(src.shape[:-1] + (D // 32,), dtype=torch.float32, device="cuda")
            hs.hs_quantize_e4m3_g32(src, codes, scales)
            x[f"{name}_src"] = src
            x[f"{name}_pages"] = codes
            x[f"{name}_scales"] = scales
    return x


def _pair_logical(w, x, b, kvh, which):
    """Oracle-side float64 rows of one pair, from the seeded inputs only (e4m3:
    the oracle quantises the bf16 source itself)."""
    B, L = w.block_size, int(x["seq_lens"][b])
    row = x["page_table"][b, kvh].cpu().numpy()
    nb = O.num_blocks(L, B)
    pages = torch.from_numpy(row[:nb]).long().cuda()
    if w.kv_dtype == "fp8":
        src = x[f"{which}_src"][pages].float().cpu().numpy().reshape(-1, w.head_dim)[:L]
        codes, scales = O.quantize_e4m3_g32(src)
        return O.kv_values("fp8", codes, scales), codes, pages
    rows = x[f"{which}_pages"][pages].float().cpu().numpy().reshape(-1, w.head_dim)[:L]
    return O.kv_values(w.kv_dtype, rows), None, pages


def _check_pairs(w, x, dec, samples, tol):
    from _parity import tie_window_ok
    sel = dec.sel.cpu().numpy()
    cnt = dec.sel_count.cpu().numpy()
    out = dec.out.float().cpu().numpy()
    lens = x["seq_lens"].cpu().numpy()
    g = w.group
    # properties of every pair
    for b in range(w.batch):
        L = int(lens[b])
        nb = O.num_blocks(L, w.block_size)
        F = O.forced_blocks(L, w.block_size, w.sink_tokens, w.window_tokens)
        for kvh in range(w.num_kv_heads):
            n = int(cnt[b, kvh])
            s = sel[b, kvh, :n].tolist()
            assert n == min(nb, len(F) + w.k_scored)
            assert s == sorted(set(s)) and set(F) <= set(s) and all(0 <= j < nb for j in s)
            assert np.all(sel[b, kvh, n:] == -1)
    assert np.isfinite(out).all()
    # element-wise parity on the sampled pairs
    for b, kvh in samples:
        K, kcodes, pages = _pair_logical(w, x, b, kvh, "k")
        V, _, _ = _pair_logical(w, x, b, kvh, "v")
        if kcodes is not None:  # the library's codes are the oracle's codes
            got = x["k_pages"][pages].cpu().numpy().reshape(-1, w.head_dim)[:K.shape[0]]
            assert np.array_equal(got, kcodes)
        qg = x["q"][b, kvh * g:(kvh + 1) * g].float().cpu().numpy().astype(np.float64)
        r = O.decode_pair(qg, K, V, w.block_size, w.kv_dtype, w.sink_tokens, w.window_tokens,
                          w.k_scored, 1 / math.sqrt(w.head_dim))
        got_sel = sel[b, kvh, :cnt[b, kvh]].tolist()
        assert tie_window_ok(r["score"], r["forced"], got_sel, r["sel"], w.k_scored), (b, kvh)
        if set(got_sel) == set(r["sel"]):
            ref = r["out"]
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
            assert np.all(np.abs(out[b, kvh * g:(kvh + 1) * g] - ref) <= np.maximum(tol, ulp)), (b, kvh)


@pytest.mark.parametrize("name,samples", [
    ("llama8b_bf16", [(0, 0), (3, 2), (7, 3)]),
    ("ragged_bf16", [(0, 0), (17, 1), (63, 3)]),
    ("fp8_g32", [(0, 0), (31, 3)]),
])
def test_full_size_step(name, samples):
    from query_aware_sparse_hs_gb300 import hs
    from query_aware_sparse_hs_gb300.decode import SparseDecode
    w = WORKLOADS[name]
    x = _dev_inputs(w)
    kv = hs.paged_kv(x["k_pages"], x["v_pages"], x["page_table"], x["seq_lens"],
                     x.get("k_scales"), x.get("v_scales"))
    dec = SparseDecode(num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                       block_size=w.block_size, kv_dtype=w.kv_dtype, batch=w.batch, max_blocks=w.max_blocks,
                       sink_tokens=w.sink_tokens, window_tokens=w.window_tokens, k_scored=w.k_scored)
    dec.build_summaries(kv)
    last_block = int((x["seq_lens"].min().item() - 1) // w.block_size)
    dec.step(kv, x["q"], refresh_from_block=last_block)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_OK, bits
    _check_pairs(w, x, dec, samples, tol=2e-3)


@pytest.mark.parametrize("overlap", [False, True])
def test_full_size_offload_steps(overlap):
    """256 requests x 32768 tokens with 64 hot slots per (request, kv head): the
    hot-buffer tables of sampled pairs follow the oracle's simulator exactly over
    several drifting decode steps, and the attention on the hot slots matches -
    with the swap-in in one call, and overlapped (page copy and attention over
    the copied blocks on 12 SMs beside attention over the resident blocks)."""
    from query_aware_sparse_hs_gb300 import hs
    from query_aware_sparse_hs_gb300.decode import SparseDecode
    from _parity import tie_window_ok
    w = WORKLOADS["offload_bf16"]
    steps = 6
    x = make_inputs(w, device="cuda")
    B, D, S, hkv, g, nb = w.block_size, w.head_dim, w.hot_slots, w.num_kv_heads, w.group, w.max_blocks
    pairs = w.batch * hkv
    host_k = torch.empty(x["k_pages"].shape, dtype=torch.bfloat16, pin_memory=True)
    host_v = torch.empty_like(host_k, pin_memory=True)
    host_k.copy_(x["k_pages"])
    host_v.copy_(x["v_pages"])
    qs = drift_queries(w, x["q"], steps)
    del x["k_pages"], x["v_pages"]
    torch.cuda.empty_cache()
    dev = torch.device("cuda")
    pool_kv = hs.paged_kv(host_k, host_v, x["page_table"], x["seq_lens"])
    table = torch.full((w.batch, hkv, nb), -1, dtype=torch.int32, device=dev)
    owner = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
    last = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
    k_slots = torch.zeros((pairs * S, B, D), dtype=torch.bfloat16, device=dev)
    v_slots = torch.zeros_like(k_slots)
    hb = hs.hot_buffer(table, owner, last, k_slots, v_slots, host_k, host_v, S)
    slot_kv = hs.paged_kv(k_slots, v_slots, table, x["seq_lens"])
    stats = torch.zeros(4, dtype=torch.int64, device=dev)
    dec = SparseDecode(num_q_heads=w.num_q_heads, num_kv_heads=hkv, head_dim=D, block_size=B, kv_dtype="bf16",
                       batch=w.batch, max_blocks=nb, sink_tokens=w.sink_tokens, window_tokens=w.window_tokens,
                       k_scored=w.k_scored)
    if overlap:
        dec.enable_swap_overlap()
    dec.build_summaries(pool_kv)
    samples = [(0, 0), (100, 2), (255, 3)]
    L = w.ctx_max
    F = O.forced_blocks(L, B, w.sink_tokens, w.window_tokens)
    orc = {}
    for b, kvh in samples:
        K = O.kv_values("bf16", host_k[b * hkv * nb + kvh * nb:b * hkv * nb + (kvh + 1) * nb].float().numpy().reshape(-1, D))
        V = O.kv_values("bf16", host_v[b * hkv * nb + kvh * nb:b * hkv * nb + (kvh + 1) * nb].float().numpy().reshape(-1, D))
        smin, smax = O.stored_summaries(*O.block_summaries(K, B), "bf16")
        orc[(b, kvh)] = (K, V, smin, smax, O.HotBuffer(nb, S, base=(b * hkv + kvh) * S), True)
    for t in range(steps):
        q = qs[t].contiguous()
        dec.step(pool_kv, q, hot=(hb, slot_kv, t, stats))
        st, bits = hs.hs_get_device_error()
        assert st == hs.HS_OK, bits
        sel, cnt = dec.sel.cpu().numpy(), dec.sel_count.cpu().numpy()
        gt, go, gl = table.cpu().numpy(), owner.cpu().numpy(), last.cpu().numpy()
        out = dec.out.float().cpu().numpy()
        for b, kvh in samples:
            K, V, smin, smax, sim, same = orc[(b, kvh)]
            qg = q[b, kvh * g:(kvh + 1) * g].float().cpu().numpy().astype(np.float64)
            _, score = O.bound_scores(qg, smin, smax)
            s = O.select_blocks(score, F, w.k_scored)
            got = sel[b, kvh, :cnt[b, kvh]].tolist()
            assert tie_window_ok(score, F, got, s, w.k_scored)
            same = same and set(got) == set(s)
            sim.step(s, t)
            if same:  # identical selections so far: the tables must be identical
                assert gt[b, kvh].tolist() == sim.page_table
                assert go[b, kvh].tolist() == sim.slot_owner
                assert gl[b, kvh].tolist() == sim.last_used
                ref, _ = O.sparse_attention(qg, K, V, s, B, 1 / math.sqrt(D))
                ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
                assert np.all(np.abs(out[b, kvh * g:(kvh + 1) * g] - ref) <= np.maximum(2e-3, ulp))
            orc[(b, kvh)] = (K, V, smin, smax, sim, same)
    st = stats.cpu().numpy()
    assert st[0] + st[1] == steps * pairs * 32  # every selected block is a hit or a miss
    assert st[1] >= pairs * 32  # the first step misses everything
