"""HiSparse swap-in on the GPU vs the oracle's hot-buffer simulator: page table,
slot owners and last-used stamps bit-exact after every step, slot contents equal
to the host pool, attention on the hot slots within tolerance.  GPU only."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import WORKLOADS, drift_queries, make_inputs

pytestmark = pytest.mark.gpu


def _setup(kv_dtype="bf16", batch=2, blocks=48, slots=16, k_scored=7):
    base = WORKLOADS["offload_bf16"] if kv_dtype == "bf16" else WORKLOADS["fp8_g32"]
    w = base.scaled(batch=batch, ctx_min=64 * blocks, ctx_max=64 * blocks, k_scored=k_scored,
                    hot_slots=slots, decode_steps=12)
    x = make_inputs(w)
    return w, x


def _pool(w, x):
    """Pinned host pool in logical order [b][kvh][j][B][D] (+ e4m3 scales)."""
    D = w.head_dim
    if w.kv_dtype == "fp8":
        kc, ks = O.quantize_e4m3_g32(x["k_pages"].float().numpy().reshape(-1, D))
        vc, vs = O.quantize_e4m3_g32(x["v_pages"].float().numpy().reshape(-1, D))
        shp = x["k_pages"].shape
        hk = torch.from_numpy(kc.reshape(shp)).pin_memory()
        hv = torch.from_numpy(vc.reshape(shp)).pin_memory()
        hks = torch.from_numpy(ks.reshape(shp[0], shp[1], D // 32)).pin_memory()
        hvs = torch.from_numpy(vs.reshape(shp[0], shp[1], D // 32)).pin_memory()
        return hk, hv, hks, hvs
    return x["k_pages"].pin_memory(), x["v_pages"].pin_memory(), None, None


@pytest.mark.parametrize("mode", ["one_call", "overlapped"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_swapin_tables_bit_exact_and_attention(kv_dtype, mode):
    """one_call: hs_swapin_misses then attention over the selection.
    overlapped: plan -> copy on a side stream (3 CTAs, several streams each)
    beside attention over the hits -> attention over the misses -> LSE merge;
    the hit and miss lists must be the oracle's partition of the selection."""
    from query_aware_sparse_hs_gb300 import hs
    from query_aware_sparse_hs_gb300.decode import SparseDecode
    w, x = _setup(kv_dtype)
    B, D, S, hkv, g = w.block_size, w.head_dim, w.hot_slots, w.num_kv_heads, w.group
    nb = w.max_blocks
    hk, hv, hks, hvs = _pool(w, x)
    dev = torch.device("cuda")
    lens = x["seq_lens"].to(dev)
    pool_table = x["page_table"].to(dev)  # identity over the pool
    pool_kv = hs.paged_kv(hk, hv, pool_table, lens, hks, hvs)
    pairs = w.batch * hkv
    hot_table = torch.full((w.batch, hkv, nb), -1, dtype=torch.int32, device=dev)
    owner = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
    last = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
    kdt = torch.uint8 if kv_dtype == "fp8" else torch.bfloat16
    k_slots = torch.zeros((pairs * S, B, D), dtype=kdt, device=dev)
    v_slots = torch.zeros_like(k_slots)
    ks_slots = vs_slots = None
    if kv_dtype == "fp8":
        ks_slots = torch.zeros((pairs * S, B, D // 32), dtype=torch.float32, device=dev)
        vs_slots = torch.zeros_like(ks_slots)
    hb = hs.hot_buffer(hot_table, owner, last, k_slots, v_slots, hk, hv, S, ks_slots, vs_slots, hks, hvs)
    slot_kv = hs.paged_kv(k_slots, v_slots, hot_table, lens, ks_slots, vs_slots)
    stats = torch.zeros(4, dtype=torch.int64, device=dev)
    dec = SparseDecode(num_q_heads=w.num_q_heads, num_kv_heads=hkv, head_dim=D, block_size=B,
                       kv_dtype=kv_dtype, batch=w.batch, max_blocks=nb, sink_tokens=w.sink_tokens,
                       window_tokens=w.window_tokens, k_scored=w.k_scored, out_is_fp32=True)
    if mode == "overlapped":
        dec.enable_swap_overlap(copy_ctas=3)
    dec.build_summaries(pool_kv)  # summaries read the pinned pool directly
    st, bits = hs.hs_get_device_error()
    assert st == 0, bits
    qs = drift_queries(w, x["q"], 12)
    sim = [O.HotBuffer(nb, S, base=p * S) for p in range(pairs)]
    # oracle logical K/V per pair (values the kernel sees)
    hk_np = hk.float().numpy() if kv_dtype != "fp8" else hk.numpy()
    hv_np = hv.float().numpy() if kv_dtype != "fp8" else hv.numpy()
    KV = {}
    for b in range(w.batch):
        for kvh in range(hkv):
            row = x["page_table"][b, kvh].numpy()
            L = int(x["seq_lens"][b])
            if kv_dtype == "fp8":
                K = O.kv_values("fp8", O.gather_rows(hk_np, row, L, B), O.gather_rows(hks.numpy(), row, L, B))
                V = O.kv_values("fp8", O.gather_rows(hv_np, row, L, B), O.gather_rows(hvs.numpy(), row, L, B))
            else:
                K = O.kv_values("bf16", O.gather_rows(hk_np, row, L, B))
                V = O.kv_values("bf16", O.gather_rows(hv_np, row, L, B))
            smin, smax = O.stored_summaries(*O.block_summaries(K, B), kv_dtype)
            KV[(b, kvh)] = (K, V, smin, smax)
    want = np.zeros(3, dtype=np.int64)
    total_misses = 0
    for t in range(12):
        q = qs[t]
        sel = np.full((w.batch, hkv, dec.capacity), -1, dtype=np.int32)
        cnt = np.zeros((w.batch, hkv), dtype=np.int32)
        ref = np.zeros((w.batch, w.num_q_heads, D))
        ref_lse = np.zeros((w.batch, w.num_q_heads))
        parts = {}
        for b in range(w.batch):
            for kvh in range(hkv):
                K, V, smin, smax = KV[(b, kvh)]
                qg = q[b, kvh * g:(kvh + 1) * g].float().numpy().astype(np.float64)
                _, score = O.bound_scores(qg, smin, smax)
                s = O.select_blocks(score, O.forced_blocks(K.shape[0], B, w.sink_tokens, w.window_tokens),
                                    w.k_scored)
                sel[b, kvh, :len(s)] = s
                cnt[b, kvh] = len(s)
                resident = {j for j, e in enumerate(sim[b * hkv + kvh].page_table) if e >= 0}
                parts[(b, kvh)] = ([j for j in s if j in resident], [j for j in s if j not in resident])
                _, st_ = sim[b * hkv + kvh].step(s, t)
                want += [st_["hits"], st_["misses"], st_["evictions"]]
                total_misses += st_["misses"]
                o_, l_ = O.sparse_attention(qg, K, V, s, B, 1 / math.sqrt(D))
                ref[b, kvh * g:(kvh + 1) * g], ref_lse[b, kvh * g:(kvh + 1) * g] = o_, l_
        dec.sel.copy_(torch.from_numpy(sel))
        dec.sel_count.copy_(torch.from_numpy(cnt))
        qd = q.to(dev)
        if mode == "one_call":
            dec.swap_in(hb, t, stats)
            dec.attend(slot_kv, qd)
        else:
            dec.swap_in_overlapped(hb, slot_kv, qd, t, stats)
        st, bits = hs.hs_get_device_error()
        assert st == 0, bits
        if mode == "overlapped":
            hs_, hc = dec.hit_sel.cpu().numpy(), dec.hit_count.cpu().numpy()
            ms_, mc = dec.miss_sel.cpu().numpy(), dec.miss_count.cpu().numpy()
            for (b, kvh), (hits, misses) in parts.items():
                assert hc[b, kvh] == len(hits) and mc[b, kvh] == len(misses), (t, b, kvh)
                assert hs_[b, kvh].tolist() == hits + [-1] * (dec.capacity - len(hits))
                assert ms_[b, kvh].tolist() == misses + [-1] * (dec.capacity - len(misses))
        gt, go, gl = hot_table.cpu().numpy(), owner.cpu().numpy(), last.cpu().numpy()
        for p in range(pairs):
            b, kvh = divmod(p, hkv)
            assert gt[b, kvh].tolist() == sim[p].page_table, (t, p)
            assert go[b, kvh].tolist() == sim[p].slot_owner, (t, p)
            assert gl[b, kvh].tolist() == sim[p].last_used, (t, p)
        tol = 2e-3
        assert np.abs(dec.out.cpu().numpy() - ref).max() <= tol, t
        assert np.abs(dec.lse.cpu().numpy() - ref_lse).max() <= 1e-4, t
    # slot contents equal the pool pages they hold
    ks_np = k_slots.cpu()
    for p in range(pairs):
        b, kvh = divmod(p, hkv)
        for s_, j in enumerate(sim[p].slot_owner):
            if j >= 0:
                src = int(x["page_table"][b, kvh, j])
                assert torch.equal(ks_np[p * S + s_], hk[src])
    got = stats.cpu().numpy()
    assert got[:3].tolist() == want.tolist()
    elem = 1 if kv_dtype == "fp8" else 2
    sc = B * (D // 32) * 4 if kv_dtype == "fp8" else 0
    assert got[3] == total_misses * 2 * (B * D * elem + sc)


def test_swapin_capacity_error_leaves_tables():
    from query_aware_sparse_hs_gb300 import hs
    w, x = _setup("bf16", batch=1, blocks=20, slots=4, k_scored=7)
    dev = torch.device("cuda")
    B, D, S, hkv = w.block_size, w.head_dim, 4, w.num_kv_heads
    hk, hv, _, _ = _pool(w, x)
    table = torch.full((1, hkv, 20), -1, dtype=torch.int32, device=dev)
    owner = torch.full((1, hkv, S), -1, dtype=torch.int32, device=dev)
    last = torch.full((1, hkv, S), -1, dtype=torch.int32, device=dev)
    ks = torch.zeros((hkv * S, B, D), dtype=torch.bfloat16, device=dev)
    hb = hs.hot_buffer(table, owner, last, ks, ks.clone(), hk, hv, S)
    sel = torch.arange(6, dtype=torch.int32, device=dev).repeat(1, hkv, 1).contiguous()
    cnt = torch.full((1, hkv), 6, dtype=torch.int32, device=dev)
    shape = hs.attn_shape(w.num_q_heads, hkv, D, B, "bf16")
    hs.hs_swapin_misses(shape, hb, sel, cnt, 6, 0)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_ERR_CAPACITY and bits & hs.HS_EBIT_CAPACITY
    assert bool((table == -1).all()) and bool((owner == -1).all())


@pytest.mark.parametrize("out_fp32", [True, False])
def test_merge_attn_partials_matches_the_oracle(out_fp32):
    """Three partials per row, some of them empty (lse = -inf, out = 0), one
    row with every part empty; against the oracle's LSE merge row by row."""
    from query_aware_sparse_hs_gb300 import hs
    parts, batch, hq, D = 3, 2, 8, 128
    g = torch.Generator().manual_seed(7)
    outs = torch.randn((parts, batch, hq, D), generator=g)
    lses = torch.randn((parts, batch, hq), generator=g) * 4
    lses[0, 0, 1] = -math.inf
    lses[1, 1, 2] = lses[2, 1, 2] = -math.inf
    lses[:, 1, 5] = -math.inf
    outs[lses == -math.inf] = 0.0
    shape = hs.attn_shape(hq, 2, D, 64, "bf16")
    out = torch.empty((batch, hq, D), dtype=torch.float32 if out_fp32 else torch.bfloat16, device="cuda")
    lse = torch.empty((batch, hq), device="cuda")
    hs.hs_merge_attn_partials(shape, outs.cuda(), lses.cuda(), out, lse)
    st, bits = hs.hs_get_device_error()
    assert st == 0, bits
    got, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(batch):
        for h in range(hq):
            ref, ref_lse = O.lse_merge([outs[p, b, h].numpy() for p in range(parts)], lses[:, b, h].numpy())
            tol = 1e-5 if out_fp32 else np.maximum(1e-5, np.abs(ref) * 2.0 ** -8)
            assert np.all(np.abs(got[b, h] - ref) <= tol), (b, h)
            if np.isneginf(ref_lse):
                assert np.isneginf(got_lse[b, h]) and np.all(got[b, h] == 0)
            else:
                assert abs(got_lse[b, h] - ref_lse) <= 1e-5 * max(1.0, abs(ref_lse)), (b, h)


def test_plan_then_copy_equals_the_one_call_swapin():
    """hs_swapin_plan + hs_swapin_copy (2 CTAs) leave the same tables and slot
    contents as hs_swapin_misses, over several steps of a drifting selection."""
    from query_aware_sparse_hs_gb300 import hs
    w, x = _setup("bf16", batch=2, blocks=40, slots=12, k_scored=6)
    dev = torch.device("cuda")
    B, D, S, hkv, nb = w.block_size, w.head_dim, w.hot_slots, w.num_kv_heads, w.max_blocks
    hk, hv, _, _ = _pool(w, x)
    pairs, cap = w.batch * hkv, 12
    shape = hs.attn_shape(w.num_q_heads, hkv, D, B, "bf16")

    def buffer():
        t = torch.full((w.batch, hkv, nb), -1, dtype=torch.int32, device=dev)
        o = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
        l = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
        k = torch.zeros((pairs * S, B, D), dtype=torch.bfloat16, device=dev)
        v = torch.zeros_like(k)
        return hs.hot_buffer(t, o, l, k, v, hk, hv, S), (t, o, l, k, v)

    hb1, st1 = buffer()
    hb2, st2 = buffer()
    g = torch.Generator().manual_seed(3)
    lists = [torch.full((w.batch, hkv, cap), -1, dtype=torch.int32, device=dev) for _ in range(2)]
    counts = [torch.zeros((w.batch, hkv), dtype=torch.int32, device=dev) for _ in range(2)]
    stats1 = torch.zeros(4, dtype=torch.int64, device=dev)
    stats2 = torch.zeros(4, dtype=torch.int64, device=dev)
    for t in range(6):
        sel = torch.full((w.batch, hkv, cap), -1, dtype=torch.int32)
        cnt = torch.zeros((w.batch, hkv), dtype=torch.int32)
        for p in range(pairs):
            k = int(torch.randint(1, cap + 1, (1,), generator=g))
            pick = torch.sort(torch.randperm(nb, generator=g)[:k]).values
            sel.view(pairs, cap)[p, :k] = pick.int()
            cnt.view(pairs)[p] = k
        sel, cnt = sel.to(dev), cnt.to(dev)
        hs.hs_swapin_misses(shape, hb1, sel, cnt, cap, t, stats1)
        hs.hs_swapin_plan(shape, hb2, sel, cnt, cap, t, lists[0], counts[0], lists[1], counts[1], stats2)
        hs.hs_swapin_copy(shape, hb2, lists[1], counts[1], cap, 2, stats2)
        st, bits = hs.hs_get_device_error()
        assert st == 0, bits
        for a, b in zip(st1, st2):
            assert torch.equal(a, b), t
    assert torch.equal(stats1, stats2)


def test_select_plan_in_one_launch_equals_the_two_calls():
    """hs_score_select_swapin_plan (each stream's plan in the selection's
    launch once the scoring takes more than one wave) leaves the same
    selection, hit and miss lists, tables and statistics as
    hs_score_select_topk followed by hs_swapin_plan, over drifting steps."""
    from query_aware_sparse_hs_gb300 import hs
    from query_aware_sparse_hs_gb300.decode import SparseDecode
    # 160 (request, kv head) pairs of one 128-block tile: more than one wave of the scorer
    w, x = _setup("bf16", batch=40, blocks=48, slots=16, k_scored=7)
    dev = torch.device("cuda")
    B, D, S, hkv, nb = w.block_size, w.head_dim, w.hot_slots, w.num_kv_heads, w.max_blocks
    hk, hv, _, _ = _pool(w, x)
    lens = x["seq_lens"].to(dev)
    pool_kv = hs.paged_kv(hk, hv, x["page_table"].to(dev), lens)
    pairs = w.batch * hkv

    def side():
        t = torch.full((w.batch, hkv, nb), -1, dtype=torch.int32, device=dev)
        o = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
        l = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
        k = torch.zeros((pairs * S, B, D), dtype=torch.bfloat16, device=dev)
        d = SparseDecode(num_q_heads=w.num_q_heads, num_kv_heads=hkv, head_dim=D, block_size=B, kv_dtype="bf16",
                         batch=w.batch, max_blocks=nb, sink_tokens=w.sink_tokens, window_tokens=w.window_tokens,
                         k_scored=w.k_scored)
        d.build_summaries(pool_kv)
        lists = [torch.full_like(d.sel, -1) for _ in range(2)] + [torch.zeros_like(d.sel_count) for _ in range(2)]
        return hs.hot_buffer(t, o, l, k, torch.zeros_like(k), hk, hv, S), (t, o, l), d, lists, \
            torch.zeros(4, dtype=torch.int64, device=dev)

    hb1, tab1, d1, l1, st1 = side()
    hb2, tab2, d2, l2, st2 = side()
    qs = drift_queries(w, x["q"], 6)
    for t in range(6):
        q = qs[t]
        d1.select(pool_kv, q)
        hs.hs_swapin_plan(d1.shape, hb1, d1.sel, d1.sel_count, d1.capacity, t, l1[0], l1[2], l1[1], l1[3], st1)
        hs.hs_score_select_swapin_plan(d2.shape, pool_kv, q, d2.smin, d2.smax, d2.sel_params, d2.sel, d2.sel_count,
                                       hb2, t, l2[0], l2[2], l2[1], l2[3], scores=d2.scores, stats=st2)
        st, bits = hs.hs_get_device_error()
        assert st == 0, bits
        assert torch.equal(d1.sel, d2.sel) and torch.equal(d1.sel_count, d2.sel_count), t
        assert torch.equal(d1.scores, d2.scores), t
        for a, b in zip(l1, l2):
            assert torch.equal(a, b), t
        for a, b in zip(tab1, tab2):
            assert torch.equal(a, b), t
    assert torch.equal(st1, st2)
    assert int(st1[1]) > 0  # the drift brought misses in
