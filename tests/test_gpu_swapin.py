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


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_swapin_tables_bit_exact_and_attention(kv_dtype):
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
        for b in range(w.batch):
            for kvh in range(hkv):
                K, V, smin, smax = KV[(b, kvh)]
                qg = q[b, kvh * g:(kvh + 1) * g].float().numpy().astype(np.float64)
                _, score = O.bound_scores(qg, smin, smax)
                s = O.select_blocks(score, O.forced_blocks(K.shape[0], B, w.sink_tokens, w.window_tokens),
                                    w.k_scored)
                sel[b, kvh, :len(s)] = s
                cnt[b, kvh] = len(s)
                _, st_ = sim[b * hkv + kvh].step(s, t)
                want += [st_["hits"], st_["misses"], st_["evictions"]]
                total_misses += st_["misses"]
                ref[b, kvh * g:(kvh + 1) * g] = O.sparse_attention(qg, K, V, s, B, 1 / math.sqrt(D))[0]
        dec.sel.copy_(torch.from_numpy(sel))
        dec.sel_count.copy_(torch.from_numpy(cnt))
        dec.swap_in(hb, t, stats)
        qd = q.to(dev)
        dec.attend(slot_kv, qd)
        st, bits = hs.hs_get_device_error()
        assert st == 0, bits
        gt, go, gl = hot_table.cpu().numpy(), owner.cpu().numpy(), last.cpu().numpy()
        for p in range(pairs):
            b, kvh = divmod(p, hkv)
            assert gt[b, kvh].tolist() == sim[p].page_table, (t, p)
            assert go[b, kvh].tolist() == sim[p].slot_owner, (t, p)
            assert gl[b, kvh].tolist() == sim[p].last_used, (t, p)
        tol = 2e-3
        assert np.abs(dec.out.cpu().numpy() - ref).max() <= tol, t
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
