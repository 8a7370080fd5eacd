"""The seeded input recipes produce what they claim (CPU, reduced sizes)."""

import math

import torch

from synth import WORKLOADS, drift_queries, make_inputs, make_layout


def test_layout_is_a_bijection_onto_the_pool():
    w = WORKLOADS["ragged_bf16"].scaled(batch=5, ctx_min=40, ctx_max=300)
    lay = make_layout(w)
    lens = lay["seq_lens"].tolist()
    assert all(40 <= L <= 300 for L in lens)
    t = lay["page_table"]
    assert t.shape == (5, 4, w.max_blocks)
    ids = t[t >= 0]
    assert ids.numel() == lay["num_pages"]
    assert torch.equal(torch.sort(ids).values, torch.arange(lay["num_pages"], dtype=torch.int32))
    for b, L in enumerate(lens):
        nb = -(-L // w.block_size)
        assert bool((t[b, :, :nb] >= 0).all()) and bool((t[b, :, nb:] == -1).all())


def test_offload_pool_is_in_logical_order():
    w = WORKLOADS["offload_bf16"].scaled(batch=2, ctx_min=256, ctx_max=256)
    lay = make_layout(w)
    t = lay["page_table"]
    assert torch.equal(t.flatten(), torch.arange(2 * 4 * 4, dtype=torch.int32))


def test_heavy_hitters_and_query_correlation():
    w = WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=2048, ctx_max=2048)
    x = make_inputs(w)
    B = w.block_size
    k = x["k_pages"].float()
    t = x["page_table"].long()
    for idx, pos in enumerate(x["heavy"]):
        b, kvh = divmod(idx, 4)
        assert pos.numel() == round(0.02 * 2048)
        rows = k[t[b, kvh, pos // B], pos % B]
        assert 3.0 < rows.norm(dim=1).mean().item() / math.sqrt(128) < 5.0
    # every query has norm sqrt(D) and a large dot product with some heavy rows
    q = x["q"].float()
    assert torch.allclose(q.norm(dim=-1), torch.full((2, 32), math.sqrt(128)), rtol=2e-2)
    for b in range(2):
        for h in range(32):
            pos = x["heavy"][b * 4 + h // 8]
            rows = k[t[b, h // 8, pos // B], pos % B]
            top = (rows @ q[b, h]).topk(8).values
            assert top.min() > 40  # about 0.6 * |q| * |k| / sqrt(8)


def test_inputs_are_deterministic():
    w = WORKLOADS["tiny_f32"]
    a, b = make_inputs(w), make_inputs(w)
    for key in ("k_pages", "v_pages", "q", "page_table", "seq_lens"):
        assert torch.equal(a[key], b[key])
    assert a["k_pages"].dtype == torch.float32 and a["q"].shape == (1, 8, 64)


def test_drift_keeps_the_norm():
    w = WORKLOADS["offload_bf16"].scaled(batch=2, ctx_min=256, ctx_max=256)
    x = make_inputs(w)
    qs = drift_queries(w, x["q"], steps=5)
    assert torch.equal(qs[0], x["q"])
    n0 = x["q"].float().norm(dim=-1)
    for s in range(1, 5):
        assert torch.allclose(qs[s].float().norm(dim=-1), n0, rtol=1e-2)
        assert not torch.equal(qs[s], qs[s - 1])


def test_drift_sigma_is_the_calibrated_one():
    import json
    import os
    from synth import DRIFT_SIGMA
    with open(os.path.join(os.path.dirname(__file__), "golden", "drift_sigma.json")) as f:
        cal = json.load(f)
    assert DRIFT_SIGMA == cal["sigma"]
    assert abs(cal["mean_overlap"] - 0.85) <= 0.02
