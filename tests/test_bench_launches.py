"""The bench's count of its own kernel launches per step follows the library's
dispatch (CPU only: the library's geometry query and the device properties
are replaced by fixed answers; nothing is launched)."""

import bench
from synth import WORKLOADS


class _Props:
    multi_processor_count = 152


def _decoder(w):
    from query_aware_sparse_hs_gb300.decode import SparseDecode
    return SparseDecode(num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                        block_size=w.block_size, kv_dtype=w.kv_dtype, batch=w.batch, max_blocks=w.max_blocks,
                        sink_tokens=w.sink_tokens, window_tokens=w.window_tokens, k_scored=w.k_scored,
                        device="cpu")


def test_step_launches_follow_the_dispatch(monkeypatch):
    import torch
    from query_aware_sparse_hs_gb300 import hs
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda *a, **k: _Props())
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    w = WORKLOADS["llama8b_bf16"]
    dec = _decoder(w)
    # 4 splits per (request, kv head), each with a CTA of its own
    assert bench.attn_splits(w, dec) == 4
    monkeypatch.setattr(hs, "hs_score_select_attend_fused", lambda *a: 1)
    assert bench.fused_step(w, dec)
    assert bench.step_launches(w, dec) == 1  # append, scoring, selection and attention in one launch
    # the same step without the single launch: append, scoring + selection in
    # one cluster launch, attention merging its splits itself
    assert bench.select_launches(w) == 1
    assert bench.step_launches(w, dec, allow_fused=False) == 3
    monkeypatch.setattr(hs, "hs_score_select_attend_fused", lambda *a: 0)
    assert not bench.fused_step(w, dec)
    assert bench.step_launches(w, dec) == 3
    # without split counters the separate attention needs the merge launch
    dec.split_counters = None
    assert bench.step_launches(w, dec) == 4
    # the single launch merges its splits inside its clusters, with or without counters
    monkeypatch.setattr(hs, "hs_score_select_attend_fused", lambda *a: 1)
    assert bench.step_launches(w, dec) == 1
    monkeypatch.setattr(hs, "hs_score_select_attend_fused", lambda *a: 0)
    # a decoder that does not use the combined call never counts it
    dec.fuse_step = False
    monkeypatch.setattr(hs, "hs_score_select_attend_fused", lambda *a: 1)
    assert bench.step_launches(w, dec) == 4


def test_ragged_selection_takes_two_launches(monkeypatch):
    import torch
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda *a, **k: _Props())
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    # 8192 blocks per request: more than 8 tiles, scoring and selection are separate launches
    assert bench.select_launches(WORKLOADS["ragged_bf16"]) == 2
    assert bench.select_launches(WORKLOADS["llama8b_bf16"]) == 1
