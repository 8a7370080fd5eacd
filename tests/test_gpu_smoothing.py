"""Score smoothing across decode steps (SparDA article §6.1) through the C ABI:
over several steps of a drifting query, the smoothed scores the library keeps
as history follow the oracle's recursion on its own bound scores, and every
selection is the oracle's top-k of the smoothed scores (up to near-ties).
Both scoring paths: tensor-core bound scoring + selection (bf16, head_dim
128) and the fused CUDA-core cluster kernel (fp32, head_dim 64).  GPU only.
"""

import numpy as np
import pytest
import torch

import oracle as O
from synth import WORKLOADS, drift_queries, make_inputs

pytestmark = pytest.mark.gpu

WEIGHT = 0.3
CASES = {
    "bf16_d128_tensor_cores": WORKLOADS["llama8b_bf16"].scaled(batch=3, ctx_min=2000, ctx_max=5000, k_scored=9),
    "f32_d64_cluster": WORKLOADS["tiny_f32"].scaled(batch=2, ctx_min=900, ctx_max=2048),
}


@pytest.mark.parametrize("name", list(CASES))
def test_smoothed_selection_follows_the_oracle(name):
    from _parity import Case, tie_window_ok
    from query_aware_sparse_hs_gb300 import hs
    w = CASES[name]
    c = Case(w, make_inputs(w))
    dec = c.decoder(score_smoothing=WEIGHT)
    dec.build_summaries(c.kv)
    steps = 5
    qs = drift_queries(w, c.x["q"], steps)
    B = w.block_size
    pairs = [(b, kvh) for b in range(w.batch) for kvh in range(w.num_kv_heads)]
    summ = {}
    for b, kvh in pairs:
        K = c.logical(b, kvh, "k")
        summ[(b, kvh)] = O.stored_summaries(*O.block_summaries(K, B), w.kv_dtype)
    hist = {p: None for p in pairs}
    changed = 0
    for t in range(steps):
        q = qs[t].to(c.q.device).contiguous()
        dec.select(c.kv, q, keep_scores=True)
        st, bits = hs.hs_get_device_error()
        assert st == hs.HS_OK, bits
        got_hist = dec.score_history.cpu().numpy()
        sel, cnt = dec.sel.cpu().numpy(), dec.sel_count.cpu().numpy()
        for b, kvh in pairs:
            smin, smax = summ[(b, kvh)]
            g = w.group
            qg = q[b, kvh * g:(kvh + 1) * g].float().cpu().numpy().astype(np.float64)
            _, raw = O.bound_scores(qg, smin, smax)
            h = np.full(raw.shape, np.nan) if hist[(b, kvh)] is None else hist[(b, kvh)]
            sm = O.smooth_scores(raw, h, WEIGHT)
            hist[(b, kvh)] = sm
            nb = len(raw)
            mag = (np.abs(qg)[:, None, :] * np.maximum(np.abs(smin), np.abs(smax))[None]).sum(-1).max(0)
            assert np.all(np.abs(got_hist[b, kvh, :nb] - sm) <= 1e-5 * mag + 1e-30), (t, b, kvh)
            F = O.forced_blocks(c.lens[b], B, w.sink_tokens, w.window_tokens)
            want = O.select_blocks(sm, F, w.k_scored)
            got = sel[b, kvh, :cnt[b, kvh]].tolist()
            assert tie_window_ok(sm, F, got, want, w.k_scored), (t, b, kvh)
            if t > 0 and want != O.select_blocks(raw, F, w.k_scored):
                changed += 1
    # the smoothing is not a no-op on this input: it changes some selections
    assert changed > 0


def test_smoothing_off_leaves_no_history_and_weight_is_checked():
    from _parity import Case
    from query_aware_sparse_hs_gb300 import hs
    w = CASES["bf16_d128_tensor_cores"]
    c = Case(w, make_inputs(w))
    dec = c.decoder()
    assert dec.score_history is None
    dec.build_summaries(c.kv)
    bad = hs.select_params(w.sink_tokens, w.window_tokens, w.k_scored, dec.capacity, 1.0, torch.zeros(4).cuda())
    with pytest.raises(hs.HSError) as e:
        hs.hs_score_select_topk(dec.shape, c.kv, c.q, dec.smin, dec.smax, bad, dec.sel, dec.sel_count, dec.scores)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    missing = hs.select_params(w.sink_tokens, w.window_tokens, w.k_scored, dec.capacity, 0.3, None)
    with pytest.raises(hs.HSError):
        hs.hs_score_select_topk(dec.shape, c.kv, c.q, dec.smin, dec.smax, missing, dec.sel, dec.sel_count,
                                dec.scores)
