"""Selection reuse (SparDA article §3.1 and §3.3): the block selection made at
one layer is reused by the following layers, each attending with its own query
and its own K/V over the same blocks; a later decode step may also reuse an
earlier step's selection.  Checked through the C ABI against the oracle's
attention over the reused selection.  GPU only.
"""

import math

import numpy as np
import pytest

import oracle as O
from synth import WORKLOADS, make_layer, make_layout

pytestmark = pytest.mark.gpu

TOL = 2e-3  # the fp32-output attention tolerance of the parity tests


def _layers(w, n):
    from _parity import Case
    layout = make_layout(w)
    return [Case(w, dict(layout, **make_layer(w, layout, "cpu", l))) for l in range(n)]


def test_deeper_layers_attend_over_the_first_layers_selection():
    from _parity import tie_window_ok
    from query_aware_sparse_hs_gb300 import hs
    w = WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=3000, ctx_max=5000, k_scored=9)
    cases = _layers(w, 3)
    decs = [c.decoder(out_is_fp32=True) for c in cases]
    decs[0].build_summaries(cases[0].kv)
    decs[0].step(cases[0].kv, cases[0].q)
    for l in (1, 2):
        decs[l].step(cases[l].kv, cases[l].q, reuse=decs[0])
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_OK, bits
    sel, cnt = decs[0].sel.cpu().numpy(), decs[0].sel_count.cpu().numpy()
    B, scale = w.block_size, 1.0 / math.sqrt(w.head_dim)
    g = w.group
    for b in range(w.batch):
        for kvh in range(w.num_kv_heads):
            r = cases[0].oracle_pair(b, kvh)
            got = sel[b, kvh, :cnt[b, kvh]].tolist()
            assert tie_window_ok(r["score"], r["forced"], got, r["sel"], w.k_scored)
            for l in (1, 2):
                c = cases[l]
                K, V = c.logical(b, kvh, "k"), c.logical(b, kvh, "v")
                ref, _ = O.sparse_attention(c.q_group(b, kvh), K, V, got, B, scale)
                out = decs[l].out[b, kvh * g:(kvh + 1) * g].cpu().numpy()
                assert np.abs(out - ref).max() <= TOL, (l, b, kvh)
    # the deeper layers never selected anything themselves
    for l in (1, 2):
        assert bool((decs[l].sel == -1).all()) and bool((decs[l].sel_count == 0).all())


def test_a_later_step_reuses_the_earlier_selection():
    from query_aware_sparse_hs_gb300 import hs
    w = WORKLOADS["llama8b_bf16"].scaled(batch=2, ctx_min=3000, ctx_max=5000, k_scored=9)
    c = _layers(w, 1)[0]
    dec = c.decoder(out_is_fp32=True)
    dec.build_summaries(c.kv)
    dec.step(c.kv, c.q)
    kept = dec.sel.clone()
    q2 = (c.q.float() * -0.5).to(c.q.dtype).contiguous()  # a different query, same blocks
    dec.step(c.kv, q2, reuse=dec)
    st, bits = hs.hs_get_device_error()
    assert st == hs.HS_OK, bits
    assert bool((dec.sel == kept).all())
    sel, cnt = dec.sel.cpu().numpy(), dec.sel_count.cpu().numpy()
    q2n = q2.float().cpu().numpy().astype(np.float64)
    g, B = w.group, w.block_size
    for b in range(w.batch):
        for kvh in range(w.num_kv_heads):
            K, V = c.logical(b, kvh, "k"), c.logical(b, kvh, "v")
            ref, _ = O.sparse_attention(q2n[b, kvh * g:(kvh + 1) * g], K, V, sel[b, kvh, :cnt[b, kvh]].tolist(), B,
                                        1.0 / math.sqrt(w.head_dim))
            assert np.abs(dec.out[b, kvh * g:(kvh + 1) * g].cpu().numpy() - ref).max() <= TOL
