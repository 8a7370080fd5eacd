"""The attention call for callers that cannot allocate device memory.

Hosts that give an operator only its input and output buffers (and keep the
device allocator to themselves) cannot pass the split-K workspace, so the
library offers hs_sparse_paged_decode_attn_noalloc, which keeps that workspace
in a fixed array of its own.  This file checks, through the C ABI, that two
calls in a row give the same attention as the regular call with a
caller-provided workspace, and that a problem too large for the fixed array is
refused.  It is collected last on purpose and needs no state from other tests.
GPU only.
"""

import numpy as np
import pytest
import torch

from synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-3  # the bf16 attention tolerance used by the parity tests
TOL_LSE = 1e-4


def _case():
    from _parity import Case
    w = WORKLOADS["llama8b_bf16"].scaled(batch=3, ctx_min=4133, ctx_max=4133, k_scored=20)
    return Case(w, make_inputs(w))


def test_noalloc_matches_the_workspace_call_twice_in_a_row():
    from query_aware_sparse_hs_gb300 import hs
    c = _case()
    dec = c.decoder(out_is_fp32=True)
    dec.build_summaries(c.kv)
    queries = [c.q, (c.q.float().flip(-1) * 0.7).to(torch.bfloat16).contiguous()]
    refs = []
    for q in queries:  # the regular call, with a caller-provided workspace
        dec.select(c.kv, q)
        dec.attend(c.kv, q)
        refs.append((dec.sel.clone(), dec.sel_count.clone(), dec.out.clone(), dec.lse.clone()))
    for q, (sel, cnt, ref_out, ref_lse) in zip(queries, refs):  # two no-allocation calls in a row
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        hs.hs_sparse_paged_decode_attn_noalloc(dec.shape, c.kv, q, sel, cnt, dec.capacity,
                                               dec.attn_params, out, lse)
        st, bits = hs.hs_get_device_error()
        assert st == hs.HS_OK, bits
        assert np.isfinite(out.cpu().numpy()).all()
        assert (out - ref_out).abs().max().item() <= TOL_OUT
        assert (lse - ref_lse).abs().max().item() <= TOL_LSE


def test_noalloc_refuses_work_larger_than_its_scratch():
    from query_aware_sparse_hs_gb300 import hs
    c = _case()
    dec = c.decoder(out_is_fp32=True)
    huge = hs.attn_params(0.088, True, blocks_per_split=1)
    need = hs.hs_workspace_bytes(dec.shape, c.w.batch, 100_000, huge)
    assert need > hs.HS_NOALLOC_SCRATCH_BYTES
    with pytest.raises(hs.HSError) as e:
        hs.hs_sparse_paged_decode_attn_noalloc(dec.shape, c.kv, c.q, dec.sel, dec.sel_count, 100_000, huge,
                                               dec.out, dec.lse)
    assert e.value.status == hs.HS_ERR_SCRATCH_LIMIT
    assert hs.hs_get_device_error() == (hs.HS_OK, 0)
