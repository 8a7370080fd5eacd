"""Pins of the CPU oracle against facts that do not come from the oracle itself:
library routines (torch float8/bf16 conversion, scaled_dot_product_attention),
brute force on tiny inputs, closed forms, invariants and hand-worked fixtures
under tests/golden.  CPU only."""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(20240611)


# ---------------------------------------------------------------- e4m3 / bf16

def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))
    assert np.nanmax(got) == 448.0


def test_e4m3_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(vals), codes)


def _encode_bruteforce(x):
    mags = [O.e4m3_decode(np.array([c]))[0] for c in range(127)]
    out = []
    for v in np.asarray(x, dtype=np.float32).tolist():
        a = abs(v)
        if a >= 448.0:
            c = 126
        else:
            best = None
            for c_ in range(127):
                d = abs(mags[c_] - a)
                if best is None or d < best[0] or (d == best[0] and c_ % 2 == 0):
                    best = (d, c_)
            c = best[1]
        if math.copysign(1.0, v) < 0:
            c |= 0x80
        out.append(c)
    return np.array(out, dtype=np.uint8)


def test_e4m3_encode_bruteforce_and_midpoints():
    mags = O.e4m3_decode(np.arange(127))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)  # exact ties
    rand = (RNG.standard_normal(400) * np.exp2(RNG.integers(-12, 10, 400))).astype(np.float32)
    big = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, -1e30, -470.0], dtype=np.float32)
    x = np.concatenate([mids, -mids, rand, big, np.array([0.0, -0.0, 1e-30], np.float32)])
    assert np.array_equal(O.e4m3_encode(x), _encode_bruteforce(x))


def test_e4m3_encode_matches_torch_in_range():
    mags = O.e4m3_decode(np.arange(127))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    rand = np.clip(RNG.standard_normal(5000).astype(np.float32) * 60, -448, 448)
    x = np.concatenate([mids, -mids, rand])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_quantize_group32_properties():
    x = RNG.standard_normal((7, 128)).astype(np.float32) * 3
    x[2, 32:64] = 0.0  # an all-zero group
    codes, scales = O.quantize_e4m3_g32(x)
    assert codes.shape == (7, 128) and scales.shape == (7, 4) and scales.dtype == np.float32
    xg = x.reshape(7, 4, 32)
    amax = np.abs(xg).max(-1)
    want = np.where(amax > 0, (amax / np.float32(448)).astype(np.float32), np.float32(1))
    assert np.array_equal(scales, want)
    vals = O.e4m3_decode(codes).reshape(7, 4, 32)
    for t in range(7):
        for gi in range(4):
            if amax[t, gi] > 0:
                assert np.abs(vals[t, gi]).max() == 448.0
            else:
                assert np.all(vals[t, gi] == 0) and scales[t, gi] == 1.0
    deq = O.dequantize_e4m3_g32(codes, scales).reshape(7, 4, 32)
    y = xg / scales[..., None]
    bound = scales[..., None] * np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) + np.abs(xg) * 2.0 ** -22
    assert np.all(np.abs(deq - xg) <= bound)


def test_bf16_rounding_against_torch_and_bracketing():
    x = (RNG.standard_normal(20000) * np.exp2(RNG.integers(-30, 30, 20000))).astype(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-45, -1e-45], np.float32)])
    rn = O.bf16_round_nearest(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(rn, ref)
    rd, ru = O.bf16_round_down(x), O.bf16_round_up(x)
    with np.errstate(over="ignore"):
        assert np.all(rd <= x) and np.all(ru >= x)
    for r in (rd, ru):
        fin = np.isfinite(r)
        assert np.array_equal(torch.from_numpy(r[fin]).to(torch.bfloat16).to(torch.float32).numpy(), r[fin])
    exact = rn == x
    assert np.array_equal(rd[exact], x[exact]) and np.array_equal(ru[exact], x[exact])
    inexact = ~exact & np.isfinite(ru) & np.isfinite(rd) & (x != 0)
    brd = rd[inexact].view(np.uint32).astype(np.int64)
    bru = ru[inexact].view(np.uint32).astype(np.int64)
    pos = x[inexact] > 0
    # adjacent bf16 values: magnitudes differ by one unit in the last place
    assert np.all(np.where(pos, bru - brd, brd - bru) == 0x10000)
    assert np.all((rn[inexact] == rd[inexact]) | (rn[inexact] == ru[inexact]))


# ---------------------------------------------------------------- paging

def test_gather_rows_hand_case():
    pages = np.array([[0, 1], [10, 11], [20, 21]], dtype=np.float32)[..., None]  # [3][2][1]
    rows = O.gather_rows(pages, np.array([2, 0, 1, -1]), seq_len=5, block_size=2)
    assert rows[:, 0].tolist() == [20, 21, 0, 1, 10]


# ---------------------------------------------------------------- summaries / bound

def test_block_summaries_bruteforce():
    L, B, D = 37, 8, 5
    K = RNG.standard_normal((L, D))
    smin, smax = O.block_summaries(K, B)
    assert smin.shape == (5, D)
    for j in range(5):
        for d in range(D):
            vals = [K[t, d] for t in range(L) if t // B == j]
            assert smin[j, d] == min(vals) and smax[j, d] == max(vals)


@pytest.mark.parametrize("kv", ["f32", "bf16", "fp8"])
def test_bound_is_an_upper_bound(kv):
    L, B, D, g = 300, 16, 64, 4
    K = RNG.standard_normal((L, D)).astype(np.float32) * 2
    if kv == "bf16":
        K = O.bf16_round_nearest(K)
    if kv == "fp8":
        codes, sc = O.quantize_e4m3_g32(K)
        K = O.dequantize_e4m3_g32(codes, sc)
    K = K.astype(np.float64)
    q = RNG.standard_normal((g, D))  # mixed signs
    smin, smax = O.stored_summaries(*O.block_summaries(K, B), kv)
    U, score = O.bound_scores(q, smin, smax)
    for j in range(O.num_blocks(L, B)):
        dots = q @ K[j * B: min((j + 1) * B, L)].T  # [g][tokens]
        true = dots.max(axis=1)
        assert np.all(U[:, j] >= true - 1e-9 * np.abs(true).max())
        assert score[j] >= true.max() - 1e-9 * abs(true.max())
        # the bound is attained when only one token decides each channel: it can
        # never be below the best single-token sum of per-channel maxima
        assert U[:, j].min() >= -np.abs(q).sum(1).max() * np.abs(K).max() - 1e-9


def test_bound_equality_cases():
    D, g = 32, 3
    q = RNG.standard_normal((g, D))
    # block size 1: U is q.k exactly and the group score is the max over heads
    K = RNG.standard_normal((9, D))
    smin, smax = O.block_summaries(K, 1)
    U, score = O.bound_scores(q, smin, smax)
    assert np.allclose(U, q @ K.T, rtol=0, atol=1e-12)
    assert np.allclose(score, (q @ K.T).max(axis=0), rtol=0, atol=1e-12)
    # last block holding a single token, and a block of identical rows
    K2 = RNG.standard_normal((17, D))
    K2[8:16] = K2[8]
    smin, smax = O.block_summaries(K2, 8)
    U, _ = O.bound_scores(q, smin, smax)
    assert np.allclose(U[:, 2], q @ K2[16], atol=1e-12)
    assert np.allclose(U[:, 1], q @ K2[8], atol=1e-12)
    # a two-token block: the bound is the per-channel max, strictly above both
    # tokens when the channels disagree
    K3 = np.array([[1.0, -1.0], [-1.0, 1.0]])
    U3, _ = O.bound_scores(np.array([[1.0, 1.0]]), *O.block_summaries(K3, 2))
    assert U3[0, 0] == 2.0


# ---------------------------------------------------------------- forced set / selection

def test_forced_blocks_golden():
    with open(os.path.join(GOLDEN, "forced_blocks.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert O.forced_blocks(c["L"], c["B"], c["sink"], c["window"]) == c["forced"], c


def _bruteforce_topk(scores, rest, k):
    found = []
    for S in itertools.combinations(rest, k):
        Sset = set(S)
        ok = all(scores[a] > scores[b] or (scores[a] == scores[b] and a < b)
                 for a in Sset for b in rest if b not in Sset)
        if ok:
            found.append(Sset)
    assert len(found) == 1
    return found[0]


def test_selection_matches_enumeration():
    for trial in range(60):
        N = int(RNG.integers(1, 13))
        B = 4
        L = N * B - int(RNG.integers(0, B))
        scores = RNG.integers(-3, 4, N).astype(np.float64)  # many ties
        sink = int(RNG.integers(0, 2 * B))
        window = int(RNG.integers(0, 2 * B))
        F = O.forced_blocks(L, B, sink, window)
        for k in range(0, N + 1):
            sel = O.select_blocks(scores, F, k)
            if len(F) + k >= N:
                assert sel == list(range(N))
                continue
            rest = [j for j in range(N) if j not in F]
            S = _bruteforce_topk(scores, rest, k)
            assert sel == sorted(set(F) | S)
            assert set(F) <= set(sel) and len(sel) == len(F) + k


def test_selection_zero_query_picks_lowest_indices():
    L, B, D = 640, 64, 16
    K = RNG.standard_normal((L, D))
    q = np.zeros((2, D))
    smin, smax = O.block_summaries(K, B)
    _, score = O.bound_scores(q, smin, smax)
    assert np.all(score == 0)
    F = O.forced_blocks(L, B, 4, 64)  # {0, 9}
    assert O.select_blocks(score, F, 3) == [0, 1, 2, 3, 9]


def test_selection_nan_scores_rank_last():
    scores = np.array([np.nan, 1.0, np.nan, -5.0, 2.0])
    assert O.select_blocks(scores, [], 3) == [1, 3, 4]
    assert O.select_blocks(scores, [], 4) == [0, 1, 3, 4]


# ---------------------------------------------------------------- attention

def _sdpa(q, K, V, scale):
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, :, None, :]  # [1][g][1][D]
    g = qt.shape[1]
    kt = torch.from_numpy(np.asarray(K, np.float64))[None, None].expand(1, g, -1, -1)
    vt = torch.from_numpy(np.asarray(V, np.float64))[None, None].expand(1, g, -1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return out[0, :, 0].numpy()


@pytest.mark.parametrize("L,B", [(128, 16), (130, 16), (1, 4), (77, 64)])
def test_attention_over_all_blocks_is_dense_sdpa(L, B):
    D, g = 32, 4
    q = RNG.standard_normal((g, D)) * 2
    K = RNG.standard_normal((L, D))
    V = RNG.standard_normal((L, D))
    scale = 1 / math.sqrt(D)
    out, lse = O.sparse_attention(q, K, V, list(range(O.num_blocks(L, B))), B, scale)
    assert np.allclose(out, _sdpa(q, K, V, scale), rtol=0, atol=1e-12)
    logits = torch.from_numpy(q @ K.T * scale)
    assert np.allclose(lse, torch.logsumexp(logits, dim=1).numpy(), atol=1e-12)


def test_attention_subset_is_sdpa_on_gathered_rows():
    L, B, D, g = 100, 16, 24, 3
    q = RNG.standard_normal((g, D))
    K = RNG.standard_normal((L, D))
    V = RNG.standard_normal((L, D))
    blocks = [0, 2, 6]  # block 6 holds the 4 tail tokens 96..99
    toks = [t for t in range(L) if t // B in blocks]
    assert len(toks) == 16 + 16 + 4
    out, lse = O.sparse_attention(q, K, V, blocks, B, 0.3)
    assert np.allclose(out, _sdpa(q, K[toks], V[toks], 0.3), atol=1e-12)
    w = np.exp(q @ K[toks].T * 0.3 - lse[:, None])
    assert np.allclose(w.sum(1), 1.0, atol=1e-12)


def test_attention_single_token_and_empty():
    D = 8
    q = RNG.standard_normal((2, D))
    K = RNG.standard_normal((5, D))
    V = RNG.standard_normal((5, D))
    out, lse = O.sparse_attention(q, K, V, [3], 1, 0.5)
    assert np.allclose(out, np.stack([V[3], V[3]]), atol=1e-15)
    assert np.allclose(lse, q @ K[3] * 0.5, atol=1e-12)
    out, lse = O.sparse_attention(q, K[:0], V[:0], [], 4, 0.5)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_lse_merge_equals_one_pass():
    L, D, g = 90, 16, 2
    q = RNG.standard_normal((g, D))
    K = RNG.standard_normal((L, D)) * 3
    V = RNG.standard_normal((L, D))
    full, lse_full = O.sparse_attention(q, K, V, list(range(L)), 1, 0.7)
    cuts = sorted(RNG.choice(np.arange(1, L), 4, replace=False).tolist())
    parts = np.split(np.arange(L), cuts)
    outs, lses = zip(*[O.sparse_attention(q, K, V, p.tolist(), 1, 0.7) for p in parts])
    out, lse = O.lse_merge(outs, lses)
    assert np.allclose(out, full, atol=1e-12) and np.allclose(lse, lse_full, atol=1e-12)
    # an empty part does not change the result
    out2, lse2 = O.lse_merge(list(outs) + [np.zeros((g, D))], list(lses) + [np.full(g, -np.inf)])
    assert np.allclose(out2, full, atol=1e-12) and np.allclose(lse2, lse_full, atol=1e-12)


def test_decode_pair_with_every_block_is_dense_attention():
    L, B, D, g = 200, 16, 32, 4
    q = RNG.standard_normal((g, D))
    K = RNG.standard_normal((L, D))
    V = RNG.standard_normal((L, D))
    r = O.decode_pair(q, K, V, B, "f32", 4, 16, k_scored=100, scale=0.2)
    assert r["sel"] == list(range(13))
    assert np.allclose(r["out"], _sdpa(q, K, V, 0.2), atol=1e-12)


# ---------------------------------------------------------------- hot buffer

def test_hot_buffer_golden_trace():
    with open(os.path.join(GOLDEN, "hot_buffer_trace.json")) as f:
        tr = json.load(f)
    hb = O.HotBuffer(tr["num_blocks"], tr["slots"], base=tr["base"])
    for st in tr["steps"]:
        copies, stats = hb.step(st["sel"], st["step"])
        assert [list(c) for c in copies] == st["copies"]
        assert (stats["hits"], stats["misses"], stats["evictions"]) == (st["hits"], st["misses"], st["evictions"])
        assert hb.slot_owner == st["slot_owner"]
        assert hb.last_used == st["last_used"]
        assert hb.page_table == st["page_table"]


def test_hot_buffer_invariants_random_walk():
    N, S = 40, 8
    hb = O.HotBuffer(N, S, base=100)
    for step in range(200):
        k = int(RNG.integers(0, S + 1))
        sel = sorted(RNG.choice(N, k, replace=False).tolist())
        before = {j for j in range(N) if hb.page_table[j] >= 0}
        free_before = sum(1 for o in hb.slot_owner if o < 0)
        copies, st = hb.step(sel, step)
        resident = {j for j in range(N) if hb.page_table[j] >= 0}
        assert set(sel) <= resident
        assert st["misses"] == len(set(sel) - before) == len(copies)
        assert st["hits"] + st["misses"] == len(sel)
        assert st["evictions"] == max(0, st["misses"] - free_before)
        # page table and slot owners are inverse maps
        for s, o in enumerate(hb.slot_owner):
            if o >= 0:
                assert hb.page_table[o] == 100 + s
        assert len(resident) == sum(1 for o in hb.slot_owner if o >= 0)
        for j in sel:
            assert hb.last_used[hb.page_table[j] - 100] == step


def test_hot_buffer_capacity_error():
    hb = O.HotBuffer(10, 2)
    with pytest.raises(O.CapacityError):
        hb.step([1, 2, 3], 0)


def test_score_smoothing_matches_its_unrolled_form():
    """s~_t = 0.7 s_t + 0.3 s~_{t-1} from an empty history unrolls to
    sum_k 0.7 * 0.3^k s_{t-k} plus 0.3^t s_0 (weights summing to one); blocks
    whose history is NaN (new blocks) take their raw score."""
    w, T, N = 0.3, 6, 9
    seq = RNG.normal(size=(T, N))
    h = np.full(N, np.nan)
    for t in range(T):
        h = O.smooth_scores(seq[t], h, w)
        closed = sum((1 - w) * w ** k * seq[t - k] for k in range(t)) + w ** t * seq[0]
        assert np.allclose(h, closed, rtol=1e-12, atol=1e-12)
    # a constant score is a fixed point; weight 0 is the identity
    c = np.full(N, 2.5)
    assert np.array_equal(O.smooth_scores(c, c, w), c)
    assert np.array_equal(O.smooth_scores(seq[1], seq[0], 0.0), seq[1])
    # mixed history: NaN entries take the raw score, the others blend
    hist = seq[0].copy()
    hist[::2] = np.nan
    got = O.smooth_scores(seq[1], hist, w)
    assert np.array_equal(got[::2], seq[1][::2])
    assert np.allclose(got[1::2], 0.7 * seq[1][1::2] + 0.3 * seq[0][1::2], rtol=1e-12)
