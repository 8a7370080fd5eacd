"""Plain, slow CPU oracle of query-aware block-sparse paged decode attention.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the library.  It shares no
code, table or constant generator with the CUDA path.

Every function is the plain definition of one step, written out in float64 with
numpy (matmul, exp, log, min/max are the only library primitives used).  No
tiling, no online softmax, no split reduction: the CUDA path's blocking is not
mirrored here.

Sources, cited by page title and section:

* [KVS] "KV 稀疏化" (KV-cache sparsity wiki page):
  §2 "Attention sink + 滑动窗口 (StreamingLLM)" - keep the first tokens and the
  most recent window; §5 "Quest" - per-block compact summary (min/max), coarse
  filter of the query against the summaries, top-k blocks, full attention on the
  chosen blocks only; §7 "HiSparse" - hot device buffer, host inactive KV,
  swap-in kernel that detects misses, updates the page table and brings KV back;
  offload target driven by the sparse attention's current access set.
* [SPD] "SparDA：把KV選擇提前一層，長上下文推理顯存帶寬雙優化":
  §1.1 KV bytes per token of an 8B GQA model; §4.2 selector = attention sink +
  local window + remote top-k; §4.3 sparse index kept over PagedAttention blocks;
  §6.1 selection scores smoothed over decode steps, 70% this step's value and
  30% the previous step's smoothed value.
* [FLL] "分块稀疏注意力与KV Cache量化：长文本推理显存优化实践":
  §2.2 tiled attention whose partial softmax statistics (running max and
  normaliser) are carried across tiles; §2.4 grouped KV quantisation along the
  channel dimension with a per-group scale; §3.2 ``kv_quant_group_size=32``.

Readings where the pages are silent (each is also listed in the design notes):

* Bound: the pages only say "coarse filter of the query against the summary";
  the oracle uses U = sum_d max(q_d * max_d, q_d * min_d), the smallest value
  that is >= q.k for every k inside the per-channel box [min, max].
* The summary "mean" named in [KVS] §5 cannot bound q.k and is not used.
* GQA: one selection per kv head, scored by the max of U over its query heads.
* Forced set: every block overlapping the first ``sink_tokens`` tokens or the
  last ``window_tokens`` tokens.  ``k_scored`` more blocks are chosen among the
  rest by (score descending, block index ascending); NaN scores rank last.
* Quantisation: symmetric e4m3 (OCP FP8 E4M3), scale = amax/448 in fp32 per 32
  channels of one token (1 when amax is 0), code = RNE(x/scale) saturated to
  +-448; the page's zero point is not used.
* Summaries are stored in the K storage precision: fp32 for fp32 K, bf16 for bf16
  K (exact), and for e4m3 K the fp32 dequantised min/max rounded outward to bf16
  (min down, max up) so the bound still holds.
* Hot buffer (per (request, kv head), S slots): hits stamp ``last_used = step``;
  misses are handled in ascending block order; the victim is the lowest free
  slot, else the slot whose block is not in the current selection with the
  smallest ``last_used`` (ties -> lowest slot); the evicted block's page-table
  entry becomes -1; no write-back (the host pool keeps every page).
* Empty selection (zero-length request): output 0, lse = -inf.
* Score smoothing ([SPD] §6.1): applied to the per-block selection score
  (the group bound) of each (request, kv head): s~_t = (1 - w) s_t + w s~_{t-1}
  with w = 0.3, and s~_t = s_t for a block without history (first step, or a
  block new since the last step).

Parity pins (``tests/test_oracle.py``): e4m3 decode against torch's
float8_e4m3fn; e4m3 encode by brute force over all codes and against torch;
bf16 rounding against torch and by bracketing; summaries by brute-force loops;
bound by the inequality over every token and the equality cases; selection by
enumeration of every k-subset; attention against
``torch.nn.functional.scaled_dot_product_attention`` in float64 and by the
weights-sum-to-one and single-token cases; LSE merge against the one-pass
softmax; hot buffer against a hand-worked trace (``tests/golden``) and the
table invariants; score smoothing against its unrolled closed form.  No
function here is unpinned.
"""

from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
QUANT_GROUP = 32


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Value of OCP FP8 E4M3 codes (exponent bias 7, no infinities, S.1111.111 = NaN).

    [FLL] §2.4 grouped quantisation; the element format is the OCP E4M3 one.
    """
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


_E4M3_MAGS = e4m3_decode(np.arange(127))  # codes 0..126: 0 .. 448, increasing


def e4m3_encode(x) -> np.ndarray:
    """Round float32 values to E4M3 codes: nearest, ties to even mantissa,
    saturating at +-448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    idx = np.searchsorted(_E4M3_MAGS, a, side="left")
    hi = np.clip(idx, 0, 126)
    lo = np.clip(idx - 1, 0, 126)
    d_hi = _E4M3_MAGS[hi] - a
    d_lo = a - _E4M3_MAGS[lo]
    pick = np.where(d_hi < d_lo, hi, np.where(d_lo < d_hi, lo, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= E4M3_MAX, 126, pick)
    code = pick.astype(np.int64) | (np.signbit(x).astype(np.int64) << 7)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_e4m3_g32(x) -> tuple[np.ndarray, np.ndarray]:
    """Grouped symmetric quantisation of the last axis ([FLL] §2.4, §3.2: 32-channel groups).

    Per token and 32-channel group: scale = amax / 448 (fp32), or 1 when amax
    is 0; code = e4m3(x / scale) computed in fp32.  Returns (codes uint8 [..., D],
    scales float32 [..., D/32]).
    """
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    assert D % QUANT_GROUP == 0
    xg = x.reshape(x.shape[:-1] + (D // QUANT_GROUP, QUANT_GROUP))
    amax = np.max(np.abs(xg), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (xg / scale[..., None]).astype(np.float32)
    codes = e4m3_encode(y).reshape(x.shape)
    return codes, scale


def dequantize_e4m3_g32(codes, scales) -> np.ndarray:
    """fp32 value that a consumer reconstructs: e4m3 value times its group scale (fp32 product)."""
    codes = np.asarray(codes)
    D = codes.shape[-1]
    vals = e4m3_decode(codes).astype(np.float32)
    vg = vals.reshape(codes.shape[:-1] + (D // QUANT_GROUP, QUANT_GROUP))
    out = (vg * np.asarray(scales, dtype=np.float32)[..., None]).astype(np.float32)
    return out.reshape(codes.shape)


def _bits(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)


def _from_bits(b):
    return (np.asarray(b, dtype=np.uint64) & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def bf16_round_nearest(x) -> np.ndarray:
    """float32 -> nearest bf16 value (ties to even), returned as float32."""
    x = np.asarray(x, dtype=np.float32)
    b = _bits(x)
    r = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return np.where(np.isnan(x), x, _from_bits(r))


def bf16_round_down(x) -> np.ndarray:
    """float32 -> largest bf16 value <= x (toward -inf), returned as float32."""
    x = np.asarray(x, dtype=np.float32)
    b = _bits(x)
    hi = b & 0xFFFF0000
    low = b & 0xFFFF
    neg = (b >> 31) & 1
    r = np.where(low == 0, b, np.where(neg == 1, hi + 0x10000, hi))
    return np.where(np.isnan(x), x, _from_bits(r))


def bf16_round_up(x) -> np.ndarray:
    """float32 -> smallest bf16 value >= x (toward +inf), returned as float32."""
    x = np.asarray(x, dtype=np.float32)
    b = _bits(x)
    hi = b & 0xFFFF0000
    low = b & 0xFFFF
    neg = (b >> 31) & 1
    r = np.where(low == 0, b, np.where(neg == 1, hi, hi + 0x10000))
    return np.where(np.isnan(x), x, _from_bits(r))


# --------------------------------------------------------------------------
# paged KV: logical rows through the page table ([SPD] §4.3, [KVS] §7)
# --------------------------------------------------------------------------

def gather_rows(pages, table_row, seq_len: int, block_size: int) -> np.ndarray:
    """Logical rows 0..L-1 of one (request, kv head): token t lives in page
    ``table_row[t // B]`` at row ``t % B``."""
    t = np.arange(int(seq_len))
    page = np.asarray(table_row)[t // block_size]
    assert np.all(page >= 0), "a needed block is not resident"
    return np.asarray(pages)[page, t % block_size]


def kv_values(kv_dtype: str, rows, scales=None) -> np.ndarray:
    """float64 values the attention sees: fp32/bf16 stored values as they are,
    e4m3 codes times their fp32 group scale (fp32 product)."""
    if kv_dtype == "fp8":
        return dequantize_e4m3_g32(rows, scales).astype(np.float64)
    return np.asarray(rows, dtype=np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Quest steps ([KVS] §5)
# --------------------------------------------------------------------------

def num_blocks(seq_len: int, block_size: int) -> int:
    return -(-int(seq_len) // int(block_size))


def block_summaries(K, block_size: int) -> tuple[np.ndarray, np.ndarray]:
    """Per block j and channel d: min and max of K over the block's valid tokens
    t in [jB, min((j+1)B, L))."""
    K = np.asarray(K, dtype=np.float64)
    L, D = K.shape
    N = num_blocks(L, block_size)
    smin = np.empty((N, D))
    smax = np.empty((N, D))
    for j in range(N):
        rows = K[j * block_size: min((j + 1) * block_size, L)]
        smin[j] = rows.min(axis=0)
        smax[j] = rows.max(axis=0)
    return smin, smax


def stored_summaries(smin, smax, kv_dtype: str) -> tuple[np.ndarray, np.ndarray]:
    """Summaries in their storage precision (as float64): fp32 as is, bf16 as is
    (min/max of bf16 values are bf16 values), e4m3 -> bf16 rounded outward."""
    if kv_dtype == "fp8":
        lo = bf16_round_down(np.asarray(smin, dtype=np.float32)).astype(np.float64)
        hi = bf16_round_up(np.asarray(smax, dtype=np.float32)).astype(np.float64)
        return lo, hi
    return np.asarray(smin, dtype=np.float64), np.asarray(smax, dtype=np.float64)


def bound_scores(q_group, smin, smax) -> tuple[np.ndarray, np.ndarray]:
    """U[h][j] = sum_d max(q_hd * smax_jd, q_hd * smin_jd) for each query head h
    of the group, and the block score = max over the group's heads."""
    q = np.asarray(q_group, dtype=np.float64)
    smin = np.asarray(smin, dtype=np.float64)
    smax = np.asarray(smax, dtype=np.float64)
    U = np.maximum(q[:, None, :] * smax[None, :, :], q[:, None, :] * smin[None, :, :]).sum(axis=-1)
    return U, U.max(axis=0)


def forced_blocks(seq_len: int, block_size: int, sink_tokens: int, window_tokens: int) -> list:
    """Blocks overlapping the attention sink [0, sink) or the recent window
    [L - window, L) ([KVS] §2, [SPD] §4.2)."""
    L, B = int(seq_len), int(block_size)
    out = []
    for j in range(num_blocks(L, B)):
        lo, hi = j * B, min((j + 1) * B, L)
        in_sink = lo < sink_tokens
        in_window = window_tokens > 0 and hi > L - window_tokens
        if in_sink or in_window:
            out.append(j)
    return out


def smooth_scores(scores, history, weight: float) -> np.ndarray:
    """Exponential smoothing of selection scores across decode steps ([SPD]
    §6.1): where ``history`` (the previous step's smoothed scores) is a number,
    the result is (1 - weight) * score + weight * history; where it is NaN (no
    history yet) the score itself.  The result is the next step's history."""
    s = np.asarray(scores, dtype=np.float64)
    h = np.asarray(history, dtype=np.float64)
    return np.where(np.isnan(h), s, (1.0 - weight) * s + weight * h)


def select_blocks(scores, forced, k_scored: int) -> list:
    """Forced blocks plus the ``k_scored`` best of the rest, by score descending
    then block index ascending (NaN last); all blocks when that covers them.
    Returned in ascending block order."""
    scores = np.asarray(scores, dtype=np.float64)
    N = scores.shape[0]
    fset = set(int(j) for j in forced)
    if len(fset) + int(k_scored) >= N:
        return list(range(N))
    rest = [j for j in range(N) if j not in fset]

    def key(j):
        s = scores[j]
        return (1, 0.0, j) if math.isnan(s) else (0, -s, j)

    rest.sort(key=key)
    return sorted(fset | set(rest[: int(k_scored)]))


# --------------------------------------------------------------------------
# attention over the selected blocks ([KVS] §5 "full attention on the chosen
# blocks"; [FLL] §2.2 - tiling with carried max/normaliser is exact softmax)
# --------------------------------------------------------------------------

def selected_tokens(blocks, seq_len: int, block_size: int) -> np.ndarray:
    toks = [np.arange(j * block_size, min((j + 1) * block_size, seq_len)) for j in blocks]
    return np.concatenate(toks) if toks else np.zeros((0,), dtype=np.int64)


def sparse_attention(q_group, K, V, blocks, block_size: int, scale: float):
    """Softmax attention of each query head over the tokens of the chosen blocks.

    s_t = (q . k_t) * scale; out = sum_t softmax(s)_t v_t; lse = log sum_t e^{s_t}.
    Empty token set: out = 0, lse = -inf.
    """
    q = np.asarray(q_group, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    toks = selected_tokens(blocks, K.shape[0], block_size)
    if toks.size == 0:
        return np.zeros((q.shape[0], V.shape[1])), np.full((q.shape[0],), -np.inf)
    s = (q @ K[toks].T) * float(scale)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ V[toks]) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def lse_merge(outs, lses):
    """Combine softmax results over disjoint token sets: m = max lse_i,
    w_i = e^{lse_i - m}, out = sum w_i out_i / sum w_i, lse = m + log sum w_i."""
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = np.asarray(lses, dtype=np.float64)
    m = np.max(lses, axis=0)
    if np.all(np.isneginf(m)):
        return np.zeros_like(outs[0]), m
    w = np.exp(lses - m)
    tot = w.sum(axis=0)
    out = sum(wi[..., None] * oi for wi, oi in zip(w, outs)) / tot[..., None]
    return out, m + np.log(tot)


def decode_pair(q_group, K, V, block_size, kv_dtype, sink_tokens, window_tokens,
                k_scored, scale):
    """One decode step of one (request, kv head): summaries -> bound -> selection
    -> attention.  ``K``/``V`` are the logical float64 values the kernel sees."""
    L = K.shape[0]
    smin, smax = block_summaries(K, block_size)
    smin, smax = stored_summaries(smin, smax, kv_dtype)
    U, score = bound_scores(q_group, smin, smax)
    F = forced_blocks(L, block_size, sink_tokens, window_tokens)
    sel = select_blocks(score, F, k_scored)
    out, lse = sparse_attention(q_group, K, V, sel, block_size, scale)
    return {"smin": smin, "smax": smax, "U": U, "score": score, "forced": F,
            "sel": sel, "out": out, "lse": lse}


# --------------------------------------------------------------------------
# HiSparse hot buffer ([KVS] §7)
# --------------------------------------------------------------------------

class CapacityError(ValueError):
    pass


class HotBuffer:
    """Device hot buffer of one (request, kv head) stream with ``slots`` pages.

    ``page_table[j]`` is the global slot (``base + s``) holding block j or -1;
    ``slot_owner[s]`` the block in slot s or -1; ``last_used[s]`` the step at
    which slot s was last part of the selection (-1 = never).
    """

    def __init__(self, num_blocks: int, slots: int, base: int = 0):
        self.slots = int(slots)
        self.base = int(base)
        self.page_table = [-1] * int(num_blocks)
        self.slot_owner = [-1] * self.slots
        self.last_used = [-1] * self.slots

    def step(self, sel, step: int):
        """Make every block of ``sel`` resident.  Returns (copies, stats): the
        (block, slot) pairs to fetch from the host pool, in order, and
        hits/misses/evictions counts."""
        sel = sorted(int(j) for j in sel)
        if len(sel) > self.slots:
            raise CapacityError(f"{len(sel)} selected blocks > {self.slots} slots")
        selset = set(sel)
        hits = misses = evictions = 0
        copies = []
        for j in sel:
            g = self.page_table[j]
            if g >= 0:
                hits += 1
                self.last_used[g - self.base] = int(step)
                continue
            misses += 1
            free = [s for s in range(self.slots) if self.slot_owner[s] < 0]
            if free:
                s = free[0]
            else:
                cands = [s for s in range(self.slots) if self.slot_owner[s] not in selset]
                s = min(cands, key=lambda s: (self.last_used[s], s))
                self.page_table[self.slot_owner[s]] = -1
                evictions += 1
            self.slot_owner[s] = j
            self.page_table[j] = self.base + s
            self.last_used[s] = int(step)
            copies.append((j, s))
        return copies, {"hits": hits, "misses": misses, "evictions": evictions}
