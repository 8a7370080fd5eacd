"""Workload recipes and seeded generators.

Five workloads, each named by what it is:

* ``tiny_f32``      - 1 request, 8 q / 2 kv heads, head_dim 64, 2048 tokens,
                      16-token blocks, fp32; q, K, V ~ N(0, 1); 16 blocks kept
                      (sink 1 block + window 2 blocks + 13 scored).
* ``llama8b_bf16``  - 8 requests, 32 q / 4 kv heads, head_dim 128, 32768
                      tokens, 64-token blocks, bf16; 2048-token budget
                      including the first 4 and the last 256 tokens.
* ``ragged_bf16``   - 64 requests with lengths uniform in [4096, 131072],
                      16-token blocks scattered over a global page pool,
                      256 scored blocks plus sink 4 + window 256 tokens.
* ``offload_bf16``  - 256 requests x 32768 tokens, 64-token blocks, a hot
                      buffer of 64 pages (4096 tokens) per (request, kv head)
                      in device memory, the full cache in pinned host memory,
                      64 decode steps with a drifting query.
* ``fp8_g32``       - 32 requests x 131072 tokens, 64-token blocks, K/V in
                      e4m3 with one fp32 scale per 32 channels per token
                      (quantised by the consumer from the bf16 values drawn
                      here), 4096-token budget including sink 4 + window 256.

Distributions ("heavy" workloads): K, V ~ N(0, 1); per (request, kv head) 2%
of the token positions are heavy hitters whose K row is multiplied by 4; each
query head takes 8 of its kv head's heavy hitters at random, u = normalised sum
of their K rows, and q = (0.6 u + 0.8 n) * sqrt(head_dim) with n a random unit
vector orthogonal to u, so cos(q, u) = 0.6.

Physical layout: per-(request, kv head) pages of ``block_size`` tokens x
``head_dim`` channels, ``pages[num_pages][block_size][head_dim]``;
``page_table[b][kvh][j]`` is the physical page of logical block j, -1 past the
end.  Resident workloads scatter the pages by a seeded random permutation of the
pool; the offload workload keeps the pool in logical order (the pool is the
host copy, ``pool[b][kvh][j]``).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

# Step size of the query random walk of the offload workload, in units of the
# query norm per sqrt(head_dim).  Found by ``oracle/calibrate_drift.py``
# (bisection on the oracle's own selection) so that on average about 85% of the
# selected blocks repeat from one decode step to the next.
DRIFT_SIGMA = 1.068


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str  # "f32" | "bf16" | "fp8"
    ctx_min: int
    ctx_max: int
    sink_tokens: int
    window_tokens: int
    k_scored: int
    heavy: bool
    hot_slots: int = 0  # > 0: pages per (request, kv head) in the device hot buffer
    decode_steps: int = 1
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks(self) -> int:
        return -(-self.ctx_max // self.block_size)

    @property
    def capacity(self) -> int:
        """Upper bound on the number of selected blocks of one (request, kv head)."""
        b = self.block_size
        forced = -(-self.sink_tokens // b) + (-(-self.window_tokens // b) + 1)
        return min(self.max_blocks, forced + self.k_scored)

    @property
    def offload(self) -> bool:
        return self.hot_slots > 0

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 8, 2, 64, 16, "f32", 2048, 2048,
                         sink_tokens=16, window_tokens=32, k_scored=13,
                         heavy=False, seed=1000),
    "llama8b_bf16": Workload("llama8b_bf16", 8, 32, 4, 128, 64, "bf16", 32768, 32768,
                             sink_tokens=4, window_tokens=256, k_scored=27,
                             heavy=True, seed=1001),
    "ragged_bf16": Workload("ragged_bf16", 64, 32, 4, 128, 16, "bf16", 4096, 131072,
                            sink_tokens=4, window_tokens=256, k_scored=256,
                            heavy=True, seed=1002),
    "offload_bf16": Workload("offload_bf16", 256, 32, 4, 128, 64, "bf16", 32768, 32768,
                             sink_tokens=4, window_tokens=256, k_scored=27,
                             heavy=True, hot_slots=64, decode_steps=64, seed=1003),
    "fp8_g32": Workload("fp8_g32", 32, 32, 4, 128, 64, "fp8", 131072, 131072,
                        sink_tokens=4, window_tokens=256, k_scored=59,
                        heavy=True, seed=1004),
}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _store_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.kv_dtype == "f32" else torch.bfloat16


def make_layout(w: Workload, device="cpu", seed_offset: int = 0) -> dict:
    """Sequence lengths and the page table (shared by every layer of a workload)."""
    dev = torch.device(device)
    g = generator(w.seed * 7 + 11 + seed_offset, dev)
    if w.ctx_min == w.ctx_max:
        lens = torch.full((w.batch,), w.ctx_max, dtype=torch.int64, device=dev)
    else:
        lens = torch.randint(w.ctx_min, w.ctx_max + 1, (w.batch,), generator=g, device=dev)
    nb = (lens + w.block_size - 1) // w.block_size  # blocks per request
    mb = w.max_blocks
    j = torch.arange(mb, device=dev)
    valid = (j[None, None, :] < nb[:, None, None]).expand(w.batch, w.num_kv_heads, mb)
    num_pages = int(valid.sum().item())
    if w.offload:
        # the host pool is laid out in logical order: pool[b][kvh][j]
        base = torch.arange(w.batch * w.num_kv_heads, device=dev)[:, None] * mb
        ids = (base + j[None, :]).reshape(w.batch, w.num_kv_heads, mb)
        table = torch.where(valid, ids, torch.full_like(ids, -1))
        num_pages = w.batch * w.num_kv_heads * mb
    else:
        perm = torch.randperm(num_pages, generator=g, device=dev)
        table = torch.full((w.batch, w.num_kv_heads, mb), -1, dtype=torch.int64, device=dev)
        table[valid] = perm
    return {
        "seq_lens": lens.to(torch.int32),
        "page_table": table.to(torch.int32).contiguous(),
        "num_pages": num_pages,
        "max_blocks": mb,
    }


def _heavy_positions(w: Workload, lens: torch.Tensor, g: torch.Generator, dev) -> list:
    """Per (request, kv head): sorted heavy-hitter token positions (2% of the context)."""
    out = []
    lens_l = lens.tolist()
    for b in range(w.batch):
        L = int(lens_l[b])
        n = max(1, round(0.02 * L))
        for _ in range(w.num_kv_heads):
            pos = torch.randperm(L, generator=g, device=dev)[:n]
            out.append(torch.sort(pos).values)
    return out


def make_layer(w: Workload, layout: dict, device="cpu", layer: int = 0) -> dict:
    """K/V pages and the decode query of one layer.

    Returns ``k_pages``/``v_pages`` ``[num_pages][block][head_dim]`` (fp32 for the
    fp32 workload, bf16 otherwise - for the fp8 workload these are the values to
    be quantised), ``q`` ``[batch][num_q_heads][head_dim]`` (fp32 / bf16) and
    ``heavy``: the list of heavy-hitter positions per (request, kv head).
    """
    dev = torch.device(device)
    g = generator(w.seed * 1_000_003 + 7919 * layer + 1, dev)
    P, B, D = layout["num_pages"], w.block_size, w.head_dim
    dt = _store_dtype(w)
    k = torch.randn((P, B, D), generator=g, device=dev, dtype=dt)
    v = torch.randn((P, B, D), generator=g, device=dev, dtype=dt)
    lens = layout["seq_lens"].to(torch.int64)
    table = layout["page_table"].to(torch.int64)
    hkv, hq, grp = w.num_kv_heads, w.num_q_heads, w.group
    if not w.heavy:
        q = torch.randn((w.batch, hq, D), generator=g, device=dev, dtype=torch.float32)
        return {"k_pages": k, "v_pages": v, "q": q.to(dt), "heavy": None}

    heavy = _heavy_positions(w, lens, g, dev)
    # scale the heavy-hitter K rows by 4 (exact in bf16)
    for idx, pos in enumerate(heavy):
        b, kvh = divmod(idx, hkv)
        pages = table[b, kvh, pos // B]
        rows = pos % B
        k[pages, rows] = k[pages, rows] * 4
    q = torch.empty((w.batch, hq, D), device=dev, dtype=torch.float32)
    for b in range(w.batch):
        for h in range(hq):
            kvh = h // grp
            pos = heavy[b * hkv + kvh]
            pick = pos[torch.randperm(pos.numel(), generator=g, device=dev)[:8]]
            rows = k[table[b, kvh, pick // B], pick % B].to(torch.float32)
            u = rows.sum(0)
            u = u / u.norm()
            n = torch.randn((D,), generator=g, device=dev, dtype=torch.float32)
            n = n - (n @ u) * u
            n = n / n.norm()
            q[b, h] = (0.6 * u + 0.8 * n) * math.sqrt(D)
    return {"k_pages": k, "v_pages": v, "q": q.to(dt), "heavy": heavy}


def make_inputs(w: Workload, device="cpu", layer: int = 0) -> dict:
    layout = make_layout(w, device)
    out = dict(layout)
    out.update(make_layer(w, layout, device, layer))
    return out


def drift_queries(w: Workload, q0: torch.Tensor, steps: int, sigma: float = DRIFT_SIGMA,
                  seed_offset: int = 0) -> torch.Tensor:
    """Seeded random walk of the decode query, one entry per decode step.

    q_{t+1} = (q_t + sigma * |q_0| * e_t / sqrt(D)) rescaled to norm |q_0|, with
    e_t ~ N(0, I) per head.  Returns ``[steps][batch][num_q_heads][head_dim]`` in
    the dtype of ``q0``; entry 0 is ``q0``.
    """
    dev = q0.device
    g = generator(w.seed * 31 + 5 + seed_offset, dev)
    q = q0.to(torch.float32)
    n0 = q.norm(dim=-1, keepdim=True)
    D = q.shape[-1]
    out = torch.empty((steps,) + tuple(q.shape), dtype=q0.dtype, device=dev)
    out[0] = q0
    for t in range(1, steps):
        e = torch.randn(q.shape, generator=g, device=dev, dtype=torch.float32)
        q = q + sigma * n0 * e / math.sqrt(D)
        q = q / q.norm(dim=-1, keepdim=True) * n0
        out[t] = q.to(q0.dtype)
    return out
