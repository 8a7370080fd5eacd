"""Throughput of one decode step of query-aware block-sparse paged attention.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|offload_bf16|llama8b_bf16|ragged_bf16|fp8_g32]
                    [--batch B] [--layers L] [--cpu-seconds S]

A step = the whole per-step path of one layer over the batch: append of the
newest token (written into its page, e4m3-quantised for the e4m3 cache, its
block's summary widened), bound scoring + top-k selection, [swap-in of the
missing pages for the offload workload], gather-attention with split-K, LSE
merge.

With ``--workload all`` (the default) every target workload is measured and ONE
JSON line is printed (rank 0): its headline keys describe the largest workload,
the HiSparse-style offload step (256 requests x 32768 tokens, a hot buffer of 64
pages per (request, kv head), the rest of the cache in pinned host memory,
64 decode steps with a drifting query); ``workloads`` holds one record with the
same keys for each of the other three (the Llama-3-8B-like layer, the paged
ragged batch and the e4m3 group-32 cache).  ``--workload NAME`` measures one
workload and prints its record as the line.

Exactly ``--steps`` steps are timed after exactly ``--warmup`` untimed steps.
Resident workloads rotate distinct layer copies (together larger than L2) from
step to step and replay their steps from CUDA graphs; the offload workload
replays the decode steps of its drifting sequence (step 0, which refills the
empty hot buffer, is run untimed before each pass).  Each record adds a
``long_run`` figure over at least half a second of timed steps.

Multi-GPU: replicas (every rank runs the same per-GPU workload; no data-path
collective), launched by torchrun.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

# the CPU baseline times the oracle single-threaded; set before numpy loads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse decode-attn steps/s (batch×heads) and achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "head-steps/s"
HEADLINE = "offload_bf16"
SUB_WORKLOADS = ("llama8b_bf16", "ragged_bf16", "fp8_g32")
LONG_RUN_S = 0.5


# ----------------------------------------------------------------------------
# algorithmic bytes (what the method must move; no implementation overheads)
# ----------------------------------------------------------------------------

def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: float) -> float:
    """K and V of one token across the model (SparDA article §1.1 arithmetic)."""
    return 2 * num_layers * num_kv_heads * head_dim * elem_bytes


def token_bytes(w) -> float:
    """K+V bytes of one token of one kv head as stored (e4m3: codes + scales)."""
    if w.kv_dtype == "fp8":
        return 2 * (w.head_dim + (w.head_dim // 32) * 4)
    return 2 * w.head_dim * (4 if w.kv_dtype == "f32" else 2)


def summary_bytes_per_block(w) -> int:
    return 2 * w.head_dim * (4 if w.kv_dtype == "f32" else 2)


def attn_bytes(w, selected_tokens: int, pairs_blocks: int) -> int:
    """Algorithmic bytes of one attention launch: the selected K/V, q, out,
    the selection indices and the page-table entries they resolve."""
    qb = w.batch * w.num_q_heads * w.head_dim * (4 if w.kv_dtype == "f32" else 2)
    return int(selected_tokens * token_bytes(w) + 2 * qb + 8 * pairs_blocks)


def append_bytes_per_step(w) -> int:
    """The newest token of every (request, kv head): its K/V read in source
    precision, written as stored, and its block's summary row pair read and
    written."""
    src = 2 * w.head_dim * (4 if w.kv_dtype == "f32" else 2)
    return int(w.batch * w.num_kv_heads * (src + token_bytes(w) + 2 * summary_bytes_per_block(w)))


def select_bytes(w, total_blocks: int) -> int:
    """Summaries of every block read once, q, the selection written."""
    qb = w.batch * w.num_q_heads * w.head_dim * (4 if w.kv_dtype == "f32" else 2)
    return int(total_blocks * summary_bytes_per_block(w) + qb + 4 * w.batch * w.num_kv_heads * w.capacity)


# ----------------------------------------------------------------------------
# launches of one step, as the library dispatches them
# ----------------------------------------------------------------------------

def _sms() -> int:
    import torch
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def select_launches(w) -> int:
    """Launches of bound scoring + selection: one fused cluster launch when
    every tile of every (request, kv head) fits one wave (tensor-core scoring,
    at most 8 tiles of 128 blocks per request), two with the tensor-core scorer
    otherwise, one on the CUDA-core path."""
    if not (w.kv_dtype != "f32" and w.head_dim == 128):
        return 1
    tiles = -(-w.max_blocks // 128)
    return 1 if tiles <= 8 and w.batch * w.num_kv_heads * tiles <= _sms() else 2


def fused_step(w, dec) -> bool:
    """Whether the decoder's step runs scoring, selection and attention as one
    launch (the library answers for this geometry on this device)."""
    from query_aware_sparse_hs_gb300 import hs
    return bool(dec.fuse_step) and hs.hs_score_select_attend_fused(
        dec.shape, w.batch, dec.max_blocks, dec.capacity, dec.attn_params) == 1


def attn_splits(w, dec, params=None) -> int:
    from query_aware_sparse_hs_gb300 import hs
    per_split = w.batch * w.num_q_heads * (w.head_dim + 1) * 4
    return hs.hs_workspace_bytes(dec.shape, w.batch, dec.capacity, params or dec.attn_params) // per_split


def merge_launches(w, dec, params) -> int:
    """1 when the attention's split partials go through the separate merge
    kernel: not with one split, nor when the tensor-core kernel merges them in
    place (split counters, and every work item a CTA of its own or balanced
    chunk ranges)."""
    from query_aware_sparse_hs_gb300 import hs
    tc = w.kv_dtype in ("bf16", "fp8") and w.head_dim == 128 and w.block_size in (16, 32, 64, 128)
    if not tc:
        return 0 if attn_splits(w, dec, params) <= 1 else 1
    splits, per = hs.hs_attn_geometry(dec.shape, w.batch, dec.capacity, params)
    if splits <= 1 or per > 0:
        return 0
    ctas = params.max_ctas if 0 < params.max_ctas < _sms() else _sms()
    inline = dec.split_counters is not None and w.batch * w.num_kv_heads * splits <= ctas
    return 0 if inline else 1


def step_launches(w, dec, hot: bool = False, overlap: bool = False, allow_fused: bool = True) -> int:
    """Kernels of one step as the library dispatches them for this workload:
    either the single append + scoring + selection + attention launch (which
    merges its splits inside its clusters), or the append (not on the
    offload path), bound scoring + selection (select_launches), the swap-in
    (offload; with the copy overlapped: plan, page copy, attention over the
    copied blocks, attention over the resident blocks and the merge of the
    two) and attention; and the split merge unless the attention merges its
    splits itself (merge_launches)."""
    n = 0 if hot else 1
    if not hot and allow_fused and fused_step(w, dec):
        return 1  # the append runs inside the single launch
    n += select_launches(w)
    if hot and overlap:
        # plan (inside the selection's launch when the scorer takes its own
        # launch and a request has at most 1024 blocks), page copy, attention
        # over the copied blocks, attention over the hits (+ its split merge),
        # merge of the parts
        plan_in_select = (select_launches(w) == 2 and w.kv_dtype == "bf16" and w.head_dim == 128
                          and w.max_blocks <= 1024)
        return n + (4 if plan_in_select else 5) + merge_launches(w, dec, dec.hit_params)
    n += 1 if hot else 0
    n += 1
    return n + merge_launches(w, dec, dec.attn_params)


# ----------------------------------------------------------------------------
# DRAM traffic of the dominant kernel, from ncu captures (profiles/*.md)
# ----------------------------------------------------------------------------

# Per workload: the kernel, the DRAM bytes read + written by one captured launch
# (ncu dram__bytes_read.sum + dram__bytes_write.sum), that launch's algorithmic
# bytes, and a fingerprint of the CUDA sources the capture was taken on.  The
# bench scales the captured traffic to the timed launch by its algorithmic
# bytes (the units processed) and reports null once the sources have changed.
_SRC = "248cb333d6cbf9df"
NCU_TRAFFIC: dict = {
    ("llama8b_bf16", "score_select_attn_kernel"): {
        "traffic": 42191360, "algorithmic": 42217600, "sources": _SRC,
        "note": "ncu dram bytes of one score_select_attn_kernel launch of this workload (2 layer copies), "
                "profiles/ncu_full_score_select_attn_llama8b_bf16.md"},
    ("ragged_bf16", "attn_tc_kernel"): {
        "traffic": 144844544, "algorithmic": 143784896, "sources": _SRC,
        "note": "ncu dram bytes of one attn_tc_kernel launch at batch 16 (1 layer copy; equal splits there, "
                "balanced chunk ranges at full size), scaled to the timed launch by its algorithmic bytes; "
                "profiles/ncu_full_attn_tc_ragged_bf16.md"},
    ("fp8_g32", "attn_tc_fp8_kernel"): {
        "traffic": 76315904, "algorithmic": 75792384, "sources": _SRC,
        "note": "ncu dram bytes of one attn_tc_fp8_kernel launch at batch 16 (1 layer copy), scaled to the "
                "timed launch by its algorithmic bytes; profiles/ncu_full_attn_tc_fp8_fp8_g32.md"},
    ("offload_bf16", "attn_tc_kernel"): {
        "traffic": 124562176, "algorithmic": 134774784, "sources": _SRC,
        "note": "ncu dram bytes of one attn_tc_kernel launch at batch 32, scaled to the timed launch by its "
                "algorithmic bytes; at that size part of the 268 MB hot buffer stays in L2 (ratio 0.92; at full size it is 2.1 GB); "
                "profiles/ncu_full_attn_tc_offload_bf16.md"},
}


def source_fingerprint() -> str:
    """SHA-256 (first 16 hex digits) over the library's CUDA sources and header."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "query_aware_sparse_hs_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for p in files + [os.path.join(ROOT, "include", "hs.h")]:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_entry(workload: str, kernel: str, algorithmic: int) -> dict:
    e = NCU_TRAFFIC.get((workload, kernel))
    if not e or e["sources"] != source_fingerprint():
        return {"traffic": None, "traffic_note": "no ncu capture of the current kernel sources"}
    scaled = e["traffic"] * algorithmic / e["algorithmic"]
    return {"traffic": int(round(scaled)), "traffic_over_algorithmic": e["traffic"] / e["algorithmic"],
            "traffic_note": e["note"]}


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        if not rows:
            once = subprocess.run(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                   "--format=csv,noheader,nounits"], capture_output=True, text=True).stdout
            rows = [r.split(", ") for r in once.strip().splitlines() if r.strip()]
        sm = [float(r[1]) for r in rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def whole_job_rate(units: float, ms: float, world: int, device) -> tuple:
    """Replicas: every rank times its own units; the job's rate is all units
    over the slowest rank's time.  Returns (rate per second, max ms)."""
    if world == 1:
        return units / (ms / 1e3), ms
    import torch
    import torch.distributed as dist
    u = torch.tensor([units], dtype=torch.float64, device=device)
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(u.item()) / (float(t.item()) / 1e3), float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def split_counts(n: int, per: int) -> list:
    """n steps as whole rotations of `per` steps and one partial rotation."""
    return [per] * (n // per) + ([n % per] if n % per else [])


# ----------------------------------------------------------------------------
# CPU baseline / reference arm: the oracle as it stands, one (request, kv head)
# pair of the same workload per step, single thread
# ----------------------------------------------------------------------------

class OracleStep:
    """The oracle's per-step work for one (request, kv head) pair of the
    workload: append the newest token (resident workloads), bound, select,
    [hot-buffer step for the offload workload], attend."""

    def __init__(self, w, pairs: int = 4):
        import numpy as np
        import oracle as O
        from synth import drift_queries, make_inputs
        self.O, self.np = O, np
        self.w = w
        wb = w.scaled(batch=1)  # the sampled pairs come from one request of the workload
        x = make_inputs(wb, device="cpu")
        self.pairs = []
        B = w.block_size
        self.drift = drift_queries(wb, x["q"], w.decode_steps).float().numpy() if w.offload else None
        for kvh in range(min(pairs, w.num_kv_heads)):
            row = x["page_table"][0, kvh].numpy()
            L = int(x["seq_lens"][0])
            if w.kv_dtype == "fp8":
                D = w.head_dim
                kc, ks = O.quantize_e4m3_g32(x["k_pages"].float().numpy().reshape(-1, D))
                vc, vs = O.quantize_e4m3_g32(x["v_pages"].float().numpy().reshape(-1, D))
                P = x["k_pages"].shape[0]
                K = O.kv_values("fp8", O.gather_rows(kc.reshape(P, B, D), row, L, B),
                                O.gather_rows(ks.reshape(P, B, D // 32), row, L, B))
                V = O.kv_values("fp8", O.gather_rows(vc.reshape(P, B, D), row, L, B),
                                O.gather_rows(vs.reshape(P, B, D // 32), row, L, B))
            else:
                K = O.kv_values(w.kv_dtype, O.gather_rows(x["k_pages"].float().numpy(), row, L, B))
                V = O.kv_values(w.kv_dtype, O.gather_rows(x["v_pages"].float().numpy(), row, L, B))
            smin, smax = O.stored_summaries(*O.block_summaries(K, B), w.kv_dtype)
            g = w.group
            qg = x["q"][0, kvh * g:(kvh + 1) * g].float().numpy().astype(np.float64)
            newest = (O.gather_rows(x["k_pages"].float().numpy(), row, L, B)[L - 1:],
                      O.gather_rows(x["v_pages"].float().numpy(), row, L, B)[L - 1:])
            hb = O.HotBuffer(O.num_blocks(L, B), w.hot_slots) if w.offload else None
            self.pairs.append((kvh, K, V, smin, smax, qg, L, newest, hb))
        self.i = 0

    def step(self):
        """One pair's per-step work.  Returns the query heads served."""
        O, w, np = self.O, self.w, self.np
        kvh, K, V, smin, smax, qg, L, newest, hb = self.pairs[self.i % len(self.pairs)]
        t = self.i // len(self.pairs)
        self.i += 1
        B, g = w.block_size, w.group
        if w.offload:
            # the drifting query of decode step t; the context is held fixed
            t = t % w.decode_steps
            qg = self.drift[t, 0, kvh * g:(kvh + 1) * g].astype(np.float64)
        else:
            if w.kv_dtype == "fp8":
                for rows, dst in zip(newest, (K, V)):
                    dst[L - 1:] = O.kv_values("fp8", *O.quantize_e4m3_g32(rows))
            else:
                K[L - 1:], V[L - 1:] = O.kv_values(w.kv_dtype, newest[0]), O.kv_values(w.kv_dtype, newest[1])
            j = (L - 1) // B
            lo, hi = O.stored_summaries(*O.block_summaries(K[j * B:L], B), w.kv_dtype)
            smin[j], smax[j] = lo[0], hi[0]
        _, score = O.bound_scores(qg, smin, smax)
        sel = O.select_blocks(score, O.forced_blocks(L, B, w.sink_tokens, w.window_tokens), w.k_scored)
        if hb is not None:
            hb.step(sel, t)
        O.sparse_attention(qg, K, V, sel, B, 1.0 / math.sqrt(w.head_dim))
        return g


def _oracle_steps(st, seconds: float):
    t0 = time.perf_counter()
    heads, n = 0, 0
    while time.perf_counter() - t0 < seconds:
        heads += st.step()
        n += 1
    return heads, n, time.perf_counter() - t0


def cpu_baseline(w, seconds: float) -> dict:
    st = OracleStep(w)
    st.step()
    heads, n, dt = _oracle_steps(st, seconds)
    what = "bound + selection + hot-buffer step + attention" if w.offload else \
        "append + bound + selection + attention"
    return {"value": heads / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} single-(request, kv head) steps of {w.name} ({w.group} query heads each, "
                      f"request 0's {w.ctx_max if w.ctx_min == w.ctx_max else 'sampled'} tokens, {what}), "
                      f"numpy float64, 1 thread, {dt:.1f} s"}


def _oracle_worker(args):
    """One host process of the all-cores baseline: the oracle's per-pair step,
    repeated for `seconds`.  Returns (query heads served, seconds)."""
    name, seconds, seed = args
    from synth import WORKLOADS
    st = OracleStep(WORKLOADS[name])
    st.i = seed
    st.step()
    heads, _, dt = _oracle_steps(st, seconds)
    return heads, dt


def cpu_baseline_all_cores(w, seconds: float) -> dict:
    """The same oracle step on every host core: one process per core, each on
    its own (request, kv head) pairs (the pairs are independent).  Processes are
    started with 'spawn', so no CUDA state is inherited."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(w.name, seconds, i) for i in range(cores)])
    heads = sum(r[0] for r in res)
    dt = max(r[1] for r in res)
    return {"value": heads / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes x {seconds:.0f} s of single-(request, kv head) steps of {w.name}, "
                      f"numpy float64, 1 thread each"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    st = OracleStep(w)
    for _ in range(args.warmup):
        st.step()
    t0 = time.perf_counter()
    heads = 0
    for _ in range(args.steps):
        heads += st.step()
    dt = time.perf_counter() - t0
    value = heads / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"each step = one (request, kv head) pair of {w.name}, numpy float64, "
                                       f"1 thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w, layers: int | None = None) -> dict:
    c = {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
         "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
         "kv_dtype": w.kv_dtype,
         "context": w.ctx_max if w.ctx_min == w.ctx_max else [w.ctx_min, w.ctx_max],
         "sink_tokens": w.sink_tokens, "window_tokens": w.window_tokens, "k_scored": w.k_scored,
         "parallelism": "replicas"}
    if w.offload:
        c.update(hot_slots_per_stream=w.hot_slots, decode_steps=w.decode_steps,
                 l2="inputs larger than L2: hot buffer 2.1 GB and summaries 268 MB read every step")
    elif layers is not None:
        c.update(layer_copies=layers, l2=f"inputs larger than L2: {layers} distinct layer copies rotate step to step",
                 early_summaries=layers > 1)
    return c


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def attn_work(dec) -> dict:
    """How the tensor-core attention divides its work (hs_attn_geometry):
    balanced chunk ranges of chunks_per_cta chunks, or equal splits per pair."""
    from query_aware_sparse_hs_gb300 import hs
    splits, per = hs.hs_attn_geometry(dec.shape, dec.batch, dec.capacity, dec.attn_params)
    return {"mode": "balanced_ranges" if per > 0 else "equal_splits", "splits": splits, "chunks_per_cta": per}


class Graphs:
    """CUDA graphs of `fn(i)` over step ranges, captured once per range."""

    def __init__(self, stream, fn):
        self.stream, self.fn, self.cache = stream, fn, {}

    def get(self, first: int, n: int):
        import torch
        key = (first, n)
        if key not in self.cache:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(first, first + n):
                    self.fn(i)
            self.cache[key] = g
        return self.cache[key]


def _events():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def measure_resident(args, w, dev, world) -> dict:
    """One of the workloads whose whole cache is in HBM.  Steps rotate over
    distinct layer copies and replay from CUDA graphs."""
    import torch

    from query_aware_sparse_hs_gb300 import hs
    from query_aware_sparse_hs_gb300.decode import SparseDecode
    from synth import make_layer, make_layout

    layout = make_layout(w, dev)
    layers = args.layers
    if layers <= 0:  # as many distinct layer copies as fit in ~24 GB, at most 32
        per_layer = layout["num_pages"] * w.block_size * token_bytes(w)
        layers = int(max(1, min(32, (24 << 30) // max(per_layer, 1))))
    lens, table = layout["seq_lens"], layout["page_table"]
    B, D = w.block_size, w.head_dim
    decs, kvs, qs, news, inputs, keep = [], [], [], [], [], []
    for layer in range(layers):
        x = make_layer(w, layout, dev, layer)
        k, v, q = x["k_pages"], x["v_pages"], x["q"]
        # the newest token's K/V (source precision), appended again every step
        t_last = (lens.long() - 1)[:, None].expand(w.batch, w.num_kv_heads)
        pg = table[torch.arange(w.batch, device=dev)[:, None], torch.arange(w.num_kv_heads, device=dev)[None, :],
                   t_last // w.block_size].long()
        # q and the new K/V share one device buffer, so the end-to-end step
        # brings its inputs over in one host-to-device copy
        nq, nkv = q.numel(), w.batch * w.num_kv_heads * w.head_dim
        packed = torch.empty(nq + 2 * nkv, dtype=q.dtype, device=dev)
        packed[:nq].copy_(q.reshape(-1))
        packed[nq:nq + nkv].copy_(k[pg, t_last % w.block_size].reshape(-1))
        packed[nq + nkv:].copy_(v[pg, t_last % w.block_size].reshape(-1))
        q = packed[:nq].view(q.shape)
        new_kv = (packed[nq:nq + nkv].view(w.batch, w.num_kv_heads, w.head_dim),
                  packed[nq + nkv:].view(w.batch, w.num_kv_heads, w.head_dim))
        inputs.append(packed)
        ks = vs = None
        if w.kv_dtype == "fp8":
            kc = torch.empty(k.shape, dtype=torch.uint8, device=dev)
            vc = torch.empty_like(kc)
            ks = torch.empty(k.shape[:-1] + (D // 32,), dtype=torch.float32, device=dev)
            vs = torch.empty_like(ks)
            hs.hs_quantize_e4m3_g32(k, kc, ks)
            hs.hs_quantize_e4m3_g32(v, vc, vs)
            del k, v
            k, v = kc, vc
        kv = hs.paged_kv(k, v, table, lens, ks, vs)
        # layers are stepped in turn, so with two or more the kernel before a
        # layer's step never writes that layer's summaries
        dec = SparseDecode(num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=D,
                           block_size=B, kv_dtype=w.kv_dtype, batch=w.batch, max_blocks=w.max_blocks,
                           sink_tokens=w.sink_tokens, window_tokens=w.window_tokens,
                           k_scored=w.k_scored, early_summaries=layers > 1, device=dev)
        dec.build_summaries(kv)
        decs.append(dec)
        kvs.append(kv)
        qs.append(q)
        news.append(new_kv)
        keep.append((k, v, ks, vs))
    torch.cuda.synchronize()
    st_, bits, where = hs.hs_get_device_error_detail()
    assert st_ == hs.HS_OK, (st_, bits, where)

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.current_stream().wait_stream(stream)

    def one_step(i):
        li = i % layers
        lead = li - li % args.select_every  # layer whose selection this layer uses
        decs[li].step(kvs[li], qs[li], new_kv=news[li], reuse=None if lead == li else decs[lead], stream=stream)

    # eager warm-up (module load, cluster attributes) before capture
    with torch.cuda.stream(stream):
        for i in range(layers):
            one_step(i)
    stream.synchronize()
    steps_g = Graphs(stream, one_step)

    def run_steps(n):
        """Exactly n steps: whole rotations over the layers, then a partial one."""
        for c in split_counts(n, layers):
            steps_g.get(0, c).replay()

    # set-up, outside the W + K steps: every graph the warm-up, the timed
    # steps and the long run replay is captured and launched once (its
    # upload), so no capture or first launch falls into a timed region
    with torch.cuda.stream(stream):
        for c in sorted(set(split_counts(args.warmup, layers) + split_counts(args.steps, layers) + [layers])):
            steps_g.get(0, c).replay()
    stream.synchronize()
    with torch.cuda.stream(stream):
        run_steps(args.warmup)
    stream.synchronize()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = _events()
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(args.steps)
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    value, ms = whole_job_rate(args.steps * w.batch * w.num_q_heads, e0.elapsed_time(e1), world, dev)
    ms_per_step = ms / args.steps
    # a long run (at least half a second of timed steps) beside the exact-K figure
    rot_ms = ms_per_step * layers
    long_reps = max(1, math.ceil(LONG_RUN_S * 1e3 / max(rot_ms, 1e-3)))
    full = steps_g.get(0, layers)
    a, b = _events()
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(long_reps):
            full.replay()
        b.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    long_steps = long_reps * layers
    long_ms = a.elapsed_time(b)
    long_run = {"steps": long_steps, "seconds": long_ms / 1e3, "ms_per_step": long_ms / long_steps,
                "value": long_steps * w.batch * w.num_q_heads / (long_ms / 1e3)}

    # ---- per-kernel times (each kernel alone, the same rotating layers) ----
    def timed_graph(fn, rr=None):
        g = Graphs(stream, fn).get(0, layers)
        with torch.cuda.stream(stream):
            g.replay()
            g.replay()
        stream.synchronize()
        rr = rr or max(3, min(long_reps, 200))
        x0, x1 = _events()
        with torch.cuda.stream(stream):
            x0.record(stream)
            for _ in range(rr):
                g.replay()
            x1.record(stream)
        stream.synchronize()
        return x0.elapsed_time(x1) * 1e3 / (rr * layers)  # microseconds per launch

    def lead_of(li):
        return decs[li - li % args.select_every]

    t_attn = timed_graph(lambda i: decs[i % layers].attend(kvs[i % layers], qs[i % layers], stream,
                                                           selection=lead_of(i % layers)))
    fused = fused_step(w, decs[0])
    t_fused = (timed_graph(lambda i: decs[i % layers].select_attend(kvs[i % layers], qs[i % layers], stream=stream))
               if fused else None)
    t_decode = (timed_graph(lambda i: decs[i % layers].decode_step(kvs[i % layers], qs[i % layers], *news[i % layers],
                                                                    stream=stream))
                if fused else None)
    t_sel = timed_graph(lambda i: decs[i % layers].select(kvs[i % layers], qs[i % layers], stream=stream))
    t_app = timed_graph(lambda i: decs[i % layers].append(kvs[i % layers], *news[i % layers], stream))
    t_sum_full = timed_graph(lambda i: decs[i % layers].build_summaries(kvs[i % layers], 0, stream), rr=3)

    # algorithmic bytes from the actual selection
    d0 = decs[0]
    cnt = d0.sel_count.cpu().numpy()
    sel = d0.sel.cpu().numpy()
    lens_np = lens.cpu().numpy()
    sel_tokens = 0
    for bq in range(w.batch):
        L = int(lens_np[bq])
        for kvh in range(w.num_kv_heads):
            for j in sel[bq, kvh, :cnt[bq, kvh]]:
                sel_tokens += min(B, L - int(j) * B)
    pairs_blocks = int(cnt.sum())
    total_blocks = int(sum(w.num_kv_heads * ((int(L) + B - 1) // B) for L in lens_np))
    a_bytes = attn_bytes(w, sel_tokens, pairs_blocks)
    s_bytes = select_bytes(w, total_blocks)
    append_bytes = append_bytes_per_step(w)
    step_bytes = a_bytes + s_bytes + append_bytes
    full_sum_bytes = total_blocks * (B * token_bytes(w) / 2 + summary_bytes_per_block(w))
    peak, peak_kind = load_peaks()
    attn_gbs = a_bytes / (t_attn * 1e-6) / 1e9
    # the dominant kernel: the single scoring + selection + attention launch
    # where the step uses it, else the attention launch (with its merge)
    if fused:
        dom = {"kernel": "score_select_attn_kernel", "what": "decode_step: append + scoring + selection + "
                                                             "attention + split merge in one launch",
               "bytes": a_bytes + s_bytes + append_bytes, "us": t_decode}
    else:
        dom = {"kernel": "attn_tc_fp8_kernel" if w.kv_dtype == "fp8" else "attn_tc_kernel",
               "what": "sparse_paged_decode_attn", "bytes": a_bytes, "us": t_attn}
    dom_gbs = dom["bytes"] / (dom["us"] * 1e-6) / 1e9

    # ---- end to end through the C ABI with host buffers ----
    # per step: one copy of the step's inputs (q, new K/V) from pinned host
    # memory, the step, one copy of its results (out, lse) back; the results
    # drain on a side stream while the next step runs (the next step's inputs
    # are not fetched ahead: in a model they depend on this step)
    in_host = [inputs[i].cpu().pin_memory() for i in range(layers)]
    res_host = torch.empty((layers, d0.results.numel()), dtype=torch.uint8).pin_memory()
    drain = torch.cuda.Stream(device=dev)

    def e2e_step(i):
        li = i % layers
        inputs[li].copy_(in_host[li], non_blocking=True)
        one_step(i)
        drain.wait_stream(stream)
        with torch.cuda.stream(drain):
            res_host[li].copy_(decs[li].results, non_blocking=True)

    class E2EGraphs(Graphs):
        def get(self, first, n):
            key = (first, n)
            if key not in self.cache:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    for i in range(first, first + n):
                        e2e_step(i)
                    self.stream.wait_stream(drain)  # every result is on the host when the graph ends
                self.cache[key] = g
            return self.cache[key]

    e2e_g = E2EGraphs(stream, None)

    def run_e2e(n):
        for c in split_counts(n, layers):
            e2e_g.get(0, c).replay()

    with torch.cuda.stream(stream):  # capture and upload, then the W warm-up steps
        for c in sorted(set(split_counts(args.warmup, layers) + split_counts(args.steps, layers))):
            e2e_g.get(0, c).replay()
        run_e2e(args.warmup)
    stream.synchronize()
    barrier(world)
    a, b_ = _events()
    with torch.cuda.stream(stream):
        a.record(stream)
        run_e2e(args.steps)
        b_.record(stream)
    stream.synchronize()
    e2e_value, ms_e2e = whole_job_rate(args.steps * w.batch * w.num_q_heads, a.elapsed_time(b_), world, dev)
    last = (args.steps - 1) % layers
    assert torch.equal(res_host[last], decs[last].results.cpu()), "results drained to the host differ"
    h2d = inputs[0].numel() * inputs[0].element_size()
    d2h = d0.results.numel()

    st_, bits, where = hs.hs_get_device_error_detail()
    assert st_ == hs.HS_OK, (st_, bits, where)
    # a layer that reuses a selection runs append + attention (+ merge)
    reuse_launches = (1 if fused_step(w, d0) else
                      step_launches(w, d0, allow_fused=False) - select_launches(w))
    launches_per_step = step_launches(w, d0) / args.select_every + reuse_launches * (1 - 1 / args.select_every)
    rec = {
        "value": value, "unit": UNIT, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "dtype": w.kv_dtype, "config": dict(workload_config(w, layers), select_every=args.select_every,
                                            attn_work=attn_work(d0)),
        "hbm_gbs_step": step_bytes / (ms_per_step * 1e-3) / 1e9,
        "roofline": dict({"bound": "hbm", "kernel": dom["kernel"], "what": dom["what"], "achieved": dom_gbs,
                          "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": dom_gbs / peak},
                         **traffic_entry(w.name, dom["kernel"], dom["bytes"]),
                         algorithmic_bytes_per_launch=dom["bytes"], avg_launch_us=dom["us"]),
        "kernels_us": {"decode_step": t_decode, "append": t_app, "score_select_attend": t_fused, "score_select": t_sel,
                       "attention_with_merge": t_attn, "summary_build_full": t_sum_full},
        "kernels_gbs": {"decode_step": dom_gbs if fused else None,
                        "score_select": s_bytes / (t_sel * 1e-6) / 1e9,
                        "attention_with_merge": attn_gbs,
                        "summary_build_full": full_sum_bytes / (t_sum_full * 1e-6) / 1e9},
        "bytes_per_step": {"attention": a_bytes, "score_select": s_bytes, "append": int(append_bytes)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": ms_e2e / args.steps},
        "long_run": long_run,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clk,
    }
    del decs, kvs, qs, news, inputs, keep, steps_g, e2e_g
    return rec


def measure_offload(args, w, dev, world) -> dict:
    """HiSparse workload: every step = score/select against the summaries of the
    whole cache, swap-in of the missing pages from the pinned host pool into the
    hot device buffer (overlapped with the attention over the blocks already
    resident), attention over the hot slots, merge.  A pass is the 64-step
    drifting-query sequence; step 0 (empty buffer) refills it untimed, steps
    1..63 are the timed steps.  Reports the miss rate and the swap-in bandwidth
    next to the measured host-to-device copy bandwidth."""
    import torch

    from query_aware_sparse_hs_gb300 import hs
    from query_aware_sparse_hs_gb300.decode import SparseDecode
    from synth import drift_queries, make_layer, make_layout

    B, D, S, hkv = w.block_size, w.head_dim, w.hot_slots, w.num_kv_heads
    nb, pairs, steps_seq = w.max_blocks, w.batch * w.num_kv_heads, w.decode_steps
    layout = make_layout(w, dev)
    x = make_layer(w, layout, dev, 0)
    host_k = torch.empty(x["k_pages"].shape, dtype=x["k_pages"].dtype, pin_memory=True)
    host_v = torch.empty_like(host_k, pin_memory=True)
    host_k.copy_(x["k_pages"])
    host_v.copy_(x["v_pages"])
    qs = drift_queries(w, x["q"], steps_seq)
    del x
    torch.cuda.empty_cache()
    lens, ptab = layout["seq_lens"], layout["page_table"]
    pool_kv = hs.paged_kv(host_k, host_v, ptab, lens)
    table = torch.full((w.batch, hkv, nb), -1, dtype=torch.int32, device=dev)
    owner = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
    last = torch.full((w.batch, hkv, S), -1, dtype=torch.int32, device=dev)
    k_slots = torch.empty((pairs * S, B, D), dtype=host_k.dtype, device=dev)
    v_slots = torch.empty_like(k_slots)
    hb = hs.hot_buffer(table, owner, last, k_slots, v_slots, host_k, host_v, S)
    slot_kv = hs.paged_kv(k_slots, v_slots, table, lens)
    stats = torch.zeros(4, dtype=torch.int64, device=dev)
    dec = SparseDecode(num_q_heads=w.num_q_heads, num_kv_heads=hkv, head_dim=D, block_size=B, kv_dtype=w.kv_dtype,
                       batch=w.batch, max_blocks=nb, sink_tokens=w.sink_tokens, window_tokens=w.window_tokens,
                       k_scored=w.k_scored, score_smoothing=args.score_smoothing, device=dev)
    dec.build_summaries(pool_kv)  # read over the host link once
    if args.swap_overlap:
        dec.enable_swap_overlap(args.swap_copy_ctas, args.swap_attn_ctas)
    stream = torch.cuda.Stream(device=dev)
    # the query of the step being run: the end-to-end form copies each step's
    # query from pinned host memory into this buffer; the resident form uses
    # the device copy of the whole drift sequence
    q_in = torch.empty_like(qs[0])

    def reset():
        table.fill_(-1)
        owner.fill_(-1)
        last.fill_(-1)
        dec.reset_score_history()

    def step(t, st=None, q=None):
        dec.step(pool_kv, qs[t] if q is None else q, hot=(hb, slot_kv, t, st), stream=stream)

    timed_per_pass = steps_seq - 1
    # graphs over decode steps first..first+n-1 of a pass (first >= 1)
    step_g = Graphs(stream, lambda t: step(t, stats))

    def segments(start, n):
        """Positions start..start+n-1 of the endless run of decode steps
        (position p = decode step 1 + p % 63 of pass p // 63) as graph
        segments (first step, count, refill before): a pass begins with an
        untimed reset and step 0, the refill of the empty hot buffer."""
        out, p, end = [], start, start + n
        while p < end:
            t = 1 + p % timed_per_pass
            c = min(end - p, timed_per_pass - (t - 1))
            out.append((t, c, t == 1))
            p += c
        return out

    def run_segments(segs, graphs=step_g, timed=False):
        """Replays the segments; returns the device time of their steps (ms)
        when timed (the refills are outside the events)."""
        total = 0.0
        for first, cnt, refill in segs:
            g = graphs.get(first, cnt)
            with torch.cuda.stream(stream):
                if refill:
                    reset()
                    step(0)
                if timed:
                    a, b = _events()
                    a.record(stream)
                g.replay()
                if timed:
                    b.record(stream)
            if timed:
                stream.synchronize()
                total += a.elapsed_time(b)
        stream.synchronize()
        return total

    def upload(segs, graphs=step_g):
        """Set-up: capture each segment's graph and launch it once (its upload)
        on a throw-away pass, so that no capture or first launch is timed."""
        for first, cnt, _ in segs:
            run_segments([(first, cnt, True)], graphs)

    warm_segs = segments(0, args.warmup)
    timed_segs = segments(args.warmup, args.steps)
    long_start = -(-(args.warmup + args.steps) // timed_per_pass) * timed_per_pass
    # eager pass (module load, attributes), then the graphs' set-up
    with torch.cuda.stream(stream):
        reset()
        for t in range(steps_seq):
            step(t, stats)
    stream.synchronize()
    upload(warm_segs + timed_segs + [(1, timed_per_pass, True)])
    # the run: W warm-up steps, then exactly K timed steps that follow them
    run_segments(warm_segs)
    stats.zero_()
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ms = run_segments(timed_segs, timed=True)
    torch.cuda.synchronize()
    barrier(world)
    st = stats.cpu().tolist()
    value, ms = whole_job_rate(args.steps * w.batch * w.num_q_heads, ms, world, dev)
    ms_per_step = ms / args.steps
    # long run: whole passes, at least half a second of timed steps
    long_passes = max(1, math.ceil(LONG_RUN_S * 1e3 / max(ms_per_step * timed_per_pass, 1e-3)))
    stats.zero_()
    long_ms = run_segments(segments(long_start, long_passes * timed_per_pass), timed=True)
    clk = clocks.stop()
    long_steps = long_passes * timed_per_pass
    st_long = stats.cpu().tolist()
    long_run = {"steps": long_steps, "seconds": long_ms / 1e3, "ms_per_step": long_ms / long_steps,
                "value": long_steps * w.batch * w.num_q_heads / (long_ms / 1e3),
                "miss_rate": st_long[1] / max(1, st_long[0] + st_long[1]),
                "what": f"{long_passes} whole passes of decode steps 1..{timed_per_pass}"}

    # the same steps with the swap-in and the attention one after the other
    side, dec.side_stream = getattr(dec, "side_stream", None), None
    serial_g = Graphs(stream, lambda t: step(t, stats))
    serial_g.get(1, timed_per_pass)
    dec.side_stream = side
    run_segments(segments(0, timed_per_pass), serial_g)
    ms_serial = run_segments(segments(0, timed_per_pass), serial_g, timed=True) / timed_per_pass

    # per-kernel times over one pass, each call bracketed by events (eager,
    # serial form); the pass's own swap-in statistics go with its times
    stats_pass = torch.zeros(4, dtype=torch.int64, device=dev)
    ev = {k: [] for k in ("select", "swapin", "attention")}
    with torch.cuda.stream(stream):
        reset()
        step(0)
        for t in range(1, steps_seq):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            dec.select(pool_kv, qs[t], stream=stream)
            e[1].record(stream)
            dec.swap_in(hb, t, stats_pass, stream)
            e[2].record(stream)
            dec.attend(slot_kv, qs[t], stream=stream)
            e[3].record(stream)
            ev["select"].append(e[:2])
            ev["swapin"].append(e[1:3])
            ev["attention"].append(e[2:4])
    stream.synchronize()
    t_us = {k: 1e3 * sum(a.elapsed_time(b) for a, b in v) / len(v) for k, v in ev.items()}
    sel_blocks_step = int(dec.sel_count.sum().item())
    st_pass = stats_pass.cpu().tolist()

    # ---- end to end through the C ABI with host buffers: every step copies
    # its query from pinned host memory and its results (out, lse) back ----
    q_host = qs.cpu().pin_memory()
    res_host = torch.empty((steps_seq, dec.results.numel()), dtype=torch.uint8).pin_memory()
    drain = torch.cuda.Stream(device=dev)

    def e2e_step(t):
        q_in.copy_(q_host[t], non_blocking=True)
        step(t, stats, q_in)
        drain.wait_stream(stream)
        with torch.cuda.stream(drain):
            res_host[t].copy_(dec.results, non_blocking=True)

    class E2EGraphs(Graphs):
        def get(self, first, n):
            key = (first, n)
            if key not in self.cache:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    for t in range(first, first + n):
                        e2e_step(t)
                    self.stream.wait_stream(drain)  # every result is on the host when the graph ends
                self.cache[key] = g
            return self.cache[key]

    e2e_g = E2EGraphs(stream, None)
    upload(warm_segs + timed_segs, e2e_g)
    run_segments(warm_segs, e2e_g)
    barrier(world)
    ms_e2e = run_segments(timed_segs, e2e_g, timed=True)
    e2e_value, ms_e2e = whole_job_rate(args.steps * w.batch * w.num_q_heads, ms_e2e, world, dev)
    t_last = 1 + (args.warmup + args.steps - 1) % timed_per_pass
    assert torch.equal(res_host[t_last], dec.results.cpu()), "results drained to the host differ"
    st_, bits, where = hs.hs_get_device_error_detail()
    assert st_ == hs.HS_OK, (st_, bits, where)

    # host -> device link bandwidth: 1 GiB from pinned memory, best of 5
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    link = 0.0
    for _ in range(5):
        a, b = _events()
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        link = max(link, (1 << 30) / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst

    hits, misses, evictions, bytes_in = st
    page_bytes = B * token_bytes(w)  # K+V of one block
    a_bytes = attn_bytes(w, sel_blocks_step * B, sel_blocks_step)
    s_bytes = select_bytes(w, pairs * nb)
    peak, peak_kind = load_peaks()
    attn_gbs = a_bytes / (t_us["attention"] * 1e-6) / 1e9
    swap_bytes_step = bytes_in / args.steps
    pass_swap_bytes = st_pass[3] / timed_per_pass  # the eager pass whose swap-in was timed
    rec = {
        "value": value, "unit": UNIT, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "dtype": w.kv_dtype,
        "config": dict(workload_config(w), overlapped_swap_in=bool(args.swap_overlap),
                       score_smoothing=args.score_smoothing),
        "hbm_gbs_step": (a_bytes + s_bytes) / (ms_per_step * 1e-3) / 1e9,
        "roofline": dict({"bound": "hbm", "kernel": "attn_tc_kernel",
                          "what": "sparse_paged_decode_attn over the hot slots (all selected blocks)",
                          "achieved": attn_gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                          "frac": attn_gbs / peak},
                         **traffic_entry(w.name, "attn_tc_kernel", a_bytes),
                         algorithmic_bytes_per_launch=a_bytes, avg_launch_us=t_us["attention"]),
        "swap": {"miss_rate": misses / max(1, hits + misses), "misses_per_step": misses / args.steps,
                 "evictions_per_step": evictions / args.steps, "bytes_in_per_step": swap_bytes_step,
                 "timed_steps": f"the {args.steps} decode steps after {args.warmup} warm-up steps of the "
                                f"{steps_seq}-step drifting sequence (step 0 of a pass refills the empty buffer, untimed)",
                 "swapin_us_per_pass_step": t_us["swapin"],
                 "swapin_bytes_per_pass_step": pass_swap_bytes,
                 "miss_rate_pass": st_pass[1] / max(1, st_pass[0] + st_pass[1]),
                 "swapin_gbs": pass_swap_bytes / (t_us["swapin"] * 1e-6) / 1e9,
                 "link_h2d_gbs_measured": link,
                 "link_frac": pass_swap_bytes / (t_us["swapin"] * 1e-6) / 1e9 / link,
                 "page_bytes": page_bytes},
        "kernels_us": {"score_select": t_us["select"], "swapin": t_us["swapin"],
                       "attention_with_merge": t_us["attention"]},
        "kernels_gbs": {"score_select": s_bytes / (t_us["select"] * 1e-6) / 1e9, "attention_with_merge": attn_gbs},
        "bytes_per_step": {"attention": a_bytes, "score_select": s_bytes, "swap_in_host": int(swap_bytes_step)},
        "serial_ms_per_step": ms_serial,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": q_in.numel() * q_in.element_size(),
                "d2h_bytes_per_step": dec.results.numel(), "ms_per_step": ms_e2e / args.steps,
                "note": "the swap-in's own reads of the pinned host pool are part of the step, not of these copies"},
        "long_run": long_run,
        "gpu_launches": step_launches(w, dec, hot=True, overlap=bool(args.swap_overlap)) * args.steps,
        "clocks": clk,
    }
    del dec, hb, slot_kv, pool_kv, host_k, host_v, k_slots, v_slots, step_g, serial_g, e2e_g
    return rec


def run_ours(args, names):
    import torch
    from synth import WORKLOADS

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    recs = {}
    for name in names:
        w = WORKLOADS[name]
        if args.batch > 0:
            w = w.scaled(batch=args.batch)
        rec = measure_offload(args, w, dev, world) if w.offload else measure_resident(args, w, dev, world)
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        recs[name] = rec
    if rank != 0:
        return
    if world == 1 and args.cpu_seconds > 0:
        for name in names:
            w = WORKLOADS[name]
            recs[name]["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        recs[names[0]]["cpu_baseline_all_cores"] = cpu_baseline_all_cores(WORKLOADS[names[0]], args.cpu_seconds)
    head = recs[names[0]]
    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
            "config": head["config"]}
    for k, v in head.items():
        if k not in line and k not in ("steps", "warmup"):
            line[k] = v
    if len(names) > 1:
        line["workloads"] = {n: recs[n] for n in names[1:]}
        line["gpu_launches_all_workloads"] = sum(recs[n]["gpu_launches"] for n in names)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all", help="all, or one workload name")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling captures)")
    ap.add_argument("--layers", type=int, default=0, help="distinct layer copies (0 = fit ~24 GB, max 32)")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--select-every", type=int, default=1,
                    help="layers per selection: the first layer of each group selects, the others reuse it "
                         "(SparDA-style cross-layer reuse); 1 = every layer selects")
    ap.add_argument("--score-smoothing", type=float, default=0.0,
                    help="offload workload: weight of the previous step's block scores (0.3 in the SparDA article)")
    ap.add_argument("--swap-overlap", type=int, default=1,
                    help="offload workload: 1 = page copy overlapped with attention over the hits, 0 = one after the other")
    ap.add_argument("--swap-copy-ctas", type=int, default=12, help="CTAs (SMs) of the overlapped page copy")
    ap.add_argument("--swap-attn-ctas", type=int, default=0,
                    help="CTAs of the attention beside the copy (0 = the SMs the copy leaves)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    if args.select_every < 1:
        ap.error("--select-every must be >= 1")
    from synth import WORKLOADS
    names = [HEADLINE, *SUB_WORKLOADS] if args.workload == "all" else [args.workload]
    for n in names:
        if n not in WORKLOADS:
            ap.error(f"unknown workload {n}")
    if args.impl == "reference":
        w = WORKLOADS[names[0]]
        run_reference(args, w.scaled(batch=args.batch) if args.batch > 0 else w)
    else:
        run_ours(args, names)


if __name__ == "__main__":
    main()
