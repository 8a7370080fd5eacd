"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs.  The oracle only ever receives the
seeded inputs (or its own results), never something the CUDA path computed."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
from query_aware_sparse_hs_gb300 import hs
from query_aware_sparse_hs_gb300.decode import SparseDecode

TOL = {"f32": 1e-5, "bf16": 2e-3, "fp8": 2e-2, "fp8_dequant": 2e-3}


def np32(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.numpy()


class Case:
    """Seeded inputs of one workload on the GPU plus the CPU copies the oracle reads."""

    def __init__(self, w, x: dict, device="cuda", tail_nan=True):
        self.w = w
        dev = torch.device(device)
        self.x = x
        self.seq_lens = x["seq_lens"].to(dev)
        self.page_table = x["page_table"].to(dev)
        self.q = x["q"].to(dev)
        src_k, src_v = x["k_pages"], x["v_pages"]
        self.k_src_np = np32(src_k)  # values before quantisation (fp8) / as stored
        self.v_src_np = np32(src_v)
        if w.kv_dtype == "fp8":
            D = w.head_dim
            kc, ks = O.quantize_e4m3_g32(self.k_src_np.reshape(-1, D))
            vc, vs = O.quantize_e4m3_g32(self.v_src_np.reshape(-1, D))
            P, B = src_k.shape[0], src_k.shape[1]
            self.k_codes_np, self.v_codes_np = kc.reshape(P, B, D), vc.reshape(P, B, D)
            self.k_scales_np, self.v_scales_np = ks.reshape(P, B, D // 32), vs.reshape(P, B, D // 32)
            k_dev = torch.from_numpy(self.k_codes_np).to(dev)
            v_dev = torch.from_numpy(self.v_codes_np).to(dev)
            self.k_scales = torch.from_numpy(self.k_scales_np).to(dev)
            self.v_scales = torch.from_numpy(self.v_scales_np).to(dev)
        else:
            k_dev, v_dev = src_k.to(dev).clone(), src_v.to(dev).clone()
            self.k_scales = self.v_scales = None
        if tail_nan:
            self._poison_tails(k_dev, v_dev)
        self.k_pages, self.v_pages = k_dev.contiguous(), v_dev.contiguous()
        self.kv = hs.paged_kv(self.k_pages, self.v_pages, self.page_table, self.seq_lens,
                              self.k_scales, self.v_scales)
        self.lens = x["seq_lens"].tolist()
        self.table_np = x["page_table"].numpy()

    def _poison_tails(self, k, v):
        """Rows past the end of each request's last block hold NaN: they must never
        reach a result."""
        B = self.w.block_size
        for b, L in enumerate(self.x["seq_lens"].tolist()):
            if L % B == 0 or L == 0:
                continue
            j = (L - 1) // B
            bad = 0x7F if k.dtype == torch.uint8 else float("nan")  # e4m3 NaN code
            for kvh in range(self.w.num_kv_heads):
                p = int(self.x["page_table"][b, kvh, j])
                k[p, L % B:] = bad
                v[p, L % B:] = bad

    def decoder(self, **kw) -> SparseDecode:
        w = self.w
        args = dict(num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                    block_size=w.block_size, kv_dtype=w.kv_dtype, batch=w.batch,
                    max_blocks=self.page_table.shape[-1], sink_tokens=w.sink_tokens,
                    window_tokens=w.window_tokens, k_scored=w.k_scored)
        args.update(kw)
        return SparseDecode(**args)

    # ---- oracle side ----
    def logical(self, b, kvh, which="k", dequant=True):
        """float64 logical rows [L][D] of (b, kvh) as the kernel sees them."""
        L, B = self.lens[b], self.w.block_size
        row = self.table_np[b, kvh]
        if self.w.kv_dtype == "fp8":
            codes = self.k_codes_np if which == "k" else self.v_codes_np
            scales = self.k_scales_np if which == "k" else self.v_scales_np
            if not dequant:
                src = self.k_src_np if which == "k" else self.v_src_np
                return O.gather_rows(src, row, L, B).astype(np.float64)
            c = O.gather_rows(codes, row, L, B)
            s = O.gather_rows(scales, row, L, B)
            return O.kv_values("fp8", c, s)
        src = self.k_src_np if which == "k" else self.v_src_np
        return O.kv_values(self.w.kv_dtype, O.gather_rows(src, row, L, B))

    def q_group(self, b, kvh):
        g = self.w.group
        return np32(self.x["q"][b, kvh * g:(kvh + 1) * g]).astype(np.float64)

    def oracle_pair(self, b, kvh, scale=None, dequant=True):
        w = self.w
        scale = scale if scale is not None else 1.0 / math.sqrt(w.head_dim)
        K = self.logical(b, kvh, "k", dequant=True)
        V = self.logical(b, kvh, "v", dequant=dequant)
        Kq = K if dequant else self.logical(b, kvh, "k", dequant=False)
        r = O.decode_pair(self.q_group(b, kvh), K, V, w.block_size, w.kv_dtype, w.sink_tokens,
                          w.window_tokens, w.k_scored, scale)
        if not dequant:
            r["out"], r["lse"] = O.sparse_attention(self.q_group(b, kvh), Kq, V, r["sel"],
                                                    w.block_size, scale)
        return r


def tie_window_ok(oracle_score, forced, sel_gpu, sel_oracle, k_scored, rel=1e-5):
    """Selections may differ only among blocks whose oracle score lies within the
    relative tie window of the k-th best non-forced score."""
    if set(sel_gpu) == set(sel_oracle):
        return True
    if len(sel_gpu) != len(sel_oracle) or not set(forced) <= set(sel_gpu):
        return False
    fset = set(forced)
    rest = sorted((s, j) for j, s in enumerate(oracle_score) if j not in fset)
    rest.sort(key=lambda t: (-t[0], t[1]))
    kth = rest[k_scored - 1][0]
    nxt = rest[k_scored][0] if k_scored < len(rest) else -np.inf
    if abs(kth - nxt) >= rel * max(abs(kth), 1e-30):
        return False
    diff = set(sel_gpu) ^ set(sel_oracle)
    return all(abs(oracle_score[j] - kth) <= rel * max(abs(kth), 1e-30) for j in diff)
