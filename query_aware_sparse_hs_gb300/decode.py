"""Decode-step driver: owns the per-step device buffers and issues the library
calls of one step in order (token append or summary refresh -> score/select
-> [swap-in] -> attention).  All buffers are torch allocations made once in the constructor;
a step itself allocates nothing, so it can be captured in a CUDA graph.
"""

from __future__ import annotations

import math

import torch

from . import hs

_SUMMARY_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.bfloat16}
_Q_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.bfloat16}


class SparseDecode:
    """Buffers and calls of one decode step for one layer.

    score_smoothing: weight of the previous step's block scores (0 = off).
    inline_merge: give the tensor-core attention split counters so that it
    merges its splits itself.  fuse_step: a step without a hot buffer or a
    reused selection runs selection and attention as one library call
    (hs_score_select_attend, a single launch where the geometry allows).
    early_summaries: this layer's summaries are never written by the kernel
    launched just before its step (e.g. layers stepped in turn), so the
    single-launch step may start reading them early (HS_ATTN_EARLY_SUMMARIES).
    ranges: balanced chunk ranges of the tensor-core attention (True = always
    where they apply, False = never, None = the library's cost estimate)."""

    def __init__(self, *, num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype, batch,
                 max_blocks, sink_tokens, window_tokens, k_scored, capacity=None, scale=None,
                 out_is_fp32=False, algo="auto", blocks_per_split=0, score_smoothing=0.0,
                 inline_merge=True, fuse_step=True, early_summaries=False, ranges=None, device="cuda"):
        self.kv_dtype = kv_dtype
        self.shape = hs.attn_shape(num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype)
        self.batch, self.max_blocks = int(batch), int(max_blocks)
        if capacity is None:
            forced = -(-sink_tokens // block_size) + ((-(-window_tokens // block_size) + 1) if window_tokens > 0 else 0)
            capacity = min(self.max_blocks, forced + k_scored)
        self.capacity = int(capacity)
        dev = torch.device(device)
        # scores smoothed across steps (weight of the previous step), NaN = no history
        self.score_history = (torch.full((batch, num_kv_heads, max_blocks), float("nan"), device=dev)
                              if score_smoothing > 0 else None)
        self.sel_params = hs.select_params(sink_tokens, window_tokens, k_scored, self.capacity, score_smoothing,
                                           self.score_history)
        # split arrival counters: the tensor-core attention merges its splits itself
        self.split_counters = (torch.zeros(batch * num_kv_heads, dtype=torch.int32, device=dev)
                               if inline_merge else None)
        self.attn_params = hs.attn_params(scale if scale is not None else 1.0 / math.sqrt(head_dim),
                                          out_is_fp32, blocks_per_split, algo, split_counters=self.split_counters,
                                          early_summaries=early_summaries, ranges=ranges)
        sdt = _SUMMARY_DTYPE[kv_dtype]
        self.smin = torch.empty((batch, num_kv_heads, max_blocks, head_dim), dtype=sdt, device=dev)
        self.smax = torch.empty_like(self.smin)
        self.sel = torch.full((batch, num_kv_heads, self.capacity), -1, dtype=torch.int32, device=dev)
        self.sel_count = torch.zeros((batch, num_kv_heads), dtype=torch.int32, device=dev)
        self.scores = torch.empty((batch, num_kv_heads, max_blocks), dtype=torch.float32, device=dev)
        # out and lse share one byte buffer (out first, 16-byte aligned), so a
        # host read of a step's results is one transfer of ``results``
        odt = torch.float32 if out_is_fp32 else torch.bfloat16
        ob = batch * num_q_heads * head_dim * (4 if out_is_fp32 else 2)
        ob16 = (ob + 15) // 16 * 16
        self.results = torch.empty((ob16 + batch * num_q_heads * 4,), dtype=torch.uint8, device=dev)
        self.out = self.results[:ob].view(odt).view(batch, num_q_heads, head_dim)
        self.lse = self.results[ob16:].view(torch.float32).view(batch, num_q_heads)
        # one workspace serves the attention alone (from its start) and the
        # combined selection + attention call
        self.fuse_step = bool(fuse_step)
        ws = max(hs.hs_workspace_bytes(self.shape, batch, self.capacity, self.attn_params),
                 hs.hs_score_select_attend_workspace_bytes(self.shape, batch, max_blocks, self.capacity,
                                                           self.attn_params))
        self.workspace = torch.empty((max(ws, 256),), dtype=torch.uint8, device=dev)

    def reset_score_history(self):
        """Forget the smoothed scores (a new sequence of decode steps)."""
        if self.score_history is not None:
            self.score_history.fill_(float("nan"))

    def build_summaries(self, kv: hs.PagedKV, first_block: int = 0, stream=None):
        hs.hs_build_block_summaries(self.shape, kv, first_block, self.smin, self.smax, stream)

    def append(self, kv: hs.PagedKV, new_k: torch.Tensor, new_v: torch.Tensor, stream=None):
        """Writes the newest token's K/V ([batch][Hkv][D]) at seq_lens - 1 and
        widens its block's summaries (the caller has advanced seq_lens)."""
        hs.hs_append_token(self.shape, kv, new_k, new_v, self.smin, self.smax, stream)

    def select(self, kv: hs.PagedKV, q: torch.Tensor, keep_scores: bool = True, stream=None):
        hs.hs_score_select_topk(self.shape, kv, q, self.smin, self.smax, self.sel_params, self.sel,
                                self.sel_count, self.scores if keep_scores else None, None, stream)

    def attend(self, kv: hs.PagedKV, q: torch.Tensor, stream=None, selection=None):
        """Attention over the selected blocks: this decoder's own selection, or
        ``selection`` = another decoder whose selection is reused (a layer
        that borrows the block mask of an earlier layer, as SparDA's deep layers
        reuse the shallow layers' mask, §3.1 of its article)."""
        src = self if selection is None else selection
        if src.capacity != self.capacity:
            raise ValueError("a reused selection must have the same capacity")
        hs.hs_sparse_paged_decode_attn(self.shape, kv, q, src.sel, src.sel_count, self.capacity,
                                       self.attn_params, self.out, self.lse, self.workspace, stream)

    def decode_step(self, kv: hs.PagedKV, q: torch.Tensor, new_k: torch.Tensor, new_v: torch.Tensor,
                    keep_scores: bool = True, stream=None):
        """append() then select_attend() as one library call: the newest
        token is appended inside the single step launch where the shapes allow
        it."""
        hs.hs_decode_step(self.shape, kv, q, new_k, new_v, self.smin, self.smax, self.sel_params, self.sel,
                          self.sel_count, self.scores if keep_scores else None, self.attn_params, self.out, self.lse,
                          self.workspace, stream)

    def decode_step_reuse(self, kv: hs.PagedKV, q: torch.Tensor, new_k: torch.Tensor, new_v: torch.Tensor,
                          selection, stream=None):
        """append() then attend(selection=...) as one library call: a layer
        that reuses another layer's selection runs as the single step launch
        without its scoring and selection where the shapes allow it."""
        if selection.capacity != self.capacity:
            raise ValueError("a reused selection must have the same capacity")
        hs.hs_decode_step_reuse(self.shape, kv, q, new_k, new_v, self.smin, self.smax, selection.sel,
                                selection.sel_count, self.capacity, self.attn_params, self.out, self.lse,
                                self.workspace, stream)

    def select_attend(self, kv: hs.PagedKV, q: torch.Tensor, keep_scores: bool = True, stream=None):
        """select() then attend() as one library call (a single launch where
        the shapes allow it)."""
        hs.hs_score_select_attend(self.shape, kv, q, self.smin, self.smax, self.sel_params, self.sel,
                                  self.sel_count, self.scores if keep_scores else None, self.attn_params,
                                  self.out, self.lse, self.workspace, stream)

    def swap_in(self, hb: hs.HotBuffer, step: int, stats=None, stream=None):
        hs.hs_swapin_misses(self.shape, hb, self.sel, self.sel_count, self.capacity, step, stats, stream)

    def enable_swap_overlap(self, copy_ctas: int = 12, attn_ctas: int = 0):
        """Allocates what the overlapped swap-in step needs: hit and miss lists,
        two fp32 partial results, a side stream for the page copy.  The copy
        kernel runs ``copy_ctas`` CTAs, each on an SM of its own; the attention
        over the hits runs at most ``attn_ctas`` CTAs (0 = the SMs the copy
        leaves).  The copy kernel also computes the attention over the blocks
        it brings in."""
        dev = self.sel.device
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        if not 0 < copy_ctas < sms or attn_ctas < 0:
            raise ValueError(f"copy_ctas must be in [1, {sms - 1}], attn_ctas >= 0")
        self.copy_ctas = int(copy_ctas)
        attn_ctas = int(attn_ctas) if attn_ctas > 0 else sms - self.copy_ctas
        self.hit_sel = torch.full_like(self.sel, -1)
        self.miss_sel = torch.full_like(self.sel, -1)
        self.hit_count = torch.zeros_like(self.sel_count)
        self.miss_count = torch.zeros_like(self.sel_count)
        b, hq, d = self.out.shape
        self.part_out = torch.empty((2, b, hq, d), dtype=torch.float32, device=dev)
        self.part_lse = torch.empty((2, b, hq), dtype=torch.float32, device=dev)
        p = self.attn_params
        # (with the split counters the attention over the hits can cut its
        # work into balanced chunk ranges over the CTAs it is given)
        self.hit_params = hs.attn_params(p.scale, True, p.blocks_per_split, p.algo, max_ctas=attn_ctas,
                                         split_counters=self.split_counters)
        ws = hs.hs_workspace_bytes(self.shape, self.batch, self.capacity, self.hit_params)
        if ws > self.workspace.numel():
            self.workspace = torch.empty((ws,), dtype=torch.uint8, device=dev)
        self.side_stream = torch.cuda.Stream(device=dev)

    def swap_in_overlapped(self, hb: hs.HotBuffer, slot_kv: hs.PagedKV, q: torch.Tensor, step: int,
                           stats=None, stream=None, planned=False):
        """Swap-in and attention with the page copy overlapped: plan (hit and
        miss lists; already made when ``planned``) -> [side stream: copy the
        missed pages and attend over them] | attention over the hits -> LSE
        merge of the two parts into ``out``/``lse``.  Needs
        enable_swap_overlap() first."""
        main = stream if stream is not None else torch.cuda.current_stream(self.sel.device)
        if not planned:
            hs.hs_swapin_plan(self.shape, hb, self.sel, self.sel_count, self.capacity, step, self.hit_sel,
                              self.hit_count, self.miss_sel, self.miss_count, stats, main)
        side = self.side_stream
        side.wait_stream(main)
        hs.hs_swapin_copy_attend(self.shape, hb, slot_kv.seq_lens, q, self.miss_sel, self.miss_count, self.capacity,
                                 self.attn_params.scale, self.part_out[1], self.part_lse[1], self.copy_ctas, stats,
                                 side)
        hs.hs_sparse_paged_decode_attn(self.shape, slot_kv, q, self.hit_sel, self.hit_count, self.capacity,
                                       self.hit_params, self.part_out[0], self.part_lse[0], self.workspace, main)
        main.wait_stream(side)
        hs.hs_merge_attn_partials(self.shape, self.part_out, self.part_lse, self.out, self.lse, main)

    def step(self, kv: hs.PagedKV, q: torch.Tensor, refresh_from_block: int | None = None,
             hot: tuple | None = None, new_kv: tuple | None = None, reuse=None, stream=None):
        """One decode step.  ``new_kv``: (new_k, new_v) of the token at
        seq_lens - 1, appended to the cache with its summary widened before
        selecting.  ``refresh_from_block``: instead rebuild summaries of blocks
        from there on (the block holding the newest token) before selecting.
        ``hot``: (hot_buffer, slot_kv_view, step, stats) for the offload path:
        the selection is made against ``kv`` (summaries), pages are swapped into
        the hot slots and attention reads ``slot_kv_view`` (with the page copy
        overlapped once enable_swap_overlap() was called).  ``reuse``: skip
        the scoring and selection and attend over the selection of ``reuse``
        (another decoder, or ``self`` to keep this decoder's previous one)."""
        if new_kv is not None and hot is None and reuse is None and refresh_from_block is None and self.fuse_step:
            # append, selection and attention in one library call (one launch where it fuses)
            hs.hs_decode_step(self.shape, kv, q, new_kv[0], new_kv[1], self.smin, self.smax, self.sel_params,
                              self.sel, self.sel_count, self.scores, self.attn_params, self.out, self.lse,
                              self.workspace, stream)
            return self.out, self.lse
        if new_kv is not None and hot is None and reuse is not None and refresh_from_block is None and self.fuse_step:
            # append and attention over the reused selection in one library call
            self.decode_step_reuse(kv, q, new_kv[0], new_kv[1], reuse, stream)
            return self.out, self.lse
        if new_kv is not None:
            self.append(kv, new_kv[0], new_kv[1], stream)
        if refresh_from_block is not None:
            self.build_summaries(kv, refresh_from_block, stream)
        if reuse is not None:
            if hot is not None:
                raise ValueError("the offload path selects every step")
            self.attend(kv, q, stream, selection=reuse)
            return self.out, self.lse
        if hot is None and self.fuse_step:
            self.select_attend(kv, q, stream=stream)
            return self.out, self.lse
        if hot is not None and getattr(self, "side_stream", None) is not None:
            # selection and the swap-in plan (one launch where it fits), then the overlapped copy
            hb, slot_kv, step_idx, stats = hot
            hs.hs_score_select_swapin_plan(self.shape, kv, q, self.smin, self.smax, self.sel_params, self.sel,
                                           self.sel_count, hb, step_idx, self.hit_sel, self.hit_count,
                                           self.miss_sel, self.miss_count, scores=self.scores, stats=stats,
                                           stream=stream)
            self.swap_in_overlapped(hb, slot_kv, q, step_idx, stats, stream, planned=True)
            return self.out, self.lse
        self.select(kv, q, stream=stream)
        if hot is not None:
            hb, slot_kv, step_idx, stats = hot
            if getattr(self, "side_stream", None) is not None:
                self.swap_in_overlapped(hb, slot_kv, q, step_idx, stats, stream)
            else:
                self.swap_in(hb, step_idx, stats, stream)
                self.attend(slot_kv, q, stream)
        else:
            self.attend(kv, q, stream)
        return self.out, self.lse
