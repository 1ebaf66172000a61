"""One indexer step on one GPU: the six C-ABI calls chained over device-resident
buffers.

Order of a step (the new tokens' caches are written before anything reads them):
  1. ix_quant_write_k     new tokens' indexer K -> paged indexer-K cache
  2. dsmla_quant_write    new tokens' NoPE/RoPE -> fp8_ds_mla cache
  3. ix_gather_k          prefill requests' paged K -> contiguous K + scales
  4. ix_mqa_logits        prefill rows' logits over the gathered K
  5. ix_paged_mqa_logits  decode rows' logits over the paged cache
  6. ix_topk_to_global    top-k + remap, once for the decode rows and once for the
                          prefill rows (they live in logits buffers of different ld)

``fused`` names the parts ("decode", "prefill"; True = both) whose logits call
and top-k run as one call (ix_paged_mqa_logits_topk, ix_mqa_logits_topk): the
logits kernel also builds each row's first-digit histogram and the selection
starts from it.  Each fused call keeps a histogram workspace of its own,
zeroed once here.

All buffers are allocated once here (torch, on the device); ``run`` allocates
nothing and never synchronises, so it can be captured in a CUDA graph.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import (BLOCK_SIZE, DSMLA_ENTRY_BYTES, HEAD_DIM, HEADS, INDEXER_BLOCK_BYTES,
               dsmla_quant_write, ix_gather_k, ix_mqa_logits, ix_mqa_logits_hist, ix_mqa_logits_topk,
               ix_paged_mqa_logits, ix_paged_mqa_logits_hist, ix_paged_mqa_logits_topk,
               ix_quant_write_k, ix_topk_from_hist, ix_topk_hist_workspace_size, ix_topk_to_global)


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclass
class DecodePart:
    context_lens: torch.Tensor   # int32 [B]
    q: torch.Tensor              # uint8/e4m3 [B, next_n, 64, 128]
    w: torch.Tensor              # f32 [B*next_n, 64]
    row_len: torch.Tensor        # int32 [B*next_n]
    row_req: torch.Tensor        # int32 [B*next_n] (rows of block_table)
    ld: int                      # logits row stride (>= longest row, multiple of 4)


@dataclass
class PrefillPart:
    req: list                    # request ids (rows of block_table)
    cu_seq_lens: torch.Tensor    # int32 [C+1] over the requests' whole contexts
    ks: torch.Tensor             # int32 [T]
    ke: torch.Tensor             # int32 [T]
    row_len: torch.Tensor        # int32 [T]
    row_req: torch.Tensor        # int32 [T]
    q: torch.Tensor              # uint8/e4m3 [T, 64, 128]
    w: torch.Tensor              # f32 [T, 64]
    gathered: int                # cu_seq_lens[-1] (host copy, sizes the gather buffers)
    ld: int


class IndexerStep:
    def __init__(self, *, num_blocks: int, block_table: torch.Tensor, topk: int,
                 new_k: torch.Tensor, new_slot: torch.Tensor,
                 decode: Optional[DecodePart] = None, prefill: Optional[PrefillPart] = None,
                 nope: Optional[torch.Tensor] = None, rope: Optional[torch.Tensor] = None,
                 clean_logits: bool = False, with_local: bool = False, fused=False):
        if fused is True:
            fused = ("decode", "prefill")
        fused = set(fused or ())
        if fused and clean_logits:
            raise ValueError("the fused calls leave the logits past each row's end untouched (no clean_logits)")
        dev = block_table.device
        self.num_blocks = num_blocks
        self.block_table = block_table
        self.topk = topk
        self.new_k = new_k
        self.new_slot = new_slot
        self.decode = decode
        self.prefill = prefill
        self.nope = nope
        self.rope = rope
        self.clean = clean_logits
        self.fused_dec = "decode" in fused
        self.fused_pf = "prefill" in fused
        self._graph = None
        self.cache = torch.zeros(num_blocks, INDEXER_BLOCK_BYTES, dtype=torch.uint8, device=dev)
        self.dsmla_cache = None
        if nope is not None:
            self.dsmla_cache = torch.zeros(num_blocks, BLOCK_SIZE, DSMLA_ENTRY_BYTES,
                                           dtype=torch.uint8, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        if decode is not None:
            R = decode.w.shape[0]
            self.dec_logits = torch.empty(R, decode.ld, dtype=torch.float32, device=dev)
            self.dec_global = torch.empty(R, topk, **i32)
            self.dec_local = torch.empty(R, topk, **i32) if with_local else None
            self.dec_ws = (torch.zeros(ix_topk_hist_workspace_size(R), dtype=torch.uint8, device=dev)
                           if self.fused_dec else None)
        if prefill is not None:
            T = prefill.w.shape[0]
            self.k_fp8 = torch.empty(max(prefill.gathered, 1), HEAD_DIM, dtype=torch.uint8,
                                     device=dev)
            self.k_scale = torch.empty(max(prefill.gathered, 1), dtype=torch.float32, device=dev)
            self.pf_bt = block_table[prefill.req]
            self.pf_logits = torch.empty(T, prefill.ld, dtype=torch.float32, device=dev)
            self.pf_global = torch.empty(T, topk, **i32)
            self.pf_local = torch.empty(T, topk, **i32) if with_local else None
            self.pf_ws = (torch.zeros(ix_topk_hist_workspace_size(T), dtype=torch.uint8, device=dev)
                          if self.fused_pf else None)

    def graph(self) -> "torch.cuda.CUDAGraph":
        """The step as one CUDA graph (captured on first use, on a side stream,
        after at least one eager run() has done the library's one-time set-up):
        replaying it issues the same kernels as run() with less launch overhead.
        The graph reads and writes this step's buffers in place."""
        if self._graph is None:
            dev = self.block_table.device
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    self.run(stream=side)
            torch.cuda.current_stream(dev).wait_stream(side)
            self._graph = g
        return self._graph

    def write_history(self, k_bf16: torch.Tensor, slots: torch.Tensor, chunk: int = 1 << 20):
        """Fill the indexer-K cache with already-cached positions (set-up, not a step)."""
        for i in range(0, k_bf16.shape[0], chunk):
            ix_quant_write_k(k_bf16[i:i + chunk], slots[i:i + chunk], self.cache)

    def kernels_per_step(self) -> int:
        """Kernel launches of one step (a fused call launches two kernels, as
        does the unfused pair)."""
        n = 1 + (self.nope is not None)
        if self.prefill is not None:
            n += 3 + (1 if self.clean else 0)
        if self.decode is not None:
            n += 2 + (1 if self.clean else 0)
        return n

    def run(self, stream=None, events=None, split: bool = False):
        """One step.  ``events``: optional dict name -> (start, end) CUDA events
        recorded around the logits and top-k launches on ``stream``.  With
        ``split`` a fused step issues each fused call as its two halves (the
        same kernels, in the same order), so events can bracket each kernel.

        Order: cache writes, then the decode pair (paged logits streaming the
        cache, top-k), then the prefill pair (gather, logits, top-k).  The
        prefill logits leave L2 full of freshly written rows; run right after
        them, the HBM-bound decode pass would pay for writing those lines back,
        while the prefill top-k reads them where they are."""
        s = stream

        def timed(name, fn):
            if events and name in events:
                events[name][0].record(s)
            fn()
            if events and name in events:
                events[name][1].record(s)

        ix_quant_write_k(self.new_k, self.new_slot, self.cache, stream=s)
        if self.nope is not None:
            dsmla_quant_write(self.nope, self.rope, self.new_slot, self.dsmla_cache, stream=s)
        if self.decode is not None:
            d = self.decode
            if self.fused_dec and not split:
                timed("paged_mqa_logits_topk", lambda: ix_paged_mqa_logits_topk(
                    d.q, d.w, self.cache, d.context_lens, self.block_table, self.dec_logits, self.topk,
                    self.dec_global, self.dec_ws, out_local=self.dec_local, stream=s))
            elif self.fused_dec:
                timed("paged_mqa_logits", lambda: ix_paged_mqa_logits_hist(
                    d.q, d.w, self.cache, d.context_lens, self.block_table, self.dec_logits, self.topk,
                    self.dec_ws, stream=s))
                timed("topk_decode", lambda: ix_topk_from_hist(
                    self.dec_logits, d.row_len, d.row_req, self.block_table, self.topk, self.dec_global,
                    self.dec_ws, out_local=self.dec_local, stream=s))
            else:
                timed("paged_mqa_logits", lambda: ix_paged_mqa_logits(
                    d.q, d.w, self.cache, d.context_lens, self.block_table, self.dec_logits,
                    clean_logits=self.clean, stream=s))
                timed("topk_decode", lambda: ix_topk_to_global(
                    self.dec_logits, d.row_len, d.row_req, self.block_table, self.topk,
                    self.dec_global, self.dec_local, stream=s))
        if self.prefill is not None:
            p = self.prefill
            ix_gather_k(self.cache, self.pf_bt, p.cu_seq_lens, self.k_fp8, self.k_scale, stream=s)
            if self.fused_pf and not split:
                timed("mqa_logits_topk", lambda: ix_mqa_logits_topk(
                    p.q, p.w, self.k_fp8, self.k_scale, p.ks, p.ke, self.pf_logits, p.row_req,
                    self.block_table, self.topk, self.pf_global, self.pf_ws, out_local=self.pf_local,
                    stream=s))
            elif self.fused_pf:
                timed("mqa_logits", lambda: ix_mqa_logits_hist(
                    p.q, p.w, self.k_fp8, self.k_scale, p.ks, p.ke, self.pf_logits, self.topk, self.pf_ws,
                    stream=s))
                timed("topk_prefill", lambda: ix_topk_from_hist(
                    self.pf_logits, p.row_len, p.row_req, self.block_table, self.topk, self.pf_global,
                    self.pf_ws, out_local=self.pf_local, stream=s))
            else:
                timed("mqa_logits", lambda: ix_mqa_logits(
                    p.q, p.w, self.k_fp8, self.k_scale, p.ks, p.ke, self.pf_logits,
                    clean_logits=self.clean, stream=s))
                timed("topk_prefill", lambda: ix_topk_to_global(
                    self.pf_logits, p.row_len, p.row_req, self.block_table, self.topk,
                    self.pf_global, self.pf_local, stream=s))
