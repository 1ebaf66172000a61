"""Move a synthetic ``Workload`` onto the GPU as an ``IndexerStep``.

Bookkeeping only (copies and index arrays); the method's arithmetic happens in
the CUDA library.  Kept apart from ``workloads/__init__.py`` so that the input
generator itself never imports the product package.
"""
from __future__ import annotations

import numpy as np
import torch

from . import Workload


def _ld(max_len: int) -> int:
    return max(4, (int(max_len) + 3) // 4 * 4)


def make_step(wl: Workload, device="cuda", clean: bool = False, with_local: bool = False,
              write_history: bool = True, fused=False):
    from deepseek_v3_sparse_gb300.step import DecodePart, IndexerStep, PrefillPart

    dev = torch.device(device)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    bt = i32(wl.block_table)
    decode = prefill = None
    if wl.n_decode:
        rl, rq = wl.decode_rows()
        decode = DecodePart(context_lens=i32(wl.context_lens), q=wl.q_decode.to(dev),
                            w=wl.w_decode.to(dev), row_len=i32(rl), row_req=i32(rq),
                            ld=_ld(rl.max()))
    if wl.prefill_req:
        ks, ke, rl, rq = wl.prefill_rows()
        cu = wl.prefill_gather()
        prefill = PrefillPart(req=list(wl.prefill_req), cu_seq_lens=i32(cu), ks=i32(ks),
                              ke=i32(ke), row_len=i32(rl), row_req=i32(rq),
                              q=wl.q_prefill.to(dev), w=wl.w_prefill.to(dev),
                              gathered=int(cu[-1]), ld=_ld(rl.max()))
    step = IndexerStep(num_blocks=wl.num_blocks, block_table=bt, topk=wl.topk,
                       new_k=wl.new_k.to(dev),
                       new_slot=torch.from_numpy(wl.new_slot.copy()).to(dev),
                       decode=decode, prefill=prefill,
                       nope=None if wl.nope_bf16 is None else wl.nope_bf16.to(dev),
                       rope=None if wl.rope_bf16 is None else wl.rope_bf16.to(dev),
                       clean_logits=clean, with_local=with_local, fused=fused)
    if write_history and (~wl.is_new).any():
        step.write_history(wl.hist_k.to(dev), torch.from_numpy(wl.hist_slot.copy()).to(dev))
    return step
