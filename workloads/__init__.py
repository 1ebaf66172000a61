"""Seeded synthetic inputs for the DeepSeek-V3.2 indexer hot path.

This module only draws random inputs; it holds none of the method's arithmetic
(no quantisation of K, no scores, no selection).  Both the CUDA path and the
CPU oracle consume what it returns, each through its own code.

One ``torch.Generator`` (CPU, seed 0 unless stated) is drawn in a fixed order:
lengths -> block tables -> K -> q -> w -> fp8_ds_mla inputs.

* K of every cached position: N(0,1) f32 rounded to bf16 (per token, 128 dims).
* q: N(0,1) f32 cast to float8 e4m3 (64 heads x 128 dims per query token).
* w: N(0,1)/8 in f32, one weight per (query token, head).
* Block tables: one ``randperm`` of the block pool, sliced per request in
  request order (decode requests first, then prefill requests).
* fp8_ds_mla inputs: NoPE N(0,1) with each element scaled by 20 with
  probability 0.001 (Bernoulli from the same generator), RoPE N(0,1), both bf16.

The named workloads follow the indexer configurations: a tiny decode batch,
batch-32 decode, next_n=2 MTP decode, an 8192-token causal prefill chunk, and a
long-context mixed batch.  The pages' own workload is a random-token serving
benchmark; these synthetic inputs stand in for it (no dataset is used).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

HEADS = 64
HEAD_DIM = 128
BLOCK_SIZE = 64
NOPE_DIM = 512
ROPE_DIM = 64


@dataclass
class Workload:
    name: str
    block_size: int
    heads: int
    head_dim: int
    topk: int
    num_blocks: int
    # per request (decode requests first, then prefill requests)
    req_ctx: np.ndarray            # int64 [R] cached positions per request
    block_table: np.ndarray        # int32 [R, max_blocks]
    # every cached position of every request, request-major
    k_bf16: torch.Tensor           # bfloat16 [Ntot, head_dim]
    slot: np.ndarray               # int64 [Ntot]
    is_new: np.ndarray             # bool [Ntot]: written during the step
    # decode part
    n_decode: int = 0
    next_n: int = 1
    context_lens: Optional[np.ndarray] = None   # int32 [n_decode]
    q_decode: Optional[torch.Tensor] = None     # uint8 [n_decode, next_n, H, D] (e4m3 bits)
    w_decode: Optional[torch.Tensor] = None     # f32 [n_decode*next_n, H]
    # prefill part (each chunk = the last chunk_len positions of its request)
    prefill_req: List[int] = field(default_factory=list)   # request ids
    chunk_len: List[int] = field(default_factory=list)
    q_prefill: Optional[torch.Tensor] = None    # uint8 [T, H, D]
    w_prefill: Optional[torch.Tensor] = None    # f32 [T, H]
    # fp8_ds_mla inputs for the new tokens (same order as k_bf16[is_new])
    nope_bf16: Optional[torch.Tensor] = None    # bfloat16 [Nnew, 512]
    rope_bf16: Optional[torch.Tensor] = None    # bfloat16 [Nnew, 64]

    # ---- derived views (index bookkeeping only) ----
    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def new_slot(self) -> np.ndarray:
        return self.slot[self.is_new]

    @property
    def new_k(self) -> torch.Tensor:
        return self.k_bf16[torch.from_numpy(self.is_new)]

    @property
    def hist_slot(self) -> np.ndarray:
        return self.slot[~self.is_new]

    @property
    def hist_k(self) -> torch.Tensor:
        return self.k_bf16[torch.from_numpy(~self.is_new)]

    def new_positions(self) -> np.ndarray:
        """int64 [n_new]: each new token's position in its request (cached order)."""
        pos = np.concatenate([np.arange(int(c), dtype=np.int64) for c in self.req_ctx])
        return pos[self.is_new]

    def decode_rows(self):
        """(row_len int32 [B*next_n], row_req int32 [B*next_n]) for decode rows."""
        B, n = self.n_decode, self.next_n
        j = np.tile(np.arange(n), B)
        b = np.repeat(np.arange(B), n)
        L = self.context_lens.astype(np.int64)[b] - n + 1 + j
        return np.maximum(L, 0).astype(np.int32), b.astype(np.int32)

    @property
    def n_prefill_rows(self) -> int:
        return int(sum(self.chunk_len))

    def prefill_gather(self):
        """cu_seq_lens int32 [C+1] over the prefill requests' whole contexts."""
        lens = [int(self.req_ctx[r]) for r in self.prefill_req]
        return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)

    def prefill_rows(self):
        """(ks, ke, row_len, row_req) int32 [T] for prefill rows over the
        gathered contiguous K: row i of chunk c sits at request position
        p = ctx - chunk_len + i and sees request keys 0..p."""
        cu = self.prefill_gather()
        ks, ke, rl, rq = [], [], [], []
        for c, (r, n) in enumerate(zip(self.prefill_req, self.chunk_len)):
            ctx = int(self.req_ctx[r])
            p = np.arange(ctx - n, ctx)
            ks.append(np.full(n, cu[c]))
            ke.append(cu[c] + p + 1)
            rl.append(p + 1)
            rq.append(np.full(n, r))
        cat = lambda xs: np.concatenate(xs).astype(np.int32)
        return cat(ks), cat(ke), cat(rl), cat(rq)

    def prefill_block_table(self) -> np.ndarray:
        return self.block_table[self.prefill_req]


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _fp8_bits(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def build(name: str, *, decode_ctx=(), next_n: int = 1, prefill=(), topk: int = 2048,
          seed: int = 0, pool_blocks: Optional[int] = None, blocks_per_req=None,
          lengths_fn=None, dsmla: bool = False, heads: int = HEADS,
          head_dim: int = HEAD_DIM, block_size: int = BLOCK_SIZE) -> Workload:
    """Generic generator.

    decode_ctx: cached positions per decode request (the last next_n of them
      are the step's new tokens), or None when ``lengths_fn`` draws them.
    prefill: list of (context, chunk_len); the last chunk_len positions are new.
    pool_blocks: block pool size (default: exactly what the requests need).
    blocks_per_req: blocks handed to each request from the permutation (default:
      ceil(ctx/bs)).
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    # 1. lengths
    if lengths_fn is not None:
        decode_ctx = [int(v) for v in lengths_fn(g)]
    decode_ctx = [int(v) for v in decode_ctx]
    prefill = [(int(c), int(n)) for c, n in prefill]
    req_ctx = np.array(decode_ctx + [c for c, _ in prefill], dtype=np.int64)
    R = len(req_ctx)
    need = [(int(c) + block_size - 1) // block_size for c in req_ctx]
    if blocks_per_req is None:
        give = need
    else:
        give = [int(blocks_per_req)] * R
        assert all(gv >= nd for gv, nd in zip(give, need))
    pool = int(pool_blocks) if pool_blocks is not None else int(sum(give))
    assert pool >= sum(give)
    # 2. block tables
    perm = torch.randperm(pool, generator=g).numpy().astype(np.int32)
    max_blocks = max(give) if give else 1
    bt = np.zeros((R, max_blocks), dtype=np.int32)
    o = 0
    for r in range(R):
        bt[r, :give[r]] = perm[o:o + give[r]]
        o += give[r]
    # 3. K for every cached position (request-major), bf16
    k_parts, slot_parts, new_parts = [], [], []
    for r in range(R):
        ctx = int(req_ctx[r])
        k_parts.append(_bf16(torch.randn(ctx, head_dim, generator=g)))
        p = np.arange(ctx, dtype=np.int64)
        slot_parts.append(bt[r, p // block_size].astype(np.int64) * block_size + p % block_size)
        n_new = next_n if r < len(decode_ctx) else prefill[r - len(decode_ctx)][1]
        nm = np.zeros(ctx, dtype=bool)
        nm[max(ctx - n_new, 0):] = True
        new_parts.append(nm)
    k_bf16 = torch.cat(k_parts) if k_parts else torch.zeros(0, head_dim, dtype=torch.bfloat16)
    slot = np.concatenate(slot_parts) if slot_parts else np.zeros(0, np.int64)
    is_new = np.concatenate(new_parts) if new_parts else np.zeros(0, bool)
    wl = Workload(name=name, block_size=block_size, heads=heads, head_dim=head_dim, topk=topk,
                  num_blocks=pool, req_ctx=req_ctx, block_table=bt, k_bf16=k_bf16, slot=slot,
                  is_new=is_new)
    B = len(decode_ctx)
    T = sum(n for _, n in prefill)
    # 4. q
    if B:
        wl.n_decode, wl.next_n = B, next_n
        wl.context_lens = np.array(decode_ctx, dtype=np.int32)
        wl.q_decode = _fp8_bits(torch.randn(B, next_n, heads, head_dim, generator=g))
    if T:
        wl.prefill_req = list(range(B, R))
        wl.chunk_len = [n for _, n in prefill]
        wl.q_prefill = _fp8_bits(torch.randn(T, heads, head_dim, generator=g))
    # 5. w
    if B:
        wl.w_decode = torch.randn(B * next_n, heads, generator=g) / 8
    if T:
        wl.w_prefill = torch.randn(T, heads, generator=g) / 8
    # 6. fp8_ds_mla inputs for the new tokens
    if dsmla:
        n_new = int(is_new.sum())
        nope = torch.randn(n_new, NOPE_DIM, generator=g)
        outlier = torch.rand(n_new, NOPE_DIM, generator=g) < 0.001
        nope = torch.where(outlier, nope * 20, nope)
        wl.nope_bf16 = _bf16(nope)
        wl.rope_bf16 = _bf16(torch.randn(n_new, ROPE_DIM, generator=g))
    return wl


# ---------------------------------------------------------------------------
# Named workloads
# ---------------------------------------------------------------------------

def tiny_decode(seed: int = 0) -> Workload:
    """Batch 2, one query token each, contexts [37, 300]; a pool of 16 blocks
    in one permutation, 8 blocks to each request; top_k 64."""
    return build("tiny_decode_b2", decode_ctx=[37, 300], next_n=1, topk=64, seed=seed,
                 pool_blocks=16, blocks_per_req=8)


def decode_b32(seed: int = 0) -> Workload:
    """Batch 32, one query token each, contexts uniform in [1024, 8192], pool of
    8192 blocks; top_k 2048."""
    return build("decode_b32_ctx1k-8k", next_n=1, topk=2048, seed=seed, pool_blocks=8192,
                 lengths_fn=lambda g: torch.randint(1024, 8193, (32,), generator=g).tolist())


def decode_mtp2_b128(seed: int = 0) -> Workload:
    """Batch 128, next_n = 2; context log-uniform in [4096, 32768]; the second
    query token sees ctx + 1 keys, so context_lens = ctx + 1; top_k 2048."""
    def lengths(g):
        u = torch.rand(128, generator=g, dtype=torch.float64)
        ctx = torch.floor(torch.exp(math.log(4096) + u * (math.log(32768) - math.log(4096))))
        return (ctx.to(torch.int64) + 1).tolist()
    return build("decode_mtp2_b128_ctx4k-32k", next_n=2, topk=2048, seed=seed,
                 lengths_fn=lengths)


def prefill_8k(seed: int = 0) -> Workload:
    """One request, 8192 new tokens, causal (token t sees keys 0..t); top_k 2048."""
    return build("prefill_causal_8192", prefill=[(8192, 8192)], topk=2048, seed=seed)


def mixed_long(seed: int = 0) -> Workload:
    """16 decode requests at context 131072 plus 4 prefill chunks of 2048 tokens
    (the last 2048 positions of 8192-token contexts); fp8_ds_mla inputs for all
    8208 new tokens; top_k 2048."""
    return build("mixed_16x131072dec_4x2048pf", decode_ctx=[131072] * 16, next_n=1,
                 prefill=[(8192, 2048)] * 4, topk=2048, seed=seed, dsmla=True)


NAMED = {
    "tiny_decode": tiny_decode,
    "decode_b32": decode_b32,
    "decode_mtp2_b128": decode_mtp2_b128,
    "prefill_8k": prefill_8k,
    "mixed_long": mixed_long,
}


# ---------------------------------------------------------------------------
# numpy views for the oracle side
# ---------------------------------------------------------------------------

def norm_rope_params(max_pos: int, seed: int = 0):
    """Synthetic parameters of the fused RMSNorm + RoPE cache write, from a
    generator of their own (the draws above are unchanged):
    norm weights bf16 [512] drawn as 1 + N(0,1)/8, and a rotary table f32
    [max_pos, 64] holding the cosines (columns 0-31) and sines (32-63) of angles
    drawn uniformly in [0, 2 pi) -- a valid rotation for every (position, pair),
    not a particular frequency schedule."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7919)
    gamma = _bf16(1 + torch.randn(NOPE_DIM, generator=g) / 8)
    ang = torch.rand(max_pos, ROPE_DIM // 2, generator=g, dtype=torch.float64) * (2 * math.pi)
    table = torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32)
    return gamma, table


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """bfloat16 tensor -> uint16 numpy array of its bit patterns."""
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().numpy()


@dataclass
class SparseDecodeInputs:
    """Inputs of one sparse MLA decode call (attention over the fp8_ds_mla cache).

    The cache entries come from ``nope_bf16`` / ``rope_bf16`` written at
    ``slots``; ``indices`` [tokens, topk] names, per token, distinct slots drawn
    from its own context (the shape of a top-k row), padded with -1 when the
    context is shorter than topk."""
    q_nope: torch.Tensor  # bf16 [T, 128, 512]
    q_pe: torch.Tensor  # bf16 [T, 128, 64]
    nope_bf16: torch.Tensor  # bf16 [n, 512]: values written into the cache
    rope_bf16: torch.Tensor  # bf16 [n, 64]
    slots: np.ndarray  # int64 [n]: where entry i is written
    indices: np.ndarray  # int32 [T, topk]
    num_blocks: int
    sm_scale: float


MLA_HEADS = 128


def sparse_decode_inputs(tokens: int, topk: int, ctx: int, *, seed: int = 0, q_scale: float = 1.0,
                         block_size: int = BLOCK_SIZE) -> SparseDecodeInputs:
    """Token t attends over a context of ``ctx`` cached positions held in its
    own random blocks; its index row takes min(topk, ctx) distinct positions of
    that context (uniform without replacement, in random order) and pads with
    -1.  Only the selected positions are written into the cache.  q: N(0,1) *
    q_scale in bf16; cache values drawn like the fp8_ds_mla inputs above;
    sm_scale = 1/sqrt(192) (the 128 + 64 query-key head width of DeepSeek-V3)."""
    g = torch.Generator().manual_seed(seed)
    blocks_per_ctx = -(-ctx // block_size)
    num_blocks = tokens * blocks_per_ctx
    perm = torch.randperm(num_blocks, generator=g).numpy()
    q_nope = _bf16(torch.randn(tokens, MLA_HEADS, NOPE_DIM, generator=g) * q_scale)
    q_pe = _bf16(torch.randn(tokens, MLA_HEADS, ROPE_DIM, generator=g) * q_scale)
    take = min(topk, ctx)
    indices = np.full((tokens, topk), -1, np.int32)
    slots = []
    for t in range(tokens):
        pos = torch.randperm(ctx, generator=g)[:take].numpy()
        table = perm[t * blocks_per_ctx:(t + 1) * blocks_per_ctx]
        gl = table[pos // block_size].astype(np.int64) * block_size + pos % block_size
        indices[t, :take] = gl
        slots.append(gl)
    slots = np.concatenate(slots) if slots else np.zeros(0, np.int64)
    n = slots.shape[0]
    nope = torch.randn(n, NOPE_DIM, generator=g)
    out = torch.rand(n, NOPE_DIM, generator=g) < 0.001
    nope = _bf16(torch.where(out, nope * 20, nope))
    rope = _bf16(torch.randn(n, ROPE_DIM, generator=g))
    return SparseDecodeInputs(q_nope, q_pe, nope, rope, slots.astype(np.int64), indices, num_blocks,
                              1.0 / math.sqrt(192.0))


@dataclass
class QueryInputs:
    """Inputs of the query side of a step for `tokens` query tokens: the MLA
    query pair before RoPE (ql_nope, q_pe; 128 heads) and the indexer's bf16
    query and head weights (64 heads x 128).  Drawn like the cache inputs:
    N(0,1) with each element scaled by 20 with probability 0.001, in bf16;
    weights N(0,1)/8 in f32."""
    ql_nope: torch.Tensor   # bf16 [T, 128, 512]
    q_pe: torch.Tensor      # bf16 [T, 128, 64]
    index_q: torch.Tensor   # bf16 [T, 64, 128]
    index_w: torch.Tensor   # f32 [T, 64]


def query_inputs(tokens: int, seed: int = 0) -> QueryInputs:
    g = torch.Generator().manual_seed(seed + 104729)

    def draw(*shape):
        x = torch.randn(*shape, generator=g)
        out = torch.rand(*shape, generator=g) < 0.001
        return _bf16(torch.where(out, x * 20, x))

    qn = draw(tokens, MLA_HEADS, NOPE_DIM)
    qp = draw(tokens, MLA_HEADS, ROPE_DIM)
    iq = draw(tokens, HEADS, HEAD_DIM)
    iw = torch.randn(tokens, HEADS, generator=g) / 8
    return QueryInputs(qn, qp, iq, iw)
