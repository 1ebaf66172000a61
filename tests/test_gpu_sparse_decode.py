"""GPU parity: sparse MLA decode over the fp8_ds_mla cache (dsmla_sparse_decode)
against the oracle on the same seeded inputs.

Tolerance, from the kernel's rounding steps (keys, values and softmax weights
rounded to bf16 -- an 8-bit significand, unit roundoff 2^-8 each -- products
accumulated in f32, output rounded to bf16): per (token, head),
    |out - out_ref| <= 2^-8 |out_ref| + 2^-7 max_j |v_j|     (elementwise)
    |lse - lse_ref| <= 2^-7 + 2^-9 |lse_ref|
where max_j |v_j| is the largest value magnitude over the keys the row names.
The first term is the output rounding; the second bounds the weight and value
roundings, whose independent errors (standard deviation about 2^-8 / sqrt(3)
relative each) move a convex combination by far less than 2^-7 of its largest
value.  The lse (returned in f32) carries the weighted mean of the score
errors plus the rounding of the sum.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import require_gpu

pytestmark = pytest.mark.gpu

IX_DEV_BAD_SLOT = 1


@pytest.fixture(scope="module")
def dsix():
    require_gpu()
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v3_sparse_gb300 as m
    m.ix_device_status()  # clear
    return m


def _cache_bytes(x, bs, entry=656, extra=0):
    """Entries written by the oracle's fp8_ds_mla writer (CPU), as flat bytes."""
    dense = np.zeros((x.num_blocks, bs, 656), np.uint8)
    oracle.dsmla_quant_write(W.bf16_bits(x.nope_bf16), W.bf16_bits(x.rope_bf16), x.slots, dense, bs)
    if entry == 656 and extra == 0:
        return dense, dense.reshape(-1), bs * 656, 656
    bstride = bs * entry + extra
    flat = np.full(x.num_blocks * bstride, 0x7F, np.uint8)   # NaN codes in the padding
    for b in range(x.num_blocks):
        for o in range(bs):
            flat[b * bstride + o * entry:b * bstride + o * entry + 656] = dense[b, o]
    return dense, flat, bstride, entry


def _run_gpu(dsix, x, flat, bs, bstride, entry, indices=None):
    idx = torch.from_numpy(np.ascontiguousarray(x.indices if indices is None else indices)).cuda()
    T, topk = idx.shape
    nb = x.num_blocks
    cache = torch.from_numpy(flat).cuda()
    out = torch.empty(T, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, 128, dtype=torch.float32, device="cuda")
    ws = torch.empty(dsix.dsmla_sparse_decode_workspace_size(T, 128, topk), dtype=torch.uint8, device="cuda")
    qn, qp = x.q_nope.cuda(), x.q_pe.cuda()   # held until the call has run
    lib = dsix.load()
    rc = lib.dsmla_sparse_decode(qn.data_ptr(), qp.data_ptr(), cache.data_ptr(), nb, bs,
                                 bstride, entry, idx.data_ptr(), T, 128, topk, x.sm_scale, out.data_ptr(),
                                 lse.data_ptr(), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0, dsix.ix_status_string(rc)
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _vmax(dense, indices, bs):
    """Per token: the largest |v| over the entries its row names (decoded with torch)."""
    flat = dense.reshape(-1, 656)
    res = np.zeros(indices.shape[0])
    for t in range(indices.shape[0]):
        sel = indices[t][indices[t] >= 0]
        if sel.size == 0:
            continue
        e = flat[sel]
        codes = torch.from_numpy(e[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64)
        sc = torch.from_numpy(e[:, 512:528].copy()).view(torch.float32).to(torch.float64)
        res[t] = float((codes * sc.repeat_interleave(128, dim=1)).abs().max())
    return res


def _compare(out, lse, ref_o, ref_l, vmax):
    tol_o = 2.0 ** -8 * np.abs(ref_o) + 2.0 ** -7 * vmax[:, None, None]
    err = np.abs(out - ref_o)
    bad = err > tol_o
    assert not bad.any(), (int(bad.sum()), float((err - tol_o).max()), np.argwhere(bad)[:5])
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(lse[~fin] == -np.inf) and np.all(out[~fin] == 0)
    tol_l = 2.0 ** -7 + 2.0 ** -9 * np.abs(ref_l[fin])
    assert np.all(np.abs(lse[fin] - ref_l[fin]) <= tol_l), float(np.max(np.abs(lse[fin] - ref_l[fin]) - tol_l))
    return float(np.max(err / np.maximum(vmax[:, None, None], 1e-30)))


def _oracle(x, dense, bs, indices=None):
    idx = x.indices if indices is None else indices
    ref_o, ref_l, ok = oracle.dsmla_sparse_decode(W.bf16_bits(x.q_nope), W.bf16_bits(x.q_pe), dense, bs,
                                                  idx, x.sm_scale)
    return ref_o, ref_l, ok


@pytest.mark.parametrize("tokens,topk,ctx,q_scale", [(3, 600, 1000, 1.0), (2, 256, 300, 1.0),
                                                      (4, 2048, 1500, 1.0), (2, 1, 50, 1.0),
                                                      (3, 512, 4096, 3.0)])
def test_sparse_decode_matches_oracle(dsix, tokens, topk, ctx, q_scale):
    x = W.sparse_decode_inputs(tokens, topk, ctx, seed=tokens * 7 + topk, q_scale=q_scale)
    dense, flat, bstride, entry = _cache_bytes(x, 64)
    out, lse = _run_gpu(dsix, x, flat, 64, bstride, entry)
    ref_o, ref_l, ok = _oracle(x, dense, 64)
    assert ok
    _compare(out, lse, ref_o, ref_l, _vmax(dense, x.indices, 64))
    assert dsix.ix_device_status() == 0


def test_sparse_decode_padding_duplicates_and_empty_rows(dsix):
    x = W.sparse_decode_inputs(4, 700, 900, seed=11)
    idx = x.indices.copy()
    idx[0, 100:400] = -1                  # a hole spanning split boundaries
    idx[1, :] = -1                        # no key at all
    idx[2, 256:512] = -1                  # one whole split without keys
    idx[3, 1::2] = idx[3, 0::2]           # every key twice
    dense, flat, bstride, entry = _cache_bytes(x, 64)
    out, lse = _run_gpu(dsix, x, flat, 64, bstride, entry, idx)
    ref_o, ref_l, ok = _oracle(x, dense, 64, idx)
    assert ok
    assert ref_l[1].max() == -np.inf
    _compare(out, lse, ref_o, ref_l, _vmax(dense, idx, 64))
    assert dsix.ix_device_status() == 0


@pytest.mark.parametrize("bs,entry,extra", [(16, 672, 32), (64, 656, 0)])
def test_sparse_decode_strided_layout_and_bad_index(dsix, bs, entry, extra):
    x = W.sparse_decode_inputs(2, 300, 600, seed=bs, block_size=bs)
    idx = x.indices.copy()
    idx[1, 5] = x.num_blocks * bs          # one past the pool: flagged, treated as none
    dense, flat, bstride, e = _cache_bytes(x, bs, entry, extra)
    out, lse = _run_gpu(dsix, x, flat, bs, bstride, e, idx)
    ref_o, ref_l, ok = _oracle(x, dense, bs, idx)
    assert not ok
    _compare(out, lse, ref_o, ref_l, _vmax(dense, np.where(idx < x.num_blocks * bs, idx, -1), bs))
    assert dsix.ix_device_status() == IX_DEV_BAD_SLOT
    assert dsix.ix_device_status() == 0


def test_sparse_decode_full_size_decode_batch(dsix):
    # 16 decode tokens x 128 heads x top-2048 over 131072-position contexts
    # (the long-context decode batch); every output compared.
    x = W.sparse_decode_inputs(16, 2048, 131072, seed=5)
    dense, flat, bstride, entry = _cache_bytes(x, 64)
    out, lse = _run_gpu(dsix, x, flat, 64, bstride, entry)
    ref_o, ref_l, ok = _oracle(x, dense, 64)
    assert ok
    worst = _compare(out, lse, ref_o, ref_l, _vmax(dense, x.indices, 64))
    print(f"worst |err| / max|v|: {worst:.3e}")
    # deterministic: a second run gives the same bits
    out2, lse2 = _run_gpu(dsix, x, flat, 64, bstride, entry)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_sparse_decode_binding_checks_workspace(dsix):
    x = W.sparse_decode_inputs(1, 64, 64, seed=3)
    dense, flat, _, _ = _cache_bytes(x, 64)
    cache = torch.from_numpy(dense).cuda()
    out = torch.empty(1, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 128, dtype=torch.float32, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dsix.DsixError):
        dsix.dsmla_sparse_decode(x.q_nope.cuda(), x.q_pe.cuda(), cache, torch.from_numpy(x.indices).cuda(),
                                 x.sm_scale, out, lse, small)
    ws = torch.empty(dsix.dsmla_sparse_decode_workspace_size(1, 128, 64), dtype=torch.uint8, device="cuda")
    dsix.dsmla_sparse_decode(x.q_nope.cuda(), x.q_pe.cuda(), cache, torch.from_numpy(x.indices).cuda(),
                             x.sm_scale, out, lse, ws)
    torch.cuda.synchronize()
    ref_o, ref_l, ok = _oracle(x, dense, 64)
    _compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_o, ref_l,
             _vmax(dense, x.indices, 64))


def test_sparse_decode_graph_capture_replays_identically(dsix):
    """Both kernels (the merge is launched as the main kernel's programmatic
    dependent) captured in a CUDA graph: replays give the eager call's bits,
    and a replay after the inputs change follows them."""
    x = W.sparse_decode_inputs(5, 700, 2000, seed=41)
    dense, _, _, _ = _cache_bytes(x, 64)
    cache = torch.from_numpy(dense).cuda()
    qn, qp, idx = x.q_nope.cuda(), x.q_pe.cuda(), torch.from_numpy(x.indices).cuda()
    ws = torch.empty(dsix.dsmla_sparse_decode_workspace_size(5, 128, 700), dtype=torch.uint8, device="cuda")
    out_e = torch.empty(5, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse_e = torch.empty(5, 128, dtype=torch.float32, device="cuda")
    dsix.dsmla_sparse_decode(qn, qp, cache, idx, x.sm_scale, out_e, lse_e, ws)
    out_g, lse_g = torch.full_like(out_e, 7.0), torch.full_like(lse_e, 7.0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dsix.dsmla_sparse_decode(qn, qp, cache, idx, x.sm_scale, out_g, lse_g, ws,
                                     stream=torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16))
    assert torch.equal(lse_g, lse_e)
    # new query values in the captured buffers: the replay follows them
    qn.copy_(torch.flip(qn, dims=[0]))
    qp.copy_(torch.flip(qp, dims=[0]))
    g.replay()
    dsix.dsmla_sparse_decode(qn, qp, cache, idx, x.sm_scale, out_e, lse_e, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16))
    assert torch.equal(lse_g, lse_e)
