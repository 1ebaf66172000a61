"""GPU parity: fused logits + top-k (ix_paged_mqa_logits_topk, ix_mqa_logits_topk)
and their halves (ix_*_logits_hist, ix_topk_from_hist).

The fused calls promise exactly what the unfused pair computes: the same
logits, bit for bit, and the same selection.  Checked against
  * the unfused GPU pair (logits bit-identical over every row's visible part,
    local and global indices identical);
  * the oracle's top-k run on the GPU's own logits (exact, ties to the lower
    index included), on every row of the small cases and on sampled rows of
    the full-size ones;
  * the oracle's logits within |d| <= 1e-3 * max|row| + 1e-4 on sampled rows.
Both selection kernels run (one warp per row when there are >= 2 x SMs rows
of <= 65536 keys, the cluster kernel otherwise), as do the threshold-digit
candidates held in shared memory and the path that re-reads the row when the
digit holds too many keys (rows of equal logits).  The workspace is zero
again after every call.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import check_logits_rows, oracle_cache, require_gpu
from workloads.device import make_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsix():
    require_gpu()
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v3_sparse_gb300 as m
    m.ix_device_status()
    return m


def _ws(dsix, rows):
    return torch.zeros(dsix.ix_topk_hist_workspace_size(rows), dtype=torch.uint8, device="cuda")


def _oracle_exact(logits, lens, reqs, bt, k, loc, glb, rows, bs=64):
    rows = np.asarray(rows)
    rl, rg = oracle.topk_to_global(np.ascontiguousarray(logits[rows]), np.asarray(lens, np.int32)[rows],
                                   np.asarray(reqs, np.int32)[rows], bt, bs, k)
    bad = np.nonzero((loc[rows] != rl).any(axis=1) | (glb[rows] != rg).any(axis=1))[0]
    assert bad.size == 0, f"rows {rows[bad[:5]]} differ from the oracle's top-k of the GPU logits"


def _same_visible(a, b, lens):
    for r, L in enumerate(lens):
        assert np.array_equal(a[r, :L].view(np.uint32), b[r, :L].view(np.uint32)), f"row {r}: logits differ"


# ---------------------------------------------------------------------------
# prefill (contiguous K)
# ---------------------------------------------------------------------------
def _prefill_inputs(tq, tk, seed, zero_q_rows=(), dup_keys=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(tq, 64, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    k = torch.randn(tk, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    if dup_keys:  # repeated keys: exact ties between different indices
        k[1::7] = k[0]
    ksc = torch.rand(tk, generator=g) * 0.01 + 1e-3
    if dup_keys:
        ksc[1::7] = ksc[0]
    w = torch.randn(tq, 64, generator=g) / 8
    for r in zero_q_rows:  # every logit of the row is zero: one digit holds the whole row
        q[r] = 0
    return q, k, ksc, w


def _run_prefill_both(dsix, q, k, ksc, w, ks, ke, req, bt, topk, ld):
    tq = q.shape[0]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    qd, kd, sd, wd = q.cuda(), k.cuda(), ksc.cuda(), w.cuda()
    ksd, ked, rqd, btd = dev(ks), dev(ke), dev(req), dev(bt)
    lg_f = torch.full((tq, ld), 55.0, device="cuda")
    glb_f = torch.full((tq, topk), -7, dtype=torch.int32, device="cuda")
    loc_f = torch.full((tq, topk), -7, dtype=torch.int32, device="cuda")
    ws = _ws(dsix, tq)
    dsix.ix_mqa_logits_topk(qd, wd, kd, sd, ksd, ked, lg_f, rqd, btd, topk, glb_f, ws, out_local=loc_f)
    lg_u = torch.full((tq, ld), 55.0, device="cuda")
    glb_u = torch.full((tq, topk), -7, dtype=torch.int32, device="cuda")
    loc_u = torch.full((tq, topk), -7, dtype=torch.int32, device="cuda")
    dsix.ix_mqa_logits(qd, wd, kd, sd, ksd, ked, lg_u)
    lens = np.clip(ke.astype(np.int64) - ks.astype(np.int64), 0, ld).astype(np.int32)
    dsix.ix_topk_to_global(lg_u, dev(lens), rqd, btd, topk, glb_u, loc_u)
    # the two halves, on a workspace of their own
    lg_h = torch.full((tq, ld), 55.0, device="cuda")
    glb_h = torch.full((tq, topk), -7, dtype=torch.int32, device="cuda")
    ws_h = _ws(dsix, tq)
    dsix.ix_mqa_logits_hist(qd, wd, kd, sd, ksd, ked, lg_h, topk, ws_h)
    dsix.ix_topk_from_hist(lg_h, dev(lens), rqd, btd, topk, glb_h, ws_h)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    assert int(ws.count_nonzero()) == 0 and int(ws_h.count_nonzero()) == 0, "workspace not left zero"
    out = dict(lg_f=lg_f.cpu().numpy(), glb_f=glb_f.cpu().numpy(), loc_f=loc_f.cpu().numpy(),
               lg_u=lg_u.cpu().numpy(), glb_u=glb_u.cpu().numpy(), loc_u=loc_u.cpu().numpy(),
               lg_h=lg_h.cpu().numpy(), glb_h=glb_h.cpu().numpy(), lens=lens)
    _same_visible(out["lg_f"], out["lg_u"], lens)
    _same_visible(out["lg_h"], out["lg_u"], lens)
    assert np.array_equal(out["glb_f"], out["glb_u"]) and np.array_equal(out["loc_f"], out["loc_u"])
    assert np.array_equal(out["glb_h"], out["glb_u"])
    return out


@pytest.mark.parametrize("tq,topk", [(640, 256), (40, 256), (640, 7), (400, 1)])
def test_prefill_windows_ties_and_edges(dsix, tq, topk):
    """Random [ks, ke) windows incl. empty, L = k, L = k + 1, full rows; rows of
    all-zero logits; repeated keys.  tq = 640/400 take the warp-per-row
    selection, tq = 40 the cluster kernel."""
    tk, ld = 3000, 3000
    q, k, ksc, w = _prefill_inputs(tq, tk, seed=tq + topk, zero_q_rows=(5, 6, tq - 1), dup_keys=7)
    rng = np.random.default_rng(tq * 31 + topk)
    ks = rng.integers(0, tk, tq).astype(np.int32)
    ke = np.minimum(ks + rng.integers(0, tk, tq), tk).astype(np.int32)
    ks[0], ke[0] = 10, 10                    # empty row
    ks[1], ke[1] = 0, tk                     # full row
    ks[2], ke[2] = 100, 100 + topk           # L = k
    ks[3], ke[3] = 7, 8 + topk               # L = k + 1
    ks[4], ke[4] = 131, 133                  # unaligned start, L = 2
    ks[5], ke[5] = 0, tk                     # all zero, full row (more than 512 equal keys)
    ks[6], ke[6] = 1, 1 + min(tk - 1, topk + 300)
    req = rng.integers(0, 4, tq).astype(np.int32)
    bt = np.random.default_rng(1).permutation(4 * 47).reshape(4, 47).astype(np.int32)
    o = _run_prefill_both(dsix, q, k, ksc, w, ks, ke, req, bt, topk, ld)
    _oracle_exact(o["lg_f"], o["lens"], req, bt, topk, o["loc_f"], o["glb_f"], np.arange(tq))
    # the all-zero rows take the lowest indices
    assert np.array_equal(o["loc_f"][5], np.arange(topk))
    ref = oracle.mqa_logits(q.numpy(), w.numpy(), k.numpy(), ksc.numpy(), ks, ke, ld=ld, rows=[1, 3, 6, 17])
    check_logits_rows(o["lg_f"][[1, 3, 6, 17]], ref, o["lens"][[1, 3, 6, 17]], "fused prefill")


def test_prefill_8k_causal_full(dsix):
    """The 8192-token causal chunk at full size, in the launch the benchmark
    times: fused = unfused on every row; oracle top-k of the GPU logits exact on
    sampled rows; oracle logits on sampled rows."""
    wl = W.prefill_8k()
    step = make_step(wl, "cuda")
    step.run()
    p = step.prefill
    T, topk = 8192, wl.topk
    ws = _ws(dsix, T)
    lg = torch.empty(T, p.ld, device="cuda")
    glb = torch.full((T, topk), -7, dtype=torch.int32, device="cuda")
    loc = torch.full((T, topk), -7, dtype=torch.int32, device="cuda")
    for _ in range(2):  # twice on one workspace: it is left zero, the second call is the same
        dsix.ix_mqa_logits_topk(p.q, p.w, step.k_fp8, step.k_scale, p.ks, p.ke, lg, p.row_req, step.block_table,
                                topk, glb, ws, out_local=loc)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    assert int(ws.count_nonzero()) == 0
    lens = p.row_len.cpu().numpy()
    got_lg = lg.cpu().numpy()
    _same_visible(got_lg, step.pf_logits.cpu().numpy(), lens)
    assert np.array_equal(glb.cpu().numpy(), step.pf_global.cpu().numpy())
    rows = [0, 1, 2046, 2047, 2048, 2049, 4095, 6000, 8190, 8191]
    _oracle_exact(got_lg, lens, p.row_req.cpu().numpy(), wl.block_table, topk, loc.cpu().numpy(),
                  glb.cpu().numpy(), rows)
    ks, ke, rl, _ = wl.prefill_rows()
    cache = oracle_cache(wl)
    kf = np.zeros((8192, 128), np.uint8)
    kscale = np.zeros(8192, np.float32)
    oracle.gather_k(cache, 64, 128, wl.prefill_block_table(), wl.prefill_gather(), kf, kscale)
    ref = oracle.mqa_logits(W.u8(wl.q_prefill), wl.w_prefill.numpy(), kf, kscale, ks, ke, ld=p.ld, rows=rows)
    check_logits_rows(got_lg[rows], ref, rl[rows], "fused prefill 8k")


# ---------------------------------------------------------------------------
# decode (paged)
# ---------------------------------------------------------------------------
def _decode_both(dsix, wl, rows_checked):
    step = make_step(wl, "cuda")
    dsix.ix_quant_write_k(step.new_k, step.new_slot, step.cache)
    d = step.decode
    R, topk = d.w.shape[0], wl.topk
    ws = _ws(dsix, R)
    lg = torch.full((R, d.ld), 55.0, device="cuda")
    glb = torch.full((R, topk), -7, dtype=torch.int32, device="cuda")
    loc = torch.full((R, topk), -7, dtype=torch.int32, device="cuda")
    dsix.ix_paged_mqa_logits_topk(d.q, d.w, step.cache, d.context_lens, step.block_table, lg, topk, glb, ws,
                                  out_local=loc)
    lg_u = torch.full((R, d.ld), 55.0, device="cuda")
    glb_u = torch.full((R, topk), -7, dtype=torch.int32, device="cuda")
    dsix.ix_paged_mqa_logits(d.q, d.w, step.cache, d.context_lens, step.block_table, lg_u)
    dsix.ix_topk_to_global(lg_u, d.row_len, d.row_req, step.block_table, topk, glb_u, None)
    lg_h = torch.full((R, d.ld), 55.0, device="cuda")
    glb_h = torch.full((R, topk), -7, dtype=torch.int32, device="cuda")
    ws_h = _ws(dsix, R)
    dsix.ix_paged_mqa_logits_hist(d.q, d.w, step.cache, d.context_lens, step.block_table, lg_h, topk, ws_h)
    dsix.ix_topk_from_hist(lg_h, d.row_len, d.row_req, step.block_table, topk, glb_h, ws_h)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    assert int(ws.count_nonzero()) == 0 and int(ws_h.count_nonzero()) == 0
    lens, reqs = wl.decode_rows()
    got = lg.cpu().numpy()
    _same_visible(got, lg_u.cpu().numpy(), lens)
    _same_visible(lg_h.cpu().numpy(), lg_u.cpu().numpy(), lens)
    g = glb.cpu().numpy()
    assert np.array_equal(g, glb_u.cpu().numpy()) and np.array_equal(g, glb_h.cpu().numpy())
    _oracle_exact(got, lens, reqs, wl.block_table, topk, loc.cpu().numpy(), g, rows_checked)
    return got, lens


def test_decode_tiny(dsix):
    wl = W.tiny_decode()
    got, lens = _decode_both(dsix, wl, [0, 1])
    ref = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), oracle_cache(wl), 64,
                                  wl.context_lens, wl.block_table, ld=got.shape[1])
    check_logits_rows(got, ref, lens, "fused tiny")


@pytest.mark.parametrize("next_n", [1, 2])
def test_decode_small_ragged(dsix, next_n):
    ctx = [1, 2, 5, 63, 64, 65, 127, 128, 129, 255, 256, 300, 1000, 1025, 3000]
    wl = W.build("small", decode_ctx=ctx, next_n=next_n, topk=128, seed=21 + next_n, pool_blocks=120)
    _decode_both(dsix, wl, np.arange(len(ctx) * next_n))


def test_decode_b32(dsix):
    _decode_both(dsix, W.decode_b32(), np.arange(32))


def test_decode_mtp2(dsix):
    _decode_both(dsix, W.decode_mtp2_b128(), [0, 1, 77, 128, 200, 255])


def test_decode_mixed_long(dsix):
    wl = W.mixed_long()
    _decode_both(dsix, wl, [0, 9, 15])


def test_prefill_long_rows_cluster_path_and_periodic_handoff(dsix):
    """Prefill rows longer than 32768 keys: the histogram variant hands each
    row's shared-memory counts off every 256 tiles (so no 16-bit counter
    overflows), and with few rows the selection runs the cluster kernel from
    the histograms.  A row of equal logits (zero query) holds all its keys in
    one digit."""
    tq, tk, topk = 24, 70000, 2048
    q, k, ksc, w = _prefill_inputs(tq, tk, seed=101, zero_q_rows=(3,), dup_keys=5)
    rng = np.random.default_rng(7)
    ks = np.zeros(tq, np.int32)
    ke = rng.integers(30000, tk + 1, tq).astype(np.int32)
    ke[0] = tk                           # the longest row (70000 keys: 547 tiles, two hand-offs)
    ke[1] = topk                         # L = k: no histogram
    ke[2] = topk + 1
    ke[3] = tk
    ld = 70000
    req = np.zeros(tq, np.int32)
    bt = np.random.default_rng(3).permutation(1100).reshape(1, 1100).astype(np.int32)
    o = _run_prefill_both(dsix, q, k, ksc, w, ks, ke, req, bt, topk, ld)
    _oracle_exact(o["lg_f"], o["lens"], req, bt, topk, o["loc_f"], o["glb_f"], np.arange(tq))
    assert np.array_equal(o["loc_f"][3], np.arange(topk))
