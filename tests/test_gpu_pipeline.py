"""GPU parity of whole indexer steps (the benchmark's launch sequence) and
CUDA-graph capture of a step."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import check_logits_rows, check_topk_rows, oracle_cache, require_gpu
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


def _decode_check(wl, step, rows=None):
    cache = oracle_cache(wl)
    rl, rq = wl.decode_rows()
    rows = list(range(len(rl))) if rows is None else rows
    ref = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                  wl.context_lens, wl.block_table, ld=step.decode.ld, rows=rows)
    got = step.dec_logits.cpu().numpy()[rows]
    check_logits_rows(got, ref, rl[rows], "decode")
    check_topk_rows(step.dec_local.cpu().numpy()[rows], step.dec_global.cpu().numpy()[rows], ref,
                    rl[rows], rq[rows], wl.block_table, 64, wl.topk, "decode top-k")
    # the GPU top-k applied to the oracle's logits is exact
    return cache


@pytest.mark.parametrize("name", ["tiny_decode", "decode_b32"])
def test_decode_pipeline(dsix, name):
    wl = W.NAMED[name]()
    step = make_step(wl, "cuda", with_local=True)
    step.run()
    torch.cuda.synchronize()
    _decode_check(wl, step)
    assert dsix.ix_device_status() == 0


def test_decode_mtp2_pipeline_sampled(dsix):
    wl = W.decode_mtp2_b128()
    step = make_step(wl, "cuda", with_local=True)
    step.run()
    torch.cuda.synchronize()
    _decode_check(wl, step, rows=[0, 3, 100, 254, 255])


def test_prefill_pipeline_sampled(dsix):
    wl = W.prefill_8k()
    step = make_step(wl, "cuda", with_local=True)
    step.run()
    torch.cuda.synchronize()
    cache = oracle_cache(wl)
    ks, ke, rl, rq = wl.prefill_rows()
    cu = wl.prefill_gather()
    kf = np.zeros((8192, 128), np.uint8)
    kscale = np.zeros(8192, np.float32)
    oracle.gather_k(cache, 64, 128, wl.prefill_block_table(), cu, kf, kscale)
    rows = [0, 2047, 2048, 3000, 8191]
    ref = oracle.mqa_logits(W.u8(wl.q_prefill), wl.w_prefill.numpy(), kf, kscale, ks, ke,
                            ld=step.prefill.ld, rows=rows)
    check_topk_rows(step.pf_local.cpu().numpy()[rows], step.pf_global.cpu().numpy()[rows], ref,
                    rl[rows], rq[rows], wl.block_table, 64, wl.topk, "prefill top-k")


def test_mixed_long_pipeline_sampled(dsix):
    wl = W.mixed_long()
    step = make_step(wl, "cuda", with_local=True)
    step.run()
    torch.cuda.synchronize()
    cache = _decode_check(wl, step, rows=[0, 9])
    ks, ke, rl, rq = wl.prefill_rows()
    cu = wl.prefill_gather()
    kf = np.zeros((int(cu[-1]), 128), np.uint8)
    kscale = np.zeros(int(cu[-1]), np.float32)
    oracle.gather_k(cache, 64, 128, wl.prefill_block_table(), cu, kf, kscale)
    rows = [0, 2049, 6143, 8191]
    ref = oracle.mqa_logits(W.u8(wl.q_prefill), wl.w_prefill.numpy(), kf, kscale, ks, ke,
                            ld=step.prefill.ld, rows=rows)
    check_topk_rows(step.pf_local.cpu().numpy()[rows], step.pf_global.cpu().numpy()[rows], ref,
                    rl[rows], rq[rows], wl.block_table, 64, wl.topk, "mixed prefill top-k")
    assert dsix.ix_device_status() == 0


@pytest.mark.parametrize("name", ["decode_b32", "mixed_long"])
def test_fused_step_matches_unfused_step(dsix, name):
    """The benchmark's step with the fused calls selects exactly what the step
    with the unfused pairs selects."""
    wl = W.NAMED[name]()
    a = make_step(wl, "cuda", with_local=True)
    b = make_step(wl, "cuda", with_local=True, fused=True)
    a.run()
    b.run()
    b.run()  # a second step on the same workspaces
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    assert torch.equal(a.dec_global, b.dec_global) and torch.equal(a.dec_local, b.dec_local)
    if wl.prefill_req:
        assert torch.equal(a.pf_global, b.pf_global) and torch.equal(a.pf_local, b.pf_local)


@pytest.mark.parametrize("fused", [False, True])
def test_graph_capture_replays_identically(dsix, fused):
    wl = W.build("graph", decode_ctx=[300, 5000, 77], next_n=2, prefill=[(1000, 300)],
                 topk=256, seed=9, dsmla=True)
    step = make_step(wl, "cuda", clean=not fused, with_local=True, fused=fused)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step.run(stream=s)          # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (step.dec_logits, step.dec_global, step.pf_logits, step.pf_global,
                                 step.dec_local, step.pf_local)]
    for t in (step.dec_logits, step.pf_logits):
        t.fill_(0.5)
    for t in (step.dec_global, step.pf_global, step.dec_local, step.pf_local):
        t.fill_(-9)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    again = (step.dec_logits, step.dec_global, step.pf_logits, step.pf_global, step.dec_local,
             step.pf_local)
    for i, (a, b) in enumerate(zip(eager, again)):
        if fused and i in (0, 2):  # the fused calls leave the logits past each row's end untouched
            lens = (step.decode if i == 0 else step.prefill).row_len.cpu().tolist()
            for r, L in enumerate(lens):
                assert torch.equal(a[r, :L], b[r, :L])
        else:
            assert torch.equal(a, b)
    assert dsix.ix_device_status() == 0
    if fused:  # each replay left the histogram workspaces zero
        assert int(step.dec_ws.count_nonzero()) == 0 and int(step.pf_ws.count_nonzero()) == 0


def test_step_graph_method_matches_eager(dsix):
    """IndexerStep.graph() (the benchmark's timed step): captured after an eager
    run, its replays give the eager step's indices and visible logits, also after
    the cache is rewritten between replays (the graph reads it in place)."""
    wl = W.build("graph_method", decode_ctx=[4100, 70], next_n=1, prefill=[(600, 200)],
                 topk=128, seed=17, dsmla=True)
    step = make_step(wl, "cuda", fused=("decode",))
    step.run()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (step.dec_global, step.pf_global)]
    g = step.graph()
    assert step.graph() is g  # captured once
    for t in (step.dec_global, step.pf_global):
        t.fill_(-9)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(step.dec_global, eager[0]) and torch.equal(step.pf_global, eager[1])
    # new cache contents: the replay follows them, as the eager step does
    step.cache.copy_(torch.roll(step.cache, shifts=1, dims=0))
    g.replay()
    torch.cuda.synchronize()
    replayed = [t.clone() for t in (step.dec_global, step.pf_global, step.dec_logits)]
    step.run()
    torch.cuda.synchronize()
    assert torch.equal(replayed[0], step.dec_global) and torch.equal(replayed[1], step.pf_global)
    for r, L in enumerate(step.decode.row_len.cpu().tolist()):
        assert torch.equal(replayed[2][r, :L], step.dec_logits[r, :L])
    assert dsix.ix_device_status() == 0
    assert int(step.dec_ws.count_nonzero()) == 0
