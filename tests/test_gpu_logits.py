"""GPU parity: paged (decode) and contiguous (prefill) FP8 MQA logits against the
oracle, |d| <= 1e-3 * max|row| + 1e-4; full rows where the oracle finishes in
seconds, sampled rows at full sizes (same launch as the benchmark)."""
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


def _decode_gpu(dsix, wl, clean, ld=None, sentinel=123.0):
    step = make_step(wl, "cuda", clean=clean)
    dsix.ix_quant_write_k(step.new_k, step.new_slot, step.cache)  # the step's new tokens
    d = step.decode
    ld = ld or d.ld
    logits = torch.full((d.w.shape[0], ld), sentinel, dtype=torch.float32, device="cuda")
    dsix.ix_paged_mqa_logits(d.q, d.w, step.cache, d.context_lens, step.block_table, logits,
                             clean_logits=clean)
    torch.cuda.synchronize()
    return step, logits.cpu().numpy()


@pytest.mark.parametrize("next_n", [1, 2])
@pytest.mark.parametrize("clean", [True, False])
def test_decode_small_ragged(dsix, next_n, clean):
    ctx = [1, 2, 5, 63, 64, 65, 127, 128, 129, 255, 256, 300, 1000, 1025]
    wl = W.build("small", decode_ctx=ctx, next_n=next_n, topk=16, seed=11 + next_n,
                 pool_blocks=80)
    step, got = _decode_gpu(dsix, wl, clean, ld=1028)
    cache = oracle_cache(wl)
    assert np.array_equal(step.cache.cpu().numpy(), cache)
    ref = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                  wl.context_lens, wl.block_table, ld=1028, clean=True)
    row_len, _ = wl.decode_rows()
    check_logits_rows(got, ref, row_len, "decode")
    for r, L in enumerate(row_len):
        if clean:
            assert np.isneginf(got[r, L:]).all()
        else:
            assert (got[r, L:] == 123.0).all()
    assert dsix.ix_device_status() == 0


def test_decode_tiny_config(dsix):
    wl = W.tiny_decode()
    _, got = _decode_gpu(dsix, wl, True)
    ref = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), oracle_cache(wl), 64,
                                  wl.context_lens, wl.block_table, ld=got.shape[1])
    check_logits_rows(got, ref, wl.decode_rows()[0], "tiny")


def test_decode_b32_full(dsix):
    wl = W.decode_b32()
    _, got = _decode_gpu(dsix, wl, False)
    ref = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), oracle_cache(wl), 64,
                                  wl.context_lens, wl.block_table, ld=got.shape[1])
    check_logits_rows(got, ref, wl.decode_rows()[0], "b32")


def test_decode_mtp2_sampled(dsix):
    wl = W.decode_mtp2_b128()
    _, got = _decode_gpu(dsix, wl, False)
    rows = [0, 1, 77, 128, 200, 255]
    ref = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), oracle_cache(wl), 64,
                                  wl.context_lens, wl.block_table, ld=got.shape[1], rows=rows)
    rl = wl.decode_rows()[0]
    check_logits_rows(got[rows], ref, rl[rows], "mtp2")


def test_decode_mixed_long_sampled(dsix):
    wl = W.mixed_long()
    step = make_step(wl, "cuda")
    step.run()
    torch.cuda.synchronize()
    got = step.dec_logits.cpu().numpy()
    rows = [0, 15]
    cache = oracle_cache(wl)
    ref = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                  wl.context_lens, wl.block_table, ld=got.shape[1], rows=rows)
    check_logits_rows(got[rows], ref, wl.decode_rows()[0][rows], "mixed decode")
    # prefill part of the same launch
    ks, ke, rl, _ = wl.prefill_rows()
    cu = wl.prefill_gather()
    kf = np.zeros((int(cu[-1]), 128), np.uint8)
    kscale = np.zeros(int(cu[-1]), np.float32)
    oracle.gather_k(cache, 64, 128, wl.prefill_block_table(), cu, kf, kscale)
    prow = [0, 1, 2047, 2048, 5000, 8191]
    pref = oracle.mqa_logits(W.u8(wl.q_prefill), wl.w_prefill.numpy(), kf, kscale, ks, ke,
                             ld=step.prefill.ld, rows=prow)
    pgot = step.pf_logits.cpu().numpy()[prow]
    check_logits_rows(pgot, pref, rl[prow], "mixed prefill")
    assert dsix.ix_device_status() == 0


@pytest.mark.parametrize("clean", [True, False])
def test_prefill_small_ranges(dsix, clean):
    g = torch.Generator().manual_seed(5)
    tq, tk = 37, 300
    q = torch.randn(tq, 64, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    k = torch.randn(tk, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    ksc = (torch.rand(tk, generator=g) * 0.01 + 1e-3)
    w = torch.randn(tq, 64, generator=g) / 8
    rng = np.random.default_rng(0)
    ks = rng.integers(0, tk, tq).astype(np.int32)
    ke = np.minimum(ks + rng.integers(0, 260, tq), tk).astype(np.int32)
    ks[0], ke[0] = 10, 10            # empty row
    ks[1], ke[1] = 0, tk             # full row
    ks[2], ke[2] = 131, 133          # unaligned start
    ld = 304
    ref = oracle.mqa_logits(q.numpy(), w.numpy(), k.numpy(), ksc.numpy(), ks, ke, ld=ld)
    out = torch.full((tq, ld), 77.0, device="cuda")
    dsix.ix_mqa_logits(q.cuda(), w.cuda(), k.cuda(), ksc.cuda(), torch.from_numpy(ks).cuda(),
                       torch.from_numpy(ke).cuda(), out, clean_logits=clean)
    got = out.cpu().numpy()
    lens = ke - ks
    check_logits_rows(got, ref, lens, "prefill small")
    for t in range(tq):
        tail = got[t, lens[t]:]
        assert (np.isneginf(tail).all() if clean else (tail == 77.0).all())
    assert dsix.ix_device_status() == 0


def test_prefill_8k_causal_sampled(dsix):
    wl = W.prefill_8k()
    step = make_step(wl, "cuda")
    step.run()
    torch.cuda.synchronize()
    ks, ke, rl, _ = wl.prefill_rows()
    cache = oracle_cache(wl)
    cu = wl.prefill_gather()
    kf = np.zeros((8192, 128), np.uint8)
    kscale = np.zeros(8192, np.float32)
    oracle.gather_k(cache, 64, 128, wl.prefill_block_table(), cu, kf, kscale)
    assert np.array_equal(step.k_fp8.cpu().numpy(), kf)
    rows = [0, 1, 7, 8, 127, 128, 129, 1000, 2047, 2048, 4095, 6000, 8190, 8191]
    ref = oracle.mqa_logits(W.u8(wl.q_prefill), wl.w_prefill.numpy(), kf, kscale, ks, ke,
                            ld=step.prefill.ld, rows=rows)
    got = step.pf_logits.cpu().numpy()[rows]
    check_logits_rows(got, ref, rl[rows], "prefill 8k")
    assert dsix.ix_device_status() == 0


def test_bad_block_is_flagged_not_faulted(dsix):
    wl = W.build("bad", decode_ctx=[200], next_n=1, topk=8, seed=3)
    step = make_step(wl, "cuda")
    bt = step.block_table.clone()
    bt[0, 1] = 1 << 30
    logits = torch.zeros(1, 200, device="cuda")
    d = step.decode
    dsix.ix_paged_mqa_logits(d.q, d.w, step.cache, d.context_lens, bt, logits)
    assert dsix.ix_device_status() & 2  # IX_DEV_BAD_BLOCK
