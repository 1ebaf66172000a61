"""Pins for the oracle's indexer logits (CPU only).

The score is k_scale[s] * sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:]).  Pins:
* closed form with one-hot q and k (one head), including a negative product
  (ReLU) and a negative weight;
* brute force on tiny shapes with exact rational arithmetic (fractions), then
  one rounding to f32 -- the oracle must agree to within one f32 ulp;
* decode visibility for next_n = 1 and 2 (row j of request b sees
  context_lens[b] - next_n + 1 + j keys) and the -inf tail when clean;
* the paged and contiguous forms agree after a gather, and the paged form is
  invariant under a relabelling of the cache blocks.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as W

E4M3 = None


def _tab():
    global E4M3
    if E4M3 is None:
        E4M3 = oracle.e4m3_decode_table()
    return E4M3


def _code(v):
    c = oracle.e4m3_encode(v)
    assert _tab()[c] == v
    return c


def _one_block_cache(kcodes, kscales, bs=64, D=128):
    """cache with one block holding the given key rows (codes) and scales."""
    n = len(kcodes)
    cache = np.zeros((1, bs * (D + 4)), np.uint8)
    for s in range(n):
        cache[0, s * D:(s + 1) * D] = kcodes[s]
        cache[0, bs * D + 4 * s:bs * D + 4 * s + 4] = np.array([kscales[s]], np.float32).view(np.uint8)
    return cache


@pytest.mark.parametrize("a,b,c,ks", [(2.0, 3.0, 0.5, 0.25), (-2.0, 3.0, 0.5, 1.0),
                                      (1.5, 448.0, -0.125, 3.0), (0.001953125, 1.0, 1.0, 2.0)])
def test_closed_form_one_hot(a, b, c, ks):
    H, D = 64, 128
    h0, d0 = 17, 90
    q = np.zeros((1, 1, H, D), np.uint8)
    q[0, 0, h0, d0] = _code(a)
    w = np.zeros((1, H), np.float32)
    w[0, h0] = c
    krow = np.zeros(D, np.uint8)
    krow[d0] = _code(b)
    cache = _one_block_cache([krow], [ks])
    out = oracle.paged_mqa_logits(q, w, cache, 64, np.array([1], np.int32),
                                  np.zeros((1, 1), np.int32), ld=4, clean=True)
    want = np.float32(ks * c * max(a * b, 0.0))
    assert out[0, 0] == want
    assert np.isneginf(out[0, 1:]).all()


def _exact_score(qc, w, kc, ksc):
    tab = _tab()
    acc = Fraction(0)
    for h in range(qc.shape[0]):
        d = sum(Fraction(float(tab[qc[h, i]])) * Fraction(float(tab[kc[i]]))
                for i in range(qc.shape[1]))
        if d > 0:
            acc += Fraction(float(w[h])) * d
    return Fraction(float(ksc)) * acc


def _f32_ulp(x):
    x = np.float32(x)
    return float(np.nextafter(np.abs(x), np.float32(np.inf)) - np.abs(x))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_exact_rational(seed):
    rng = np.random.default_rng(seed)
    H, D, n = 5, 12, 9
    # random finite codes of both signs (exclude NaN codes)
    def codes(shape):
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        return np.where((c & 0x7F) == 0x7F, c ^ 0x01, c).astype(np.uint8)
    q = codes((1, 1, H, D))
    w = (rng.standard_normal((1, H)) / 8).astype(np.float32)
    kc = codes((n, D))
    ksc = (rng.random(n) * 0.01 + 1e-3).astype(np.float32)
    bs = 4
    cache = np.zeros((3, bs * (D + 4)), np.uint8)
    bt = np.array([[2, 0, 1]], np.int32)
    for s in range(n):
        blk, off = bt[0, s // bs], s % bs
        cache[blk, off * D:(off + 1) * D] = kc[s]
        cache[blk, bs * D + 4 * off:bs * D + 4 * off + 4] = np.array([ksc[s]], np.float32).view(np.uint8)
    out = oracle.paged_mqa_logits(q, w, cache, bs, np.array([n], np.int32), bt, ld=n)
    for s in range(n):
        exact = _exact_score(q[0, 0], w[0], kc[s], ksc[s])
        want = np.float32(float(exact))
        assert abs(float(out[0, s]) - float(want)) <= _f32_ulp(want), (s, out[0, s], want)


def test_relu_all_negative_gives_zero():
    H, D = 64, 128
    q = np.full((1, 1, H, D), _code(1.0), np.uint8)
    w = np.ones((1, H), np.float32)
    krow = np.full(D, _code(-2.0), np.uint8)
    cache = _one_block_cache([krow], [1.0])
    out = oracle.paged_mqa_logits(q, w, cache, 64, np.array([1], np.int32),
                                  np.zeros((1, 1), np.int32), ld=1)
    assert out[0, 0] == 0.0


def _setup_decode(wl):
    cache = np.zeros((wl.num_blocks, wl.block_size * (wl.head_dim + 4)), np.uint8)
    oracle.quant_write_k(W.bf16_bits(wl.k_bf16), wl.slot, cache, wl.block_size)
    return cache


@pytest.mark.parametrize("next_n", [1, 2])
def test_decode_visibility_and_tail(next_n):
    wl = W.build("vis", decode_ctx=[5, 64, 130], next_n=next_n, topk=8, seed=3)
    cache = _setup_decode(wl)
    ld = 160
    out = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                  wl.context_lens, wl.block_table, ld=ld, clean=True)
    row_len, _ = wl.decode_rows()
    for r in range(out.shape[0]):
        b, j = divmod(r, next_n)
        L = int(wl.context_lens[b]) - next_n + 1 + j
        assert row_len[r] == L
        assert np.isfinite(out[r, :L]).all()
        assert np.isneginf(out[r, L:]).all()
    # the same row sets compute the same values; unclean leaves the tail alone
    out2 = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                   wl.context_lens, wl.block_table, ld=ld, clean=False)
    for r in range(out.shape[0]):
        L = row_len[r]
        assert np.array_equal(out[r, :L], out2[r, :L])
        assert (out2[r, L:] == 0).all()
    sub = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                  wl.context_lens, wl.block_table, ld=ld, rows=[2, 0])
    assert np.array_equal(sub[0], out[2]) and np.array_equal(sub[1], out[0])


def test_paged_equals_contiguous_after_gather():
    wl = W.build("pc", decode_ctx=[70, 129], next_n=1, topk=8, seed=5, pool_blocks=7)
    cache = _setup_decode(wl)
    ld = 129
    paged = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                    wl.context_lens, wl.block_table, ld=ld)
    cu = np.concatenate([[0], np.cumsum(wl.req_ctx)]).astype(np.int32)
    T = int(cu[-1])
    kf = np.zeros((T, 128), np.uint8)
    kscale = np.zeros(T, np.float32)
    oracle.gather_k(cache, 64, 128, wl.block_table, cu, kf, kscale)
    q = W.u8(wl.q_decode).reshape(2, 64, 128)
    ks = cu[:-1].copy()
    ke = cu[1:].copy()
    cont = oracle.mqa_logits(q, wl.w_decode.numpy(), kf, kscale, ks, ke, ld=ld)
    assert np.array_equal(paged.view(np.uint32), cont.view(np.uint32))


def test_block_relabelling_invariance():
    wl = W.build("perm", decode_ctx=[150], next_n=1, topk=8, seed=6, pool_blocks=5)
    cache = _setup_decode(wl)
    out = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache, 64,
                                  wl.context_lens, wl.block_table, ld=150)
    perm = np.array([3, 0, 4, 1, 2])
    cache2 = np.zeros_like(cache)
    cache2[perm] = cache
    bt2 = perm[wl.block_table].astype(np.int32)
    out2 = oracle.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), cache2, 64,
                                   wl.context_lens, bt2, ld=150)
    assert np.array_equal(out, out2)


def test_prefill_causal_ranges():
    rng = np.random.default_rng(0)
    T, H, D = 20, 64, 128
    q = torch.randn(T, H, D, generator=torch.Generator().manual_seed(1)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    k = torch.randn(T, D, generator=torch.Generator().manual_seed(2)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    ksc = rng.random(T).astype(np.float32)
    w = (rng.standard_normal((T, H)) / 8).astype(np.float32)
    ks = np.zeros(T, np.int32)
    ke = np.arange(1, T + 1, dtype=np.int32)
    out = oracle.mqa_logits(q, w, k, ksc, ks, ke, ld=T)
    for t in range(T):
        assert np.isfinite(out[t, :t + 1]).all() and np.isneginf(out[t, t + 1:]).all()
    # a shifted window [ks, ke) lands at columns 0.. of the row
    ks2 = np.full(T, 3, np.int32)
    ke2 = np.full(T, 11, np.int32)
    out2 = oracle.mqa_logits(q, w, k, ksc, ks2, ke2, ld=8)
    full = oracle.mqa_logits(q, w, k, ksc, np.zeros(T, np.int32), np.full(T, T, np.int32), ld=T)
    assert np.array_equal(out2, full[:, 3:11])
