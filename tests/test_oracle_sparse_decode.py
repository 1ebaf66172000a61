"""Pins of the oracle's sparse MLA decode over the fp8_ds_mla cache (CPU only).

The step consumes the global top-k indices (ROCm/ATOM PR #1094, Technical
Details) and the 656-byte entries of vLLM PR #47090's fp8_ds_mla layout (prhub
summary, key source snippet) with the bf16 query pair (ql_nope, q_pe) of the
same page.  The pages print no attention formula; the reading is softmax
attention over the selected entries.  Each check is pinned to something other
than the oracle: closed forms (one key, identical keys, a zero query, one-hot
queries), invariances the definition fixes (order and -1 padding of the index
row), and a float64 restatement whose fp8 decode is torch's own.
"""
import math

import numpy as np
import pytest
import torch

import oracle

BS = 8
ENTRY = 656


def make_cache(nb, rng, scales=None):
    """Random valid entries, built byte by byte (no oracle code involved)."""
    cache = np.zeros((nb, BS, ENTRY), np.uint8)
    codes = rng.integers(0, 256, (nb, BS, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C           # no NaN codes
    cache[:, :, :512] = codes
    sc = (rng.random((nb, BS, 4)) * 0.02 + 0.001).astype(np.float32) if scales is None else scales
    cache[:, :, 512:528] = sc.view(np.uint8).reshape(nb, BS, 16)
    rope = torch.randn(nb, BS, 64, generator=torch.Generator().manual_seed(int(rng.integers(1 << 30))))
    cache[:, :, 528:656] = rope.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8).reshape(nb, BS, 128)
    return cache


def torch_key(cache, g):
    """float64 [576] key of slot g, decoded with torch's float8_e4m3fn."""
    e = cache.reshape(-1, ENTRY)[g]
    codes = torch.from_numpy(e[:512].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.from_numpy(e[512:528].copy()).view(torch.float32).to(torch.float64)
    nope = codes * sc.repeat_interleave(128)
    rope = torch.from_numpy(e[528:656].copy()).view(torch.bfloat16).to(torch.float64)
    return torch.cat([nope, rope]).numpy()


def bf16_bits(x):
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def run(qn, qp, cache, idx, sm_scale):
    return oracle.dsmla_sparse_decode(qn, qp, cache, BS, np.asarray(idx, np.int32), sm_scale)


def test_single_key_returns_its_value_and_score():
    rng = np.random.default_rng(0)
    cache = make_cache(3, rng)
    g = 13
    k = torch_key(cache, g)
    qn = np.zeros((1, 2, 512), np.float32)
    qp = np.zeros((1, 2, 64), np.float32)
    qn[0, 0, 400] = 1.5          # a dim of the fourth scale tile
    qp[0, 1, 7] = -2.0           # the RoPE part only
    out, lse, ok = run(bf16_bits(qn), bf16_bits(qp), cache, [[g, -1, -1]], 0.125)
    assert ok
    for h in range(2):
        assert np.array_equal(out[0, h], k[:512])        # softmax of one key is 1
    assert lse[0, 0] == 0.125 * 1.5 * k[400]
    assert lse[0, 1] == 0.125 * -2.0 * k[512 + 7]


def test_identical_keys_add_log_n():
    rng = np.random.default_rng(1)
    cache = make_cache(2, rng)
    g = 5
    n = 7
    q = rng.standard_normal((1, 1, 576)).astype(np.float32)
    qb = bf16_bits(q)
    out, lse, ok = run(qb[..., :512], qb[..., 512:], cache, [[g] * n], 0.07)
    assert ok
    k = torch_key(cache, g)
    z = 0.07 * float(np.dot(bf16_vals(qb[0, 0]), k))
    assert np.allclose(out[0, 0], k[:512], rtol=1e-15, atol=0)
    assert abs(lse[0, 0] - (z + math.log(n))) < 1e-12 * (1 + abs(z))


def test_zero_query_is_the_mean_of_the_values():
    rng = np.random.default_rng(2)
    cache = make_cache(4, rng)
    slots = rng.permutation(4 * BS)[:11]
    z = np.zeros((1, 3, 512), np.uint16)
    out, lse, ok = run(z, np.zeros((1, 3, 64), np.uint16), cache, [slots], 1.0)
    assert ok
    mean = np.mean([torch_key(cache, g)[:512] for g in slots], axis=0)
    for h in range(3):
        assert np.allclose(out[0, h], mean, rtol=1e-13, atol=1e-14)
        assert abs(lse[0, h] - math.log(11)) < 1e-14


def test_two_keys_one_hot_rope_query():
    # q_nope = 0 and q_pe = a e_r: z_j = s * a * rope_j[r], and the output is the
    # two-point softmax of those scores -- written out by hand.
    rng = np.random.default_rng(3)
    cache = make_cache(2, rng)
    g1, g2, r, a, s = 3, 12, 21, 4.0, 0.25
    qp = np.zeros((1, 1, 64), np.float32)
    qp[0, 0, r] = a
    out, lse, ok = run(np.zeros((1, 1, 512), np.uint16), bf16_bits(qp), cache, [[g1, g2]], s)
    assert ok
    k1, k2 = torch_key(cache, g1), torch_key(cache, g2)
    z1, z2 = s * a * k1[512 + r], s * a * k2[512 + r]
    w1 = 1.0 / (1.0 + math.exp(z2 - z1))
    assert np.allclose(out[0, 0], w1 * k1[:512] + (1 - w1) * k2[:512], rtol=1e-13, atol=1e-14)
    assert abs(lse[0, 0] - (max(z1, z2) + math.log1p(math.exp(-abs(z1 - z2))))) < 1e-13


def test_index_order_and_padding_do_not_matter():
    rng = np.random.default_rng(4)
    cache = make_cache(6, rng)
    q = bf16_bits(rng.standard_normal((2, 4, 576)).astype(np.float32))
    slots = rng.permutation(6 * BS)[:20].astype(np.int32)
    base = np.stack([slots, slots])
    shuffled = np.stack([rng.permutation(slots), slots[::-1]])
    padded = np.full((2, 33), -1, np.int32)
    padded[:, 1::2][:, :16] = base[:, :16]
    padded[:, 0:8:2] = base[:, 16:]
    o1, l1, _ = run(q[..., :512], q[..., 512:], cache, base, 0.08)
    o2, l2, _ = run(q[..., :512], q[..., 512:], cache, shuffled, 0.08)
    o3, l3, _ = run(q[..., :512], q[..., 512:], cache, padded, 0.08)
    for o, l in ((o2, l2), (o3, l3)):
        # summation order moves near-zero outputs by a few ulps of the values (~4)
        assert np.allclose(o, o1, rtol=1e-13, atol=1e-13)
        assert np.allclose(l, l1, rtol=1e-14, atol=1e-14)


def test_no_key_gives_zero_and_minus_inf_and_bad_index_is_reported():
    rng = np.random.default_rng(5)
    cache = make_cache(2, rng)
    q = np.zeros((2, 1, 576), np.uint16)
    out, lse, ok = run(q[..., :512], q[..., 512:], cache, [[-1, -1], [3, -1]], 1.0)
    assert ok and np.all(out[0] == 0) and lse[0, 0] == -np.inf
    _, _, ok = run(q[:1, :, :512], q[:1, :, 512:], cache, [[2 * BS, 3]], 1.0)   # one past the cache
    assert not ok


def test_random_case_against_float64_restatement():
    # Distinct tile scales per key pin the tile index of each value; the
    # restatement decodes the fp8 bytes with torch and runs a plain softmax.
    rng = np.random.default_rng(6)
    cache = make_cache(8, rng)
    T, H, K = 3, 5, 40
    q = bf16_bits(rng.standard_normal((T, H, 576)).astype(np.float32) * 2)
    idx = np.stack([rng.permutation(8 * BS)[:K] for _ in range(T)]).astype(np.int32)
    idx[1, 30:] = -1
    out, lse, ok = run(q[..., :512], q[..., 512:], cache, idx, 0.0721)
    assert ok
    qv = bf16_vals(q)
    for t in range(T):
        keys = np.array([torch_key(cache, g) for g in idx[t] if g >= 0])
        z = 0.0721 * qv[t] @ keys.T                      # [H, n]
        m = z.max(axis=1, keepdims=True)
        p = np.exp(z - m)
        ref = (p @ keys[:, :512]) / p.sum(axis=1, keepdims=True)
        assert np.allclose(out[t], ref, rtol=1e-12, atol=1e-13)
        assert np.allclose(lse[t], m[:, 0] + np.log(p.sum(axis=1)), rtol=1e-13, atol=1e-13)


def test_block_and_entry_strides():
    # The same entries placed in a padded layout (wider entries, block padding)
    # give the same result as the dense layout.
    rng = np.random.default_rng(7)
    dense = make_cache(3, rng)
    entry, extra = 672, 48
    bstride = BS * entry + extra
    flat = np.full(3 * bstride, 0xEE, np.uint8)
    for b in range(3):
        for o in range(BS):
            flat[b * bstride + o * entry:b * bstride + o * entry + ENTRY] = dense[b, o]
    q = bf16_bits(rng.standard_normal((1, 2, 576)).astype(np.float32))
    idx = np.array([[0, 9, 23, 17, 4]], np.int32)
    o1, l1, _ = run(q[..., :512], q[..., 512:], dense, idx, 0.1)
    o2, l2, ok = oracle.dsmla_sparse_decode(q[..., :512], q[..., 512:], flat, BS, idx, 0.1,
                                            block_stride=bstride, entry_stride=entry)
    assert ok
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_dominant_key_is_exact_and_overflow_free():
    # Scores of order 1e4 (far beyond exp's range) with one key ahead of all
    # others by hundreds: every other weight underflows to exactly 0 after the
    # max is subtracted, so the output is that key's value and the lse its
    # score, bit for bit -- a sum of exp(z) without the max would overflow.
    rng = np.random.default_rng(8)
    scales = np.full((2, BS, 4), 0.015625, np.float32)
    cache = make_cache(2, rng, scales=scales)
    flat = cache.reshape(-1, ENTRY)
    flat[:, 528:656] = 0                             # RoPE zero: scores from dim 0 alone
    codes = np.array([0x50, 0x48, 0x40, 0x38, 0x30], np.uint8)   # 8, 4, 2, 1, 0.5 before scaling
    slots = [3, 9, 1, 12, 6]
    for c, g in zip(codes, slots):
        flat[g, 0] = c
    qn = np.zeros((1, 1, 512), np.float32)
    qn[0, 0, 0] = 2.0 ** 16                          # exact in bf16
    out, lse, ok = run(bf16_bits(qn), np.zeros((1, 1, 64), np.uint16), cache, [slots], 1.0)
    assert ok
    k0 = torch_key(cache, slots[0])
    assert np.array_equal(out[0, 0], k0[:512])
    assert lse[0, 0] == 2.0 ** 16 * k0[0] == 8192.0   # 8 * 2^-6 * 2^16; the next score is 4096
