"""Pins of the oracle's fused RMSNorm + RoPE + fp8_ds_mla write (CPU only).

The step is the per-token body of vLLM PR #47090's _fused_norm_rope_kernel,
fp8_ds_mla branch (prhub summary, key source snippet): the NoPE values are
RMS-normalised and scaled by the norm weights, then coded per 128-value tile;
the RoPE pairs are rotated and stored interleaved (r1 at 2i, r2 at 2i + 1).
The page prints neither the norm nor the rotation formula; the readings are in
the oracle's header.  Each check below is pinned to something other than the
oracle itself: a closed form, an exact invariance, an fp64 restatement within
the coding's error bound, or a hand-made rounding case.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")

BS = 4          # tokens per cache block in these small cases
ENTRY = 656


def bf16_bits(x):
    """f32 values that are exact bf16 values -> their bf16 bits."""
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "test inputs must be exact bf16 values"
    return (u >> 16).astype(np.uint16)


def bf16_values(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def round_bf16(x):
    """Any f32 -> nearest bf16 value (test-side helper for random inputs)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def run(kv, pe, gamma, eps, pos, cos_sin, slots=None, blocks=None):
    n = kv.shape[0]
    slots = np.arange(n, dtype=np.int64) if slots is None else np.asarray(slots, np.int64)
    nb = blocks if blocks is not None else (n + BS - 1) // BS + 1
    cache = np.full((nb, BS, ENTRY), 0xAB, np.uint8)
    ok = oracle.dsmla_norm_rope_write(bf16_bits(kv), bf16_bits(pe), bf16_bits(gamma), eps,
                                      np.asarray(pos, np.int64), np.asarray(cos_sin, np.float32),
                                      slots, cache, BS)
    return ok, cache


def entry(cache, slot):
    return cache[slot // BS, slot % BS]


def nope_decoded(e):
    codes = e[:512]
    scales = e[512:528].view(np.float32)
    dec = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    return dec * np.repeat(scales.astype(np.float64), 128)


def rope_values(e):
    return bf16_values(e[528:656].view(np.uint16))


def identity_table(max_pos=4):
    t = np.zeros((max_pos, 64), np.float32)
    t[:, :32] = 1.0
    return t


def test_constant_token_closed_form():
    # x_i = a, unit weights, eps 0: r = 1/|a| and every y_i = sign(a) * 1, so
    # each tile has amax 1, scale f32(1/448) and codes enc(1/f32(1/448)) = 448.
    for a in (2.0, 0.75, -3.0, 0.005859375):
        kv = np.full((1, 512), a, np.float32)
        ok, cache = run(kv, np.ones((1, 64), np.float32), np.ones(512, np.float32), 0.0, [0],
                        identity_table())
        assert ok
        e = entry(cache, 0)
        want = 0x7E if a > 0 else 0xFE
        assert np.all(e[:512] == want), a
        assert np.all(e[512:528].view(np.float32) == np.float32(1.0 / 448.0)), a


def test_zero_token_floor_scale():
    ok, cache = run(np.zeros((1, 512), np.float32), np.zeros((1, 64), np.float32),
                    np.ones(512, np.float32), 1e-6, [1], identity_table())
    assert ok
    e = entry(cache, 0)
    assert np.all(e[:512] == 0)
    assert np.all(e[512:528].view(np.float32) == np.float32(1.1754944e-38))
    assert np.all(e[528:656] == 0)


def test_power_of_two_scaling_is_exact_without_eps():
    # With eps = 0 the normalised values of x and 2^j x are the same f32 numbers:
    # S scales by 4^j exactly, sqrt and the reciprocal follow exactly.
    rng = np.random.default_rng(1)
    x = round_bf16(rng.standard_normal((1, 512)).astype(np.float32))
    g = round_bf16(1 + 0.1 * rng.standard_normal(512).astype(np.float32))
    kv = np.concatenate([x, x * 4, x / 8])
    ok, cache = run(kv, np.ones((3, 64), np.float32), g, 0.0, [0, 0, 0], identity_table())
    assert ok
    assert np.array_equal(entry(cache, 0)[:528], entry(cache, 1)[:528])
    assert np.array_equal(entry(cache, 0)[:528], entry(cache, 2)[:528])


def test_nope_against_fp64_restatement():
    # y = x / sqrt(mean(x^2) + eps) * g, restated in fp64; the stored value is
    # within e4m3's relative half-step (2^-4) of it, or within half the smallest
    # subnormal step (2^-10 * scale), plus f32 slack.  A large eps on small
    # inputs separates sqrt(ms + eps) from sqrt(ms) + eps; distinct weights
    # pin their indexing; mean over 512 (not 511, not the sum).
    rng = np.random.default_rng(2)
    n = 6
    x = rng.standard_normal((n, 512)).astype(np.float32)
    x[0] *= 0.01
    x[1, ::97] *= 20
    x = round_bf16(x)
    g = round_bf16((0.5 + rng.random(512)).astype(np.float32))
    for eps in (1e-6, 0.5):
        ok, cache = run(x, np.ones((n, 64), np.float32), g, eps, [0] * n, identity_table())
        assert ok
        for t in range(n):
            xd = x[t].astype(np.float64)
            ref = xd / np.sqrt(np.mean(xd * xd) + eps) * g.astype(np.float64)
            e = entry(cache, t)
            got = nope_decoded(e)
            sc = np.repeat(e[512:528].view(np.float32).astype(np.float64), 128)
            tol = 2.0 ** -4 * np.abs(ref) + 2.0 ** -10 * sc + 1e-6 * np.abs(ref)
            assert np.all(np.abs(got - ref) <= tol), (eps, t, np.max(np.abs(got - ref) - tol))


def test_rope_identity_and_quarter_turn():
    rng = np.random.default_rng(3)
    pe = round_bf16(rng.standard_normal((2, 64)).astype(np.float32) + 0.25)
    pe[pe == 0] = 1.0
    table = np.zeros((3, 64), np.float32)
    table[0, :32] = 1.0                    # position 0: cos 1, sin 0
    table[2, 32:] = 1.0                    # position 2: cos 0, sin 1
    ok, cache = run(np.ones((2, 512), np.float32), pe, np.ones(512, np.float32), 1e-6, [0, 2], table)
    assert ok
    assert np.array_equal(entry(cache, 0)[528:656].view(np.uint16), bf16_bits(pe[0]))
    got = rope_values(entry(cache, 1))
    want = np.empty(64, np.float32)
    want[0::2] = -pe[1, 1::2]
    want[1::2] = pe[1, 0::2]
    assert np.array_equal(got, want)  # -0.0 == 0.0 as values


def test_rope_against_fp64_rotation_and_table_indexing():
    # Each pair i at position p uses cos_sin[p, i] and cos_sin[p, 32 + i]: a
    # table with a different angle per (p, i) pins both indices.
    rng = np.random.default_rng(4)
    max_pos, n = 7, 5
    ang = rng.random((max_pos, 32)) * 2 * np.pi
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    pe = round_bf16(rng.standard_normal((n, 64)).astype(np.float32))
    pos = np.array([6, 0, 3, 3, 1])
    ok, cache = run(np.ones((n, 512), np.float32), pe, np.ones(512, np.float32), 1e-6, pos, table)
    assert ok
    for t in range(n):
        c = table[pos[t], :32].astype(np.float64)
        s = table[pos[t], 32:].astype(np.float64)
        x0 = pe[t, 0::2].astype(np.float64)
        x1 = pe[t, 1::2].astype(np.float64)
        ref = np.empty(64)
        ref[0::2] = x0 * c - x1 * s
        ref[1::2] = x0 * s + x1 * c
        got = rope_values(entry(cache, t)).astype(np.float64)
        scale = np.abs(x0).repeat(2) + np.abs(x1).repeat(2)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -22 * scale), t
        # each pair keeps its length (to bf16 precision)
        r0, r1 = got[0::2], got[1::2]
        assert np.allclose(r0 * r0 + r1 * r1, x0 * x0 + x1 * x1, rtol=2 ** -6, atol=1e-12)


def test_rope_bf16_rounds_half_to_even():
    # x0 = 1, x1 = 0, sin 0: r1 = cos exactly.  1 + 2^-8 lies halfway between
    # 1 (even) and 1 + 2^-7 -> 1; 1 + 3 * 2^-8 lies halfway between 1 + 2^-7
    # (odd) and 1 + 2^-6 (even) -> 1 + 2^-6.
    pe = np.zeros((1, 64), np.float32)
    pe[0, 0::2] = 1.0
    table = np.zeros((1, 64), np.float32)
    table[0, :32] = 1.0
    table[0, 0] = 1 + 2.0 ** -8
    table[0, 1] = 1 + 3 * 2.0 ** -8
    table[0, 2] = 1 + 2.0 ** -9
    ok, cache = run(np.ones((1, 512), np.float32), pe, np.ones(512, np.float32), 1e-6, [0], table)
    assert ok
    bits = entry(cache, 0)[528:656].view(np.uint16)
    assert bits[0] == 0x3F80 and bits[2] == 0x3F82 and bits[4] == 0x3F80


def test_skips_negative_slot_and_bad_position():
    kv = np.ones((3, 512), np.float32)
    pe = np.ones((3, 64), np.float32)
    ok, cache = run(kv, pe, np.ones(512, np.float32), 1e-6, [0, 9, 1], identity_table(4),
                    slots=[-1, 1, 2])
    assert not ok                                   # position 9 is outside the 4-row table
    assert np.all(entry(cache, 1) == 0xAB)          # that token is not written
    assert np.all(cache[0, 0] == 0xAB)              # slot 0 was never named
    assert np.all(entry(cache, 2)[:512] == 0x7E)    # the good token is


def test_matches_the_plain_ds_mla_write_when_the_norm_is_exact():
    # With unit weights and tokens whose normalisation is an exact power of two
    # (x_i in {+-2^j}, r = 2^-j), y = x * 2^-j; coding it is the plain ds_mla
    # write of that (bf16-exact) vector, whose oracle is separate code.
    rng = np.random.default_rng(5)
    sign = np.where(rng.random((2, 512)) < 0.5, -1.0, 1.0).astype(np.float32)
    kv = sign * np.array([[4.0], [0.25]], np.float32)
    ok, cache = run(kv, np.ones((2, 64), np.float32), np.ones(512, np.float32), 0.0, [0, 0],
                    identity_table())
    assert ok
    ref = np.full((2, BS, ENTRY), 0xAB, np.uint8)
    oracle.dsmla_quant_write(bf16_bits(sign), bf16_bits(np.ones((2, 64), np.float32)),
                             np.arange(2, dtype=np.int64), ref, BS)
    for t in range(2):
        assert np.array_equal(entry(cache, t), ref[0, t])
