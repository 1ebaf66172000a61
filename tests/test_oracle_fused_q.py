"""Pins of the oracle's query side (CPU only).

* ``fused_q``: vLLM PR #47090 (prhub summary) gives fused_q a quantize_mqa flag:
  an FP8 MQA query, or the BF16 pair (ql_nope, q_pe).  The page prints no
  formula; the readings (rotation as the cache's RoPE values, one amax/448
  scale per (token, head) over the 576 values) are in the oracle's header.
* ``quant_q``: the indexer's fp8 query with its per-(token, head) scale folded
  into the head weight, from the indexer score k_scale * sum_h w_h *
  ReLU(q_h . k) and ReLU(s x) = s ReLU(x) for s > 0.

Each check is pinned to something other than the oracle itself: closed forms,
exact invariances, numpy's IEEE f32 division with torch's own fp8 cast, an fp64
restatement of the rotation, and the indexer score restated in float64.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")
FLT_MIN = np.float32(1.1754944e-38)


def bf16_bits(x):
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "test inputs must be exact bf16 values"
    return (u >> 16).astype(np.uint16)


def bf16_values(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).float().numpy()


def torch_codes(v):
    """fp8 codes of f32 values by torch's own cast (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def independent_quant(v):
    """amax / 448 in IEEE f32 (numpy), floored at FLT_MIN; codes of v / s by torch."""
    amax = np.abs(v).max(axis=-1, keepdims=True).astype(np.float32)
    s = np.maximum(amax / np.float32(448.0), FLT_MIN).astype(np.float32)
    return torch_codes((v / s).astype(np.float32)), s[..., 0]


def dec(codes):
    return np.array([oracle.e4m3_decode(int(c)) for c in np.asarray(codes).ravel()]).reshape(np.shape(codes))


# ---------------------------------------------------------------------------
# indexer query + folded weights
# ---------------------------------------------------------------------------
def test_quant_q_constant_vector_closed_form():
    q = np.full((1, 2, 128), 0.375, np.float32)
    q[0, 1] = -3.0
    w = np.array([[0.5, -0.25]], np.float32)
    codes, w_out = oracle.quant_q(bf16_bits(q), w)
    assert (codes[0, 0] == 0x7E).all() and (codes[0, 1] == 0xFE).all()   # +448 / -448
    s = np.array([np.float32(0.375) / np.float32(448), np.float32(3.0) / np.float32(448)], np.float32)
    assert np.array_equal(w_out[0], (w[0] * s).astype(np.float32))


def test_quant_q_zero_head_takes_the_floor_scale():
    q = np.zeros((2, 3, 128), np.float32)
    w = np.full((2, 3), 2.0, np.float32)
    codes, w_out = oracle.quant_q(bf16_bits(q), w)
    assert (codes == 0).all()
    assert np.array_equal(w_out, np.full((2, 3), np.float32(2.0) * FLT_MIN, np.float32))


def test_quant_q_matches_numpy_division_and_torch_cast():
    q = rand_bf16((7, 64, 128), seed=3)
    q[0, 0, 5] = 40.0  # an outlier
    w = (rand_bf16((7, 64), seed=4) / 8).astype(np.float32)
    codes, w_out = oracle.quant_q(bf16_bits(q), w)
    ref_codes, s = independent_quant(q)
    assert np.array_equal(codes, ref_codes)
    assert np.array_equal(w_out, (w * s).astype(np.float32))
    # the amax element of every head codes to +-448
    idx = np.abs(q).argmax(axis=-1)
    top = np.take_along_axis(codes, idx[..., None], -1)[..., 0]
    assert np.isin(top, [0x7E, 0xFE]).all()


def test_quant_q_divides_by_448():
    """The scale is amax / 448, not amax * f32(1/448) (they differ for some amax)."""
    inv = np.float32(1.0 / 448.0)
    cand = bf16_values(np.arange(0x3F80, 0x4000, dtype=np.uint16))  # bf16 values in [1, 2)
    diff = cand[(cand / np.float32(448)) != (cand * inv)]
    assert diff.size > 0
    a = diff[0]
    q = np.zeros((1, 1, 128), np.float32)
    q[0, 0, 0] = a
    _, w_out = oracle.quant_q(bf16_bits(q), np.ones((1, 1), np.float32))
    assert w_out[0, 0] == np.float32(a) / np.float32(448) and w_out[0, 0] != np.float32(a) * inv


def test_quant_q_power_of_two_invariance():
    q = rand_bf16((3, 4, 128), seed=5)
    w = np.ones((3, 4), np.float32)
    c1, w1 = oracle.quant_q(bf16_bits(q), w)
    c2, w2 = oracle.quant_q(bf16_bits(q * 8.0), w)
    assert np.array_equal(c1, c2)
    assert np.array_equal(w2, w1 * np.float32(8.0))


def test_quant_q_round_trip_error_bound():
    q = rand_bf16((4, 8, 128), seed=6, scale=3.0)
    codes, w_out = oracle.quant_q(bf16_bits(q), np.ones((4, 8), np.float32))
    s = w_out[..., None].astype(np.float64)
    x = dec(codes) * s
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals; near zero
    # the subnormal step 2^-9 * s bounds the absolute error by 2^-10 * s
    err = np.abs(x - q)
    assert np.all(err <= np.maximum(np.abs(q) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-12))


def test_quant_q_folding_reproduces_the_indexer_score():
    """Logits of (q_fp8, w_out) = the score of the dequantised query with the
    original weight, sum_h w_h ReLU((s_h q_fp8_h) . k) * k_scale, in float64."""
    T, H, D, K = 3, 64, 128, 50
    q = rand_bf16((T, H, D), seed=7)
    w = (rand_bf16((T, H), seed=8) / 8).astype(np.float32)
    codes, w_out = oracle.quant_q(bf16_bits(q), w)
    g = torch.Generator().manual_seed(9)
    k = torch.randn(K, D, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ksc = (np.random.default_rng(1).random(K) * 0.01 + 1e-3).astype(np.float32)
    ks = np.zeros(T, np.int32)
    ke = np.full(T, K, np.int32)
    got = oracle.mqa_logits(codes, w_out, k, ksc, ks, ke, ld=52)
    s = w_out.astype(np.float64) / w.astype(np.float64)       # the per-head scales
    qd = dec(codes) * s[..., None]
    kd = dec(k)
    ref = np.einsum("thd,sd->ths", qd, kd)
    ref = (np.maximum(ref, 0.0) * w[..., None].astype(np.float64)).sum(axis=1) * ksc[None, :]
    tol = 1e-6 * np.abs(ref).max(axis=1, keepdims=True)
    assert np.all(np.abs(got[:, :K] - ref) <= tol)


# ---------------------------------------------------------------------------
# fused_q: rotation and quantize_mqa
# ---------------------------------------------------------------------------
def _table(max_pos, seed):
    ang = np.random.default_rng(seed).random((max_pos, 32)) * 2 * np.pi
    return np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)


def test_fused_q_identity_and_quarter_turn_are_exact():
    T, H = 2, 3
    qn = rand_bf16((T, H, 512), seed=10)
    qp = rand_bf16((T, H, 64), seed=11)
    table = np.zeros((2, 64), np.float32)
    table[0, :32] = 1.0             # position 0: c = 1, s = 0
    table[1, 32:] = 1.0             # position 1: c = 0, s = 1
    out, _, _, ok = oracle.fused_q(bf16_bits(qn), bf16_bits(qp), np.array([0, 1]), table, False)
    assert ok
    assert np.array_equal(out[0], bf16_bits(qp[0]))
    x0, x1 = qp[1][..., 0::2], qp[1][..., 1::2]
    quarter = np.empty_like(qp[1])
    quarter[..., 0::2] = -x1
    quarter[..., 1::2] = x0
    assert np.array_equal(out[1], bf16_bits(quarter))


def test_fused_q_rotation_against_fp64_and_table_rows():
    T, H, P = 5, 4, 9
    qn = rand_bf16((T, H, 512), seed=12)
    qp = rand_bf16((T, H, 64), seed=13)
    table = _table(P, 14)
    pos = np.array([8, 0, 3, 3, 5])
    out, _, _, ok = oracle.fused_q(bf16_bits(qn), bf16_bits(qp), pos, table, False)
    assert ok
    got = bf16_values(out).astype(np.float64)
    c = table[pos][:, None, :32].astype(np.float64)
    s = table[pos][:, None, 32:].astype(np.float64)
    x0, x1 = qp[..., 0::2].astype(np.float64), qp[..., 1::2].astype(np.float64)
    r = np.empty_like(got)
    r[..., 0::2] = x0 * c - x1 * s
    r[..., 1::2] = x0 * s + x1 * c
    # one bf16 rounding (2^-9 relative) plus the f32 products and sum
    assert np.all(np.abs(got - r) <= 2.0 ** -8 * np.abs(r) + 1e-6)


def test_fused_q_quantize_matches_numpy_division_and_torch_cast():
    T, H, P = 3, 5, 4
    qn = rand_bf16((T, H, 512), seed=15)
    qn[1, 2, 100] = -60.0
    qp = rand_bf16((T, H, 64), seed=16)
    table = _table(P, 17)
    pos = np.array([1, 3, 0])
    rot, _, _, ok0 = oracle.fused_q(bf16_bits(qn), bf16_bits(qp), pos, table, False)
    _, codes, scale, ok1 = oracle.fused_q(bf16_bits(qn), bf16_bits(qp), pos, table, True)
    assert ok0 and ok1
    v = np.concatenate([qn, bf16_values(rot)], axis=-1)          # [ql_nope | rotated q_pe]
    ref_codes, ref_s = independent_quant(v)
    assert np.array_equal(codes, ref_codes)
    assert np.array_equal(scale, ref_s)
    idx = np.abs(v).argmax(axis=-1)
    assert np.isin(np.take_along_axis(codes, idx[..., None], -1), [0x7E, 0xFE]).all()
    # the fp8 query decodes to the bf16 pair within e4m3's rounding
    x = dec(codes) * scale[..., None].astype(np.float64)
    assert np.all(np.abs(x - v) <= np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * scale[..., None]) * (1 + 1e-12))


def test_fused_q_zero_head_and_bad_position():
    T, H = 3, 2
    qn = np.zeros((T, H, 512), np.float32)
    qp = np.zeros((T, H, 64), np.float32)
    qn[2] = 1.0
    table = _table(4, 18)
    _, codes, scale, ok = oracle.fused_q(bf16_bits(qn), bf16_bits(qp), np.array([0, 1, 7]), table, True)
    assert not ok                                   # position 7 is outside the table
    # all values zero (the rotation may give -0.0, coded 0x80): every code decodes to 0
    assert (dec(codes[0]) == 0).all() and np.isin(codes[0], [0x00, 0x80]).all()
    assert (scale[0] == FLT_MIN).all()
    assert (codes[2] == 0).all() and (scale[2] == 0).all()   # the skipped token is untouched
