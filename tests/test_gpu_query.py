"""GPU parity: the query side -- dsmla_fused_q (RoPE of q_pe; with quantize_mqa
the 576-wide fp8 MQA query and its per-(token, head) scale) and ix_quant_q
(the indexer's fp8 query with the scale folded into the head weight).

Both are bit-exact against the oracle: codes, scales, weights and rotated bf16
values.  Shapes: the decode batch (16 tokens) and the prefill chunk (8192
tokens) x 128 query heads for fused_q; 256 (the MTP decode batch) and 8192
tokens x 64 indexer heads for quant_q, with sampled tokens where the oracle
would take minutes.  Edge cases: zero heads, outliers, a position outside the
table, odd head counts, the last half-warp of an odd (token, head) count.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsix():
    require_gpu()
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v3_sparse_gb300 as m
    m.ix_device_status()
    return m


def _bits(x):
    return W.bf16_bits(x)


def _inputs(T, H, seed, max_pos=4096):
    g = torch.Generator().manual_seed(seed)
    qn = torch.randn(T, H, 512, generator=g)
    out = torch.rand(T, H, 512, generator=g) < 0.001
    qn = torch.where(out, qn * 20, qn).to(torch.bfloat16)
    qp = torch.randn(T, H, 64, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, max_pos, (T,), generator=g, dtype=torch.int64)
    _, table = W.norm_rope_params(max_pos, seed=seed)
    return qn, qp, pos, table


def _fused_gpu(dsix, qn, qp, pos, table, quantize):
    T, H = qp.shape[:2]
    if quantize:
        out = torch.full((T, H, 576), 0xAB, dtype=torch.uint8, device="cuda")
        sc = torch.full((T, H), -1.0, device="cuda")
        dsix.dsmla_fused_q(qp.cuda(), pos.cuda(), table.cuda(), True, ql_nope_bf16=qn.cuda(), out_mqa=out,
                           out_scale=sc)
        return out.cpu().numpy(), sc.cpu().numpy()
    out = torch.full((T, H, 64), -7.0, dtype=torch.bfloat16, device="cuda")
    dsix.dsmla_fused_q(qp.cuda(), pos.cuda(), table.cuda(), False, out_pe=out)
    return _bits(out.cpu()), None


@pytest.mark.parametrize("T,H", [(16, 128), (5, 3), (1, 1)])
@pytest.mark.parametrize("quantize", [False, True])
def test_fused_q_exact(dsix, T, H, quantize):
    qn, qp, pos, table = _inputs(T, H, seed=T * 7 + H)
    if T > 1:
        qn[1, 0] = 0.0
        qp[1, 0] = 0.0            # a zero head: floor scale, all codes zero (+-0)
    got, gsc = _fused_gpu(dsix, qn, qp, pos, table, quantize)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    ref_pe, ref_mqa, ref_sc, ok = oracle.fused_q(_bits(qn), _bits(qp), pos.numpy(), table.numpy(), quantize)
    assert ok
    if quantize:
        assert np.array_equal(got, ref_mqa)
        assert np.array_equal(gsc.view(np.uint32), ref_sc.view(np.uint32))
    else:
        assert np.array_equal(got, ref_pe)


@pytest.mark.parametrize("quantize", [False, True])
def test_fused_q_prefill_chunk_sampled(dsix, quantize):
    """8192 tokens x 128 heads in one launch; the oracle checks 96 sampled tokens."""
    T, H = 8192, 128
    qn, qp, pos, table = _inputs(T, H, seed=41, max_pos=8192)
    got, gsc = _fused_gpu(dsix, qn, qp, pos, table, quantize)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    rows = np.unique(np.concatenate([[0, 1, T - 1], np.random.default_rng(2).integers(0, T, 93)]))
    sel = torch.from_numpy(rows)
    ref_pe, ref_mqa, ref_sc, ok = oracle.fused_q(_bits(qn[sel]), _bits(qp[sel]), pos.numpy()[rows], table.numpy(),
                                                 quantize)
    assert ok
    if quantize:
        assert np.array_equal(got[rows], ref_mqa) and np.array_equal(gsc[rows], ref_sc)
    else:
        assert np.array_equal(got[rows], ref_pe)


def test_fused_q_bad_position_is_flagged_and_skipped(dsix):
    T, H = 4, 8
    qn, qp, pos, table = _inputs(T, H, seed=5, max_pos=16)
    pos[2] = 16                          # one past the table
    got, gsc = _fused_gpu(dsix, qn, qp, pos, table, True)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() & 32  # IX_DEV_BAD_POSITION
    assert (got[2] == 0xAB).all() and (gsc[2] == -1.0).all()
    keep = np.array([0, 1, 3])
    _, ref_mqa, ref_sc, ok = oracle.fused_q(_bits(qn[keep]), _bits(qp[keep]), pos.numpy()[keep], table.numpy(), True)
    assert ok and np.array_equal(got[keep], ref_mqa) and np.array_equal(gsc[keep], ref_sc)


def _quant_inputs(T, H, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, 128, generator=g)
    out = torch.rand(T, H, 128, generator=g) < 0.001
    q = torch.where(out, q * 20, q).to(torch.bfloat16)
    w = torch.randn(T, H, generator=g) / 8
    return q, w


def _quant_gpu(dsix, q, w):
    T, H, D = q.shape
    qf = torch.full((T, H, D), 0xAB, dtype=torch.uint8, device="cuda")
    wo = torch.full((T, H), -1.0, device="cuda")
    dsix.ix_quant_q(q.cuda(), w.cuda(), qf, wo)
    torch.cuda.synchronize()
    return qf.cpu().numpy(), wo.cpu().numpy()


@pytest.mark.parametrize("T,H", [(256, 64), (3, 1), (7, 3)])
def test_quant_q_exact(dsix, T, H):
    q, w = _quant_inputs(T, H, seed=T + H)
    q[0, 0] = 0.0
    gq, gw = _quant_gpu(dsix, q, w)
    assert dsix.ix_device_status() == 0
    rq, rw = oracle.quant_q(_bits(q), w.numpy())
    assert np.array_equal(gq, rq)
    assert np.array_equal(gw.view(np.uint32), rw.view(np.uint32))


def test_quant_q_prefill_chunk_sampled_and_logits(dsix):
    """8192 tokens x 64 heads; sampled tokens bit-exact, and the logits of the
    GPU's (q_fp8, w_out) over a few keys equal the oracle's logits of the
    oracle's own (q_fp8, w_out) within the indexer tolerance."""
    T, H = 8192, 64
    q, w = _quant_inputs(T, H, seed=77)
    gq, gw = _quant_gpu(dsix, q, w)
    rows = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(3).integers(0, T, 254)]))
    sel = torch.from_numpy(rows)
    rq, rw = oracle.quant_q(_bits(q[sel]), w.numpy()[rows])
    assert np.array_equal(gq[rows], rq) and np.array_equal(gw[rows], rw)
    g = torch.Generator().manual_seed(5)
    K = 300
    k = torch.randn(K, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    ksc = torch.rand(K, generator=g) * 0.01 + 1e-3
    ks = torch.zeros(len(rows), dtype=torch.int32)
    ke = torch.full((len(rows),), K, dtype=torch.int32)
    out = torch.empty(len(rows), 300, device="cuda")
    dsix.ix_mqa_logits(torch.from_numpy(gq[rows]).cuda(), torch.from_numpy(gw[rows]).cuda(), k.cuda(), ksc.cuda(),
                       ks.cuda(), ke.cuda(), out)
    ref = oracle.mqa_logits(rq, rw, k.numpy(), ksc.numpy(), ks.numpy(), ke.numpy(), ld=300)
    got = out.cpu().numpy()
    tol = 1e-3 * np.abs(ref).max(axis=1, keepdims=True) + 1e-4
    assert np.all(np.abs(got - ref) <= tol)
    assert dsix.ix_device_status() == 0


def _bf16_from_fields(sign, exp, man):
    bits = (np.asarray(sign, np.uint16) << 15) | (np.asarray(exp, np.uint16) << 7) | np.asarray(man, np.uint16)
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


# Exponents of the largest value of a (token, head): ordinary, near the smallest
# scale that takes the reciprocal path (2^-90), below it, and large.
_AMAX_EXPS = [3, -80, -100, 100]


def test_fused_q_every_significand_pair(dsix):
    """The codes are quotients x / scale with scale = RN(amax / 448); their
    rounding depends only on the significands of x and amax (no quantity here
    under- or overflows).  Head h of each token holds amax = (1 + h/128) 2^E in
    slot 0 and, in the other 511 NoPE slots, all 128 bf16 significands at
    2^(E-1) .. 2^(E-4) with both signs, so the 128 heads cover every
    (x, amax) significand pair; E runs over both division paths.  Slot 1 holds
    -0 or +0 (codes 0x80 / 0x00)."""
    T, H = len(_AMAX_EXPS), 128
    sign = np.zeros((T, H, 512), np.uint16)
    exp = np.zeros((T, H, 512), np.uint16)
    man = np.zeros((T, H, 512), np.uint16)
    s = np.arange(512)
    for t, E in enumerate(_AMAX_EXPS):
        off = np.where(s == 0, 0, 1 + s // 128)
        exp[t] = (E + 127 - off)[None, :]
        man[t] = np.where(s == 0, np.arange(H)[:, None], (s % 128)[None, :])
        sign[t] = np.where(s == 0, 0, (s // 128) & 1)[None, :]
    exp[:, :, 1], man[:, :, 1], sign[:, :, 1] = 0, 0, np.arange(H) & 1  # zeros of both signs
    qn = _bf16_from_fields(sign, exp, man)
    qp = torch.zeros(T, H, 64, dtype=torch.bfloat16)
    pos = torch.arange(T, dtype=torch.int64)
    _, table = W.norm_rope_params(16, seed=1)
    got, gsc = _fused_gpu(dsix, qn, qp, pos, table, True)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    _, ref_mqa, ref_sc, ok = oracle.fused_q(_bits(qn), _bits(qp), pos.numpy(), table.numpy(), True)
    assert ok
    assert np.array_equal(gsc.view(np.uint32), ref_sc.view(np.uint32))
    bad = np.argwhere(got != ref_mqa)
    assert bad.size == 0, f"{len(bad)} codes differ, first (token, head, slot) {bad[:4].tolist()}"


def test_quant_q_every_significand_pair(dsix):
    """As above for the indexer query (128 values per head): amax significand
    (64 g + h) in slot 0 of head h of token group g, the other 127 slots all
    significands but one at 2^(E-1-v) with sign (-1)^v, for v = 0, 1."""
    H = 64
    rows = []
    for E in _AMAX_EXPS:
        for g in range(2):
            for v in range(2):
                s = np.arange(128)
                man = np.where(s == 0, (64 * g + np.arange(H))[:, None], s[None, :])
                exp = np.where(s == 0, E + 127, E + 126 - v)[None, :].repeat(H, 0)
                sign = np.where(s == 0, 0, v)[None, :].repeat(H, 0)
                rows.append((sign, exp, man))
    sign = np.stack([r[0] for r in rows])
    exp = np.stack([r[1] for r in rows])
    man = np.stack([r[2] for r in rows])
    exp[:, :, 1], man[:, :, 1], sign[:, :, 1] = 0, 0, np.arange(H) & 1  # zeros of both signs
    q = _bf16_from_fields(sign, exp, man)
    w = torch.linspace(-1, 1, q.shape[0] * H).view(q.shape[0], H)
    gq, gw = _quant_gpu(dsix, q, w)
    assert dsix.ix_device_status() == 0
    rq, rw = oracle.quant_q(_bits(q), w.numpy())
    assert np.array_equal(gw.view(np.uint32), rw.view(np.uint32))
    bad = np.argwhere(gq != rq)
    assert bad.size == 0, f"{len(bad)} codes differ, first (token, head, slot) {bad[:4].tolist()}"
