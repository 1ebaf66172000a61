"""GPU parity: indexer-K quant-write, gather, fp8_ds_mla write -- bit-exact
against the oracle on the same seeded inputs."""
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
    m.ix_device_status()  # clear
    return m


def _special_k(n, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(n, 128, generator=g)
    k[3] = 0.0
    k[4] = -0.0
    k[5] *= 1e-38          # bf16 subnormal range
    k[6] *= 1e4
    k[7, 5] = 3e38         # near bf16 max
    k[8] = torch.where(torch.rand(128, generator=g) < 0.5, 1.0, -1.0) * 448.0
    return k.to(torch.bfloat16)


@pytest.mark.parametrize("n,nb,seed", [(1, 2, 0), (37, 3, 1), (1000, 20, 2)])
def test_quant_write_k_bit_exact(dsix, n, nb, seed):
    k = _special_k(max(n, 9), seed)[:n]
    rng = np.random.default_rng(seed)
    slots = rng.permutation(nb * 64)[:n].astype(np.int64)
    if n > 10:
        slots[::7] = -1
    ref = np.zeros((nb, 8448), np.uint8)
    oracle.quant_write_k(W.bf16_bits(k), slots, ref, 64)
    cache = torch.zeros(nb, 8448, dtype=torch.uint8, device="cuda")
    dsix.ix_quant_write_k(k.cuda(), torch.from_numpy(slots).cuda(), cache)
    got = cache.cpu().numpy()
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    assert dsix.ix_device_status() == 0


def test_quant_write_k_prefill_8k(dsix):
    wl = W.prefill_8k()
    ref = np.zeros((wl.num_blocks, 8448), np.uint8)
    oracle.quant_write_k(W.bf16_bits(wl.k_bf16), wl.slot, ref, 64)
    cache = torch.zeros(wl.num_blocks, 8448, dtype=torch.uint8, device="cuda")
    dsix.ix_quant_write_k(wl.k_bf16.cuda(), torch.from_numpy(wl.slot).cuda(), cache)
    assert np.array_equal(cache.cpu().numpy(), ref)


def test_quant_write_k_bad_slot_is_flagged(dsix):
    k = _special_k(9, 3)
    cache = torch.zeros(2, 8448, dtype=torch.uint8, device="cuda")
    slots = torch.tensor([0, 1, 2, 5000, 3, 4, 5, 6, 7], dtype=torch.int64, device="cuda")
    dsix.ix_quant_write_k(k.cuda(), slots, cache)
    assert dsix.ix_device_status() & 1  # IX_DEV_BAD_SLOT
    ref = np.zeros((2, 8448), np.uint8)
    s = slots.cpu().numpy().copy()
    s[3] = -1
    oracle.quant_write_k(W.bf16_bits(k), s, ref, 64)
    assert np.array_equal(cache.cpu().numpy(), ref)


def _filled(nb, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=(nb, 8448), dtype=np.uint8)
    return c


@pytest.mark.parametrize("lens", [[0, 1, 63, 64, 65, 0, 200, 128, 1000], [5], [0, 0, 3]])
def test_gather_bit_exact(dsix, lens):
    nb = sum(-(-s // 64) for s in lens) + 3
    cache = _filled(nb, 1)
    rng = np.random.default_rng(2)
    perm = rng.permutation(nb).astype(np.int32)
    maxb = max(1, max(-(-s // 64) for s in lens))
    bt = np.full((len(lens), maxb + 2), 7, np.int32)
    o = 0
    for b, s in enumerate(lens):
        m = -(-s // 64)
        bt[b, :m] = perm[o:o + m]
        o += m
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    cap = T + 5
    ref_k = np.full((cap, 128), 0xEE, np.uint8)
    ref_s = np.full(cap, -7.0, np.float32)
    oracle.gather_k(cache, 64, 128, bt, cu, ref_k, ref_s)
    gk = torch.full((cap, 128), 0xEE, dtype=torch.uint8, device="cuda")
    gs = torch.full((cap,), -7.0, dtype=torch.float32, device="cuda")
    dsix.ix_gather_k(torch.from_numpy(cache).cuda(), torch.from_numpy(bt).cuda(),
                     torch.from_numpy(cu).cuda(), gk, gs)
    assert np.array_equal(gk.cpu().numpy(), ref_k)
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert dsix.ix_device_status() == 0


def test_gather_after_quant_write_prefill_8k(dsix):
    wl = W.prefill_8k()
    ref_cache = np.zeros((wl.num_blocks, 8448), np.uint8)
    oracle.quant_write_k(W.bf16_bits(wl.k_bf16), wl.slot, ref_cache, 64)
    cu = wl.prefill_gather()
    ref_k = np.zeros((8192, 128), np.uint8)
    ref_s = np.zeros(8192, np.float32)
    oracle.gather_k(ref_cache, 64, 128, wl.prefill_block_table(), cu, ref_k, ref_s)
    cache = torch.zeros(wl.num_blocks, 8448, dtype=torch.uint8, device="cuda")
    dsix.ix_quant_write_k(wl.k_bf16.cuda(), torch.from_numpy(wl.slot).cuda(), cache)
    gk = torch.empty(8192, 128, dtype=torch.uint8, device="cuda")
    gs = torch.empty(8192, dtype=torch.float32, device="cuda")
    dsix.ix_gather_k(cache, torch.from_numpy(wl.prefill_block_table()).cuda(),
                     torch.from_numpy(cu).cuda(), gk, gs)
    assert np.array_equal(gk.cpu().numpy(), ref_k)
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def _dsmla_inputs(n, seed):
    g = torch.Generator().manual_seed(seed)
    nope = torch.randn(n, 512, generator=g)
    out = torch.rand(n, 512, generator=g) < 0.001
    nope = torch.where(out, nope * 20, nope)
    if n > 3:
        nope[1, :128] = 0.0
        nope[2, 256:384] *= 1e-36
        nope[3, 384:] = -0.0
    return nope.to(torch.bfloat16), torch.randn(n, 64, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("n,entry,extra", [(1, 656, 0), (300, 656, 0), (300, 672, 32)])
def test_dsmla_bit_exact(dsix, n, entry, extra):
    nope, rope = _dsmla_inputs(n, n)
    nb, bs = -(-n // 64) + 2, 64
    slots = np.random.default_rng(0).permutation(nb * bs)[:n].astype(np.int64)
    if n > 10:
        slots[::9] = -1
    block_bytes = bs * entry + extra
    base = torch.full((nb * block_bytes,), 0x5C, dtype=torch.uint8, device="cuda")
    view = base.as_strided((nb, bs, entry), (block_bytes, entry, 1))
    ref = np.full(nb * block_bytes, 0x5C, np.uint8)
    # oracle writes into a dense [nb, bs, 656] buffer; place its entries at the strided spots
    dense = np.zeros((nb, bs, 656), np.uint8)
    oracle.dsmla_quant_write(W.bf16_bits(nope), W.bf16_bits(rope), slots, dense, bs)
    for t in range(n):
        if slots[t] < 0:
            continue
        b, o = divmod(int(slots[t]), bs)
        ref[b * block_bytes + o * entry:b * block_bytes + o * entry + 656] = dense[b, o]
    import deepseek_v3_sparse_gb300 as m
    d_nope, d_rope, d_slots = nope.cuda(), rope.cuda(), torch.from_numpy(slots).cuda()
    rc = m.load().dsmla_quant_write(d_nope.data_ptr(), d_rope.data_ptr(), n, d_slots.data_ptr(),
                                    base.data_ptr(), nb, bs, block_bytes, entry,
                                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    got = base.cpu().numpy()
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    del view


def test_dsmla_mixed_long_new_tokens(dsix):
    wl = W.mixed_long()
    nb = wl.num_blocks
    cache = torch.zeros(nb, 64, 656, dtype=torch.uint8, device="cuda")
    slots = torch.from_numpy(wl.new_slot.copy()).cuda()
    dsix.dsmla_quant_write(wl.nope_bf16.cuda(), wl.rope_bf16.cuda(), slots, cache)
    got = cache.view(-1, 656)[slots].cpu().numpy()
    # oracle on a compact pool: entry i of the new tokens at slot i
    n = len(wl.new_slot)
    dense = np.zeros((-(-n // 64), 64, 656), np.uint8)
    oracle.dsmla_quant_write(W.bf16_bits(wl.nope_bf16), W.bf16_bits(wl.rope_bf16),
                             np.arange(n, dtype=np.int64), dense, 64)
    assert np.array_equal(got, dense.reshape(-1, 656)[:n])


def _near_midpoint_tokens(n, seed):
    """Tokens whose quotients x / scale sit on or next to e4m3 rounding
    boundaries (midpoints between neighbouring codes, ties to even): token t
    has amax 448 * s_t, and its other values are bf16 roundings of
    (midpoint +- a few f32 ulps) * s_t for every normal e4m3 binade."""
    rng = np.random.default_rng(seed)
    mids = []
    for e in range(-6, 9):              # e4m3 normal binades
        for m in range(8):
            mids.append((1 + (2 * m + 1) / 16.0) * 2.0 ** e)
    mids = np.array([v for v in mids if v < 448], np.float64)
    k = np.zeros((n, 128), np.float32)
    for t in range(n):
        # t % 3 == 0: scale exactly 1; == 1: a power of two (quotients land exactly on
        # midpoints: ties to even); == 2: any scale
        s = 1.0 if t % 3 == 0 else 2.0 ** rng.integers(-8, 4) * (1.0 if t % 3 == 1 else 1 + rng.random())
        vals = mids[rng.integers(0, len(mids), 127)] * s * (1 + (rng.integers(-3, 4, 127) * 2.0 ** -24))
        vals *= np.where(rng.random(127) < 0.5, -1, 1)
        k[t, 0] = 448.0 * s
        k[t, 1:] = vals
    return torch.from_numpy(k).to(torch.bfloat16)


def test_quant_write_k_near_rounding_boundaries(dsix):
    """The codes of quotients on and beside e4m3 midpoints match the oracle's
    correctly rounded division (the kernels divide by multiplying with the
    reciprocal except near such boundaries)."""
    n = 600
    k = _near_midpoint_tokens(n, 5)
    slots = np.arange(n, dtype=np.int64)
    nb = -(-n // 64)
    cache = torch.zeros(nb, 64 * 132, dtype=torch.uint8, device="cuda")
    dsix.ix_quant_write_k(k.cuda(), torch.from_numpy(slots).cuda(), cache)
    torch.cuda.synchronize()
    ref = np.zeros((nb, 64 * 132), np.uint8)
    oracle.quant_write_k(W.bf16_bits(k), slots, ref, 64)
    assert np.array_equal(cache.cpu().numpy(), ref)
    # the same values through the indexer-query coding (one scale per 128 values)
    w = torch.ones(n, 1)
    qf = torch.empty(n, 1, 128, dtype=torch.uint8, device="cuda")
    wo = torch.empty(n, 1, device="cuda")
    dsix.ix_quant_q(k.view(n, 1, 128).cuda(), w.cuda(), qf, wo)
    torch.cuda.synchronize()
    rq, rw = oracle.quant_q(W.bf16_bits(k.view(n, 1, 128)), w.numpy())
    assert np.array_equal(qf.cpu().numpy(), rq) and np.array_equal(wo.cpu().numpy(), rw)
    assert dsix.ix_device_status() == 0
