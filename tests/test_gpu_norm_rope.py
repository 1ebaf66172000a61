"""GPU parity: the fused RMSNorm + RoPE + fp8_ds_mla write (dsmla_norm_rope_write)
against the oracle, bit for bit, on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._helpers import require_gpu

pytestmark = pytest.mark.gpu

IX_DEV_BAD_POSITION = 32


@pytest.fixture(scope="module")
def dsix():
    require_gpu()
    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v3_sparse_gb300 as m
    m.ix_device_status()  # clear
    return m


def _inputs(n, seed):
    g = torch.Generator().manual_seed(seed)
    kv = torch.randn(n, 512, generator=g)
    out = torch.rand(n, 512, generator=g) < 0.001
    kv = torch.where(out, kv * 20, kv)
    if n > 4:
        kv[1] = 0.0                  # zero token: floor scales, zero codes
        kv[2, 256:384] *= 1e-30      # a tile far below the others
        kv[3] = 0.75                 # constant token (closed form: all codes 0x7E)
        kv[4, :128] = -0.0
    pe = torch.randn(n, 64, generator=g)
    return kv.to(torch.bfloat16), pe.to(torch.bfloat16)


def _run_both(dsix, kv, pe, gamma, eps, pos, table, slots, nb, bs, entry, extra):
    n = kv.shape[0]
    block_bytes = bs * entry + extra
    base = torch.full((nb * block_bytes,), 0x5C, dtype=torch.uint8, device="cuda")
    dense = np.full((nb, bs, 656), 0x5C, np.uint8)
    ok = oracle.dsmla_norm_rope_write(W.bf16_bits(kv), W.bf16_bits(pe), W.bf16_bits(gamma), eps,
                                      pos, table.numpy(), slots, dense, bs)
    ref = np.full(nb * block_bytes, 0x5C, np.uint8)
    for t in range(n):
        if slots[t] < 0:
            continue
        b, o = divmod(int(slots[t]), bs)
        ref[b * block_bytes + o * entry:b * block_bytes + o * entry + 656] = dense[b, o]
    d = [x.cuda() for x in (kv, pe, gamma)]
    d_pos, d_tab, d_slots = (torch.from_numpy(pos).cuda(), table.cuda(),
                             torch.from_numpy(slots).cuda())
    rc = dsix.load().dsmla_norm_rope_write(
        d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), eps, d_pos.data_ptr(), d_tab.data_ptr(),
        table.shape[0], d_slots.data_ptr(), n, base.data_ptr(), nb, bs, block_bytes, entry,
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    return ok, base.cpu().numpy(), ref


@pytest.mark.parametrize("n,entry,extra,eps", [(1, 656, 0, 1e-6), (300, 656, 0, 1e-6),
                                               (300, 672, 32, 1e-6), (2000, 656, 0, 0.5)])
def test_norm_rope_bit_exact(dsix, n, entry, extra, eps):
    kv, pe = _inputs(n, n)
    gamma, table = W.norm_rope_params(4096, seed=n)
    rng = np.random.default_rng(n)
    pos = rng.integers(0, 4096, n).astype(np.int64)
    nb, bs = -(-n // 64) + 2, 64
    slots = rng.permutation(nb * bs)[:n].astype(np.int64)
    if n > 10:
        slots[::9] = -1
    ok, got, ref = _run_both(dsix, kv, pe, gamma, eps, pos, table, slots, nb, bs, entry, extra)
    assert ok
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    assert dsix.ix_device_status() == 0


def test_norm_rope_bad_position_is_flagged_and_skipped(dsix):
    n = 64
    kv, pe = _inputs(n, 7)
    gamma, table = W.norm_rope_params(128, seed=7)
    pos = np.arange(n, dtype=np.int64) * 2
    pos[5] = 128            # one past the table
    pos[9] = -3
    slots = np.arange(n, dtype=np.int64)
    ok, got, ref = _run_both(dsix, kv, pe, gamma, 1e-6, pos, table, slots, 2, 64, 656, 0)
    assert not ok           # the oracle reports the skipped tokens too
    assert np.array_equal(got, ref)
    assert np.all(got[5 * 656:6 * 656] == 0x5C) and np.all(got[9 * 656:10 * 656] == 0x5C)
    assert dsix.ix_device_status() == IX_DEV_BAD_POSITION
    assert dsix.ix_device_status() == 0  # read-and-clear


def test_norm_rope_mixed_long_new_tokens(dsix):
    # the 8208 new tokens of the long-context mixed step at their own positions
    wl = W.mixed_long()
    pos = wl.new_positions()
    gamma, table = W.norm_rope_params(int(pos.max()) + 1)
    cache = torch.zeros(wl.num_blocks, 64, 656, dtype=torch.uint8, device="cuda")
    slots = torch.from_numpy(wl.new_slot.copy()).cuda()
    dsix.dsmla_norm_rope_write(wl.nope_bf16.cuda(), wl.rope_bf16.cuda(), gamma.cuda(), 1e-6,
                               torch.from_numpy(pos).cuda(), table.cuda(), slots, cache)
    torch.cuda.synchronize()
    got = cache.view(-1, 656)[slots].cpu().numpy()
    n = len(pos)
    dense = np.zeros((-(-n // 64), 64, 656), np.uint8)
    assert oracle.dsmla_norm_rope_write(W.bf16_bits(wl.nope_bf16), W.bf16_bits(wl.rope_bf16),
                                        W.bf16_bits(gamma), 1e-6, pos, table.numpy(),
                                        np.arange(n, dtype=np.int64), dense, 64)
    assert np.array_equal(got, dense.reshape(-1, 656)[:n])
    assert dsix.ix_device_status() == 0


def test_norm_rope_empty_is_a_no_op(dsix):
    gamma, table = W.norm_rope_params(4)
    cache = torch.full((1, 64, 656), 7, dtype=torch.uint8, device="cuda")
    e = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    dsix.dsmla_norm_rope_write(e, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"),
                               gamma.cuda(), 1e-6, torch.empty(0, dtype=torch.int64, device="cuda"),
                               table.cuda(), torch.empty(0, dtype=torch.int64, device="cuda"), cache)
    torch.cuda.synchronize()
    assert bool((cache == 7).all())


@pytest.mark.parametrize("bs,entry,extra", [(16, 656, 0), (48, 672, 16)])
def test_norm_rope_other_block_sizes_and_edge_positions(dsix, bs, entry, extra):
    n = 257
    kv, pe = _inputs(n, bs)
    gamma, table = W.norm_rope_params(97, seed=bs)
    rng = np.random.default_rng(bs)
    pos = rng.integers(0, 97, n).astype(np.int64)
    pos[:3] = [0, 96, 96]                       # the table's first and last rows
    nb = -(-n // bs) + 3
    slots = rng.permutation(nb * bs)[:n].astype(np.int64)
    slots[7::11] = -1
    ok, got, ref = _run_both(dsix, kv, pe, gamma, 1e-6, pos, table, slots, nb, bs, entry, extra)
    assert ok
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    assert dsix.ix_device_status() == 0


def test_wide_dynamic_range_tokens_match(dsix):
    """Tokens whose values span 2^0 down to 2^-60 (squares more than 2^38 apart):
    the kernel's fixed-point sum of squares cuts squares below 2^-38 of the
    largest one's binade, the oracle's double sum keeps them while it can; the
    difference stays far inside one rounding of t = f32(S/512 + eps), so the
    bytes agree."""
    n = 64
    g = torch.Generator().manual_seed(3)
    exps = torch.arange(512) % 61                       # 2^0 .. 2^-60 across each token
    mant = 1 + torch.rand(n, 512, generator=g)
    sign = torch.where(torch.rand(n, 512, generator=g) < 0.5, -1.0, 1.0)
    kv = (sign * mant * torch.pow(2.0, -exps.float())).to(torch.bfloat16)
    kv[1] = 0.0
    kv[1, 0] = 1.0
    kv[1, 1:] = torch.pow(2.0, -torch.arange(40, 40 + 511).float().clamp(max=120)).to(torch.bfloat16)
    kv[2] = (torch.pow(2.0, -torch.arange(512).float() % 100) * 3).to(torch.bfloat16)
    pe = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    gamma, table = W.norm_rope_params(256, seed=3)
    pos = np.arange(n, dtype=np.int64)
    slots = np.arange(n, dtype=np.int64)
    for eps in (1e-6, 0.0):
        ok, got, ref = _run_both(dsix, kv, pe, gamma, eps, pos, table, slots, 2, 64, 656, 0)
        assert ok
        assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    assert dsix.ix_device_status() == 0
