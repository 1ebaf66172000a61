"""GPU parity: top-k + remap.

* On the oracle's own f32 logits the GPU result must match the oracle exactly
  (local and global indices, ties to the lower index, -0.0 == +0.0, padding).
* Row lengths cover every cluster split (1/2/4/8 CTAs per row), short rows,
  L = k, L = k + 1, L = 0, and 131072-key rows.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _run(dsix, logits, row_len, row_req, bt, k, bs=64):
    R, ld = logits.shape
    dl = torch.from_numpy(logits).cuda()
    loc = torch.full((R, k), -5, dtype=torch.int32, device="cuda")
    glb = torch.full((R, k), -5, dtype=torch.int32, device="cuda")
    dsix.ix_topk_to_global(dl, torch.from_numpy(row_len).cuda(), torch.from_numpy(row_req).cuda(),
                           torch.from_numpy(bt).cuda(), k, glb, loc, block_size=bs)
    return loc.cpu().numpy(), glb.cpu().numpy()


def _table(R, ld, bs, seed):
    nblk = -(-ld // bs)
    return np.random.default_rng(seed).permutation(R * nblk).reshape(R, nblk).astype(np.int32)


def _exact(dsix, logits, row_len, k, bs=64, seed=0):
    R, ld = logits.shape
    bt = _table(R, ld, bs, seed)
    row_req = np.arange(R, dtype=np.int32)[::-1].copy()
    loc, glb = _run(dsix, logits, row_len, row_req, bt, k, bs)
    rl, rg = oracle.topk_to_global(logits, row_len, row_req, bt, bs, k)
    bad = np.nonzero((loc != rl).any(axis=1) | (glb != rg).any(axis=1))[0]
    assert bad.size == 0, f"rows {bad[:5]} differ"


# (R >= 2 x SMs with ld <= 16384 runs one CTA per row with no cluster; the others run the cluster kernel)
@pytest.mark.parametrize("ld,R", [(64, 5), (4096, 40), (8192, 300), (20000, 8), (131072, 4),
                                  (64, 400), (8192, 640), (16384, 320)])
def test_exact_on_oracle_like_logits(dsix, ld, R):
    rng = np.random.default_rng(ld)
    logits = (rng.standard_normal((R, ld)) * 3).astype(np.float32)
    logits[:, ::5] = np.round(logits[:, ::5] * 4) / 4   # many exact ties
    logits[0, :ld // 2] = 0.0
    logits[0, 1::3] = -0.0
    k = 2048 if ld > 64 else 16
    row_len = rng.integers(0, ld + 1, R).astype(np.int32)
    row_len[0] = ld
    row_len[1 % R] = min(k, ld)
    if R > 2:
        row_len[2] = min(k + 1, ld)
    if R > 3:
        row_len[3] = 0
    _exact(dsix, logits, row_len, k)


@pytest.mark.parametrize("R", [12, 400])
@pytest.mark.parametrize("k", [1, 7, 64, 2048, 5000])
def test_exact_various_k(dsix, k, R):
    rng = np.random.default_rng(k)
    ld = 12000
    logits = rng.integers(-50, 50, size=(R, ld)).astype(np.float32)  # heavy ties
    row_len = rng.integers(k, ld + 1, R).astype(np.int32)
    _exact(dsix, logits, row_len, k, seed=k)


def test_exact_all_equal_and_extremes(dsix):
    R, ld, k = 4, 9000, 2048
    logits = np.zeros((R, ld), np.float32)
    logits[1] = -np.inf
    logits[2] = np.finfo(np.float32).max
    logits[2, ::2] = -np.finfo(np.float32).max
    logits[3] = np.linspace(-1, 1, ld, dtype=np.float32)[::-1]
    _exact(dsix, logits, np.full(R, ld, np.int32), k)


@pytest.mark.parametrize("R", [3, 400])
def test_never_reads_past_row_len(dsix, R):
    # NaNs after L must not influence the result
    ld, k = 8192, 100
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((R, ld)).astype(np.float32)
    row_len = np.resize(np.array([5000, 150, 8000], np.int32), R)
    clean = logits.copy()
    for r in range(R):
        logits[r, row_len[r]:] = np.nan
    bt = _table(R, ld, 64, 2)
    rq = np.arange(R, dtype=np.int32)
    loc, glb = _run(dsix, logits, row_len, rq, bt, k)
    rl, rg = oracle.topk_to_global(clean, row_len, rq, bt, 64, k)
    assert np.array_equal(loc, rl) and np.array_equal(glb, rg)


@pytest.mark.parametrize("R", [12, 400])
@pytest.mark.parametrize("kind", ["one_binade", "consecutive_floats", "two_values", "tiny_spread_ties"])
def test_exact_narrow_ranges(dsix, kind, R):
    # rows whose keys share many leading bits: the radix digits start below the
    # common prefix, which must not change the selected set or its order
    rng = np.random.default_rng(7)
    ld, k = 8192, 2048
    if kind == "one_binade":
        logits = (8 + 8 * rng.random((R, ld))).astype(np.float32)
    elif kind == "consecutive_floats":
        base = np.arange(ld, dtype=np.int32) + np.float32(1.0).view(np.int32)
        logits = np.stack([rng.permutation(base).view(np.float32) for _ in range(R)])
    elif kind == "two_values":
        logits = rng.choice(np.array([1.0, np.nextafter(np.float32(1), np.float32(2))], np.float32), (R, ld))
    else:
        logits = (np.float32(1000) + rng.integers(0, 20, (R, ld)).astype(np.float32) * np.float32(2 ** -16))
    logits = logits.astype(np.float32)
    row_len = rng.integers(k + 1, ld + 1, R).astype(np.int32)
    row_len[0] = ld
    _exact(dsix, logits, row_len, k, seed=3)


@pytest.mark.parametrize("R", [12, 400])
def test_exact_all_negative_ragged(dsix, R):
    # every key below 2^31 (all logits negative): the common prefix and the
    # threshold bin can start at 0, next to the slots past a ragged row end
    rng = np.random.default_rng(11)
    ld, k = 8192, 2048
    logits = (-np.abs(rng.standard_normal((R, ld))) * 4 - 1).astype(np.float32)
    logits[1::2] = -rng.integers(1, 4, (R // 2, ld)).astype(np.float32)  # three tied values
    row_len = rng.integers(k + 1, ld + 1, R).astype(np.int32)
    row_len[0] = ld
    _exact(dsix, logits, row_len, k, seed=5)


@pytest.mark.parametrize("R", [12, 400])
@pytest.mark.parametrize("bs", [16, 48])
def test_exact_other_block_sizes(dsix, bs, R):
    # the remap for a power-of-two block size other than 64, and for one that is not
    rng = np.random.default_rng(bs)
    ld, k = 8192, 2048
    logits = (rng.standard_normal((R, ld)) * 2).astype(np.float32)
    row_len = rng.integers(k + 1, ld + 1, R).astype(np.int32)
    _exact(dsix, logits, row_len, k, bs=bs, seed=bs)


@pytest.mark.parametrize("R", [12, 400])
def test_exact_ties_in_a_small_threshold_bin(dsix, R):
    # The row's k-th largest value repeated m times, spread over the row or in
    # one run: the bin that holds the k-th key has about m keys (ranked directly
    # up to 128, by a further digit pass above), and the k_rem that are taken
    # must be the lowest-index copies.
    rng = np.random.default_rng(13)
    ld, k = 8192, 2048
    logits = (rng.standard_normal((R, ld)) * 8).astype(np.float32)
    row_len = rng.integers(k + 200, ld + 1, R).astype(np.int32)
    row_len[0] = ld
    copies = [2, 5, 20, 60, 100, 126, 127, 128, 129, 140, 300]
    for r in range(R):
        L = int(row_len[r])
        v = np.sort(logits[r, :L])[::-1][k - 1]
        m = copies[r % len(copies)]
        if r % 3 == 2:  # one run of consecutive positions (one or two threads' keys)
            s0 = int(rng.integers(0, L - m))
            pos = np.arange(s0, s0 + m)
        else:
            pos = rng.choice(L, m, replace=False)
        logits[r, pos] = v
    _exact(dsix, logits, row_len, k, seed=13)
