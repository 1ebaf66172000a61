"""Pins for the oracle's top-k selection and global remap (CPU only).

Definition (ROCm/ATOM PR #1094, Technical Details, plus the readings for the
points it leaves open): per row pick the min(k, L) largest logits, ties to the
lower index, -0.0 equal to +0.0; emit them in ascending index order, pad with
-1; remap request-local s to block_table[b, s // bs] * bs + s % bs.

Pins: brute force with Python's sorted() on tiny rows full of ties; the
selection invariants on larger random rows; padding cases (L = 0, L < k,
L = k); signed zeros; remap consistency.
"""
import numpy as np
import pytest

import oracle


def _brute(row, L, k):
    order = sorted(range(L), key=lambda i: (-float(row[i]), i))
    sel = sorted(order[:min(k, L)])
    return sel + [-1] * (k - len(sel))


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    R, ld, k, bs = 12, 40, 7, 4
    # few distinct values -> many ties, both signs, some -0.0
    vals = np.array([-1.5, -0.0, 0.0, 0.25, 0.25, 1.0, 3.0], np.float32)
    logits = vals[rng.integers(0, len(vals), size=(R, ld))]
    row_len = rng.integers(0, ld + 1, size=R).astype(np.int32)
    row_req = rng.integers(0, 3, size=R).astype(np.int32)
    bt = rng.permutation(3 * 10).reshape(3, 10).astype(np.int32)
    loc, glb = oracle.topk_to_global(logits, row_len, row_req, bt, bs, k)
    for r in range(R):
        want = _brute(logits[r], int(row_len[r]), k)
        assert loc[r].tolist() == want, r
        for i, s in enumerate(want):
            g = -1 if s < 0 else int(bt[row_req[r], s // bs]) * bs + s % bs
            assert glb[r, i] == g


def test_signed_zero_ties_to_lower_index():
    logits = np.array([[-0.0, 0.0, -0.0, 0.0, -1.0]], np.float32)
    loc, _ = oracle.topk_to_global(logits, np.array([5], np.int32), np.zeros(1, np.int32),
                                   np.arange(4, dtype=np.int32)[None], 4, 2)
    assert loc[0].tolist() == [0, 1]


def test_padding_cases():
    logits = np.arange(10, dtype=np.float32)[None].repeat(3, 0)
    rl = np.array([0, 3, 4], np.int32)
    loc, glb = oracle.topk_to_global(logits, rl, np.zeros(3, np.int32),
                                     np.array([[5, 6]], np.int32), 4, 4)
    assert loc[0].tolist() == [-1] * 4 and glb[0].tolist() == [-1] * 4
    assert loc[1].tolist() == [0, 1, 2, -1]
    assert glb[1].tolist() == [20, 21, 22, -1]
    assert loc[2].tolist() == [0, 1, 2, 3]


@pytest.mark.parametrize("seed", [0, 1])
def test_selection_invariants_random(seed):
    rng = np.random.default_rng(seed)
    R, ld, k, bs = 6, 3000, 256, 64
    logits = (rng.standard_normal((R, ld)) * 10).astype(np.float32)
    logits[:, ::7] = np.round(logits[:, ::7])   # plenty of exact ties
    row_len = np.array([0, 100, 256, 257, 2999, 3000], np.int32)
    nblk = -(-ld // bs)
    bt = rng.permutation(R * nblk).reshape(R, nblk).astype(np.int32)
    row_req = np.arange(R, dtype=np.int32)
    loc, glb = oracle.topk_to_global(logits, row_len, row_req, bt, bs, k)
    for r in range(R):
        L = int(row_len[r])
        m = min(k, L)
        sel = loc[r, :m]
        assert (loc[r, m:] == -1).all() and (glb[r, m:] == -1).all()
        assert (sel >= 0).all() and (sel < L).all()
        assert (np.diff(sel) > 0).all()
        if m < L:
            mask = np.zeros(L, bool)
            mask[sel] = True
            v = logits[r, :L]
            thr = v[mask].min()
            assert v[~mask].max() <= thr
            # among values equal to the threshold, the selected ones come first
            eq = np.nonzero(v == thr)[0]
            chosen = mask[eq]
            assert not np.any(np.diff(chosen.astype(int)) > 0)
        g = glb[r, :m]
        assert np.array_equal(g // bs, bt[r, sel // bs]) and np.array_equal(g % bs, sel % bs)
