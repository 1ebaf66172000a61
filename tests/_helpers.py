"""Shared checks for the GPU parity tests.

Tolerances are the indexer parity rules: logits within
|d| <= 1e-3 * max|logit of the row| + 1e-4 (max over the row's visible
entries); top-k sets equal except for indices whose oracle logit lies within
that tolerance of the oracle's k-th value; cache writes, gathers and remaps
bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W

REL_TOL = 1e-3
ABS_TOL = 1e-4


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def row_tol(ref_row: np.ndarray) -> float:
    return REL_TOL * (float(np.abs(ref_row).max()) if ref_row.size else 0.0) + ABS_TOL


def check_logits_rows(got: np.ndarray, ref: np.ndarray, lens, what=""):
    """got/ref [R, >=L]; compare the visible prefix of every row."""
    for r, L in enumerate(lens):
        L = int(L)
        if L == 0:
            continue
        d = np.abs(got[r, :L].astype(np.float64) - ref[r, :L].astype(np.float64))
        tol = row_tol(ref[r, :L])
        assert np.all(np.isfinite(got[r, :L])), f"{what} row {r}: non-finite"
        assert d.max() <= tol, f"{what} row {r}: max|d|={d.max():.3g} > tol {tol:.3g}"


def oracle_cache(wl: W.Workload) -> np.ndarray:
    cache = np.zeros((wl.num_blocks, wl.block_size * (wl.head_dim + 4)), np.uint8)
    oracle.quant_write_k(W.bf16_bits(wl.k_bf16), wl.slot, cache, wl.block_size)
    return cache


def remap_via_oracle(local_row: np.ndarray, L: int, req: int, bt: np.ndarray, bs: int, k: int):
    """Global slots of a given index set, computed by the oracle's own remap."""
    ind = np.full((1, max(L, 1)), -1.0, np.float32)
    sel = local_row[local_row >= 0]
    ind[0, sel] = 1.0
    _, glb = oracle.topk_to_global(ind, np.array([L], np.int32), np.array([req], np.int32),
                                   bt, bs, k)
    return glb[0]


def check_topk_rows(gpu_local: np.ndarray, gpu_global: np.ndarray, ref_logits: np.ndarray,
                    lens, reqs, bt: np.ndarray, bs: int, k: int, what=""):
    """Set rule against the oracle's own top-k of the oracle logits; order,
    padding and the remap of the GPU's own choice checked exactly."""
    rl = np.asarray(lens, np.int32)
    rq = np.asarray(reqs, np.int32)
    loc, _ = oracle.topk_to_global(np.ascontiguousarray(ref_logits, np.float32), rl, rq, bt, bs, k)
    for r in range(len(rl)):
        L = int(rl[r])
        m = min(k, L)
        g = gpu_local[r]
        assert (g[m:] == -1).all() and (gpu_global[r, m:] == -1).all(), f"{what} row {r}: padding"
        sel = g[:m]
        assert (sel >= 0).all() and (sel < L).all(), f"{what} row {r}: range"
        assert (np.diff(sel) > 0).all(), f"{what} row {r}: not ascending"
        if L <= k:
            assert np.array_equal(sel, np.arange(L)), f"{what} row {r}: short row"
        else:
            row = ref_logits[r, :L].astype(np.float64)
            kth = np.sort(row)[::-1][k - 1]
            tol = row_tol(row)
            diff = set(sel.tolist()) ^ set(loc[r, :m].tolist())
            bad = [i for i in diff if abs(row[i] - kth) > tol]
            assert not bad, f"{what} row {r}: {len(bad)} indices off the threshold band"
        want_g = remap_via_oracle(g, L, int(rq[r]), bt, bs, k)
        assert np.array_equal(gpu_global[r], want_g), f"{what} row {r}: remap"
