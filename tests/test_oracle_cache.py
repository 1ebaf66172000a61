"""Pins for the oracle's cache writers and gather (CPU only).

* Indexer K quantise/write: the block layout comes from the golden fixture
  (cited to the cp_gather_indexer_k_quant_cache review of vLLM PR #25869); the
  scale is compared bit for bit with numpy's IEEE f32 division amax/448 (floored
  at FLT_MIN); the codes with torch's float8_e4m3fn cast of x/scale; plus the
  amax-element and all-zero invariants.
* Gather: an identity block table over one request equals the plain slice;
  a ragged batch (empty requests, partial last blocks) equals an independent
  vectorised index formula; rows past cu_seq_lens[B] are untouched.
* fp8_ds_mla write: offsets re-derived from the page's index arithmetic in the
  golden fixture; the scale is compared with numpy's amax * f32(1/448) (floored);
  codes with torch's cast; RoPE bit copy; zero tile; amax element.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

FLT_MIN = np.float32(np.finfo(np.float32).tiny)


def _layout(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _torch_e4m3(x_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _rand_bf16(rng_seed, shape, scale=1.0):
    g = torch.Generator().manual_seed(rng_seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# indexer K quant-write
# ---------------------------------------------------------------------------

def test_quant_write_k_layout_scale_codes(golden_dir):
    lay = _layout(golden_dir, "indexer_k_block_layout.json")
    bs, D = lay["block_size"], lay["head_dim"]
    assert lay["block_bytes"] == bs * (D + 4)
    nb, n = 6, 200
    k = _rand_bf16(3, (n, D))
    # rows with wide dynamic range, a zero row, a negative-zero row
    k[5] = k[5] * 1e-30
    k[6] = 0.0
    k[7] = -0.0
    k[8, 3] = 300.0
    rng = np.random.default_rng(0)
    slots = rng.permutation(nb * bs)[:n].astype(np.int64)
    slots[10] = -1  # skipped
    cache = np.full((nb, lay["block_bytes"]), 0xA5, dtype=np.uint8)
    oracle.quant_write_k(W.bf16_bits(k), slots, cache, bs)
    x = k.float().numpy()
    for t in range(n):
        s = slots[t]
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        row = cache[blk]
        vals = row[lay["value_offset"] + off * lay["value_token_stride"]:][:D]
        sc = row[lay["scale_offset"] + off * lay["scale_token_stride"]:][:4].view(np.float32)[0]
        amax = np.float32(np.abs(x[t]).max())
        want_sc = np.maximum(amax / np.float32(448.0), FLT_MIN)
        assert sc.view(np.uint32) == np.float32(want_sc).view(np.uint32), t
        want_codes = _torch_e4m3(x[t] / np.float32(want_sc))
        assert np.array_equal(vals, want_codes), t
        if amax > 0:
            i = int(np.argmax(np.abs(x[t])))
            assert vals[i] & 0x7F == 0x7E
    # the skipped token's bytes remain untouched: count sentinel bytes
    written = (slots >= 0).sum()
    untouched = (cache == 0xA5).all(axis=None)
    assert not untouched
    # zero rows: scale floor, codes 0 / 0x80
    for t, code in ((6, 0x00), (7, 0x80)):
        blk, off = divmod(int(slots[t]), bs)
        assert (cache[blk, off * D:(off + 1) * D] == code).all()
        sc = cache[blk, 8192 + 4 * off:8192 + 4 * off + 4].view(np.float32)[0]
        assert sc == FLT_MIN
    assert written == n - 1


def test_quant_write_k_skip_negative_slot():
    bs, D = 64, 128
    k = _rand_bf16(1, (3, D))
    cache = np.full((2, bs * (D + 4)), 0x5A, dtype=np.uint8)
    oracle.quant_write_k(W.bf16_bits(k), np.array([-1, -5, -1], np.int64), cache, bs)
    assert (cache == 0x5A).all()


def test_quant_write_k_round_trip_error_bound():
    bs, D = 64, 128
    k = _rand_bf16(5, (128, D))
    slots = np.arange(128, dtype=np.int64)
    cache = np.zeros((2, bs * (D + 4)), dtype=np.uint8)
    oracle.quant_write_k(W.bf16_bits(k), slots, cache, bs)
    tab = oracle.e4m3_decode_table()
    x = k.float().numpy().astype(np.float64)
    for t in range(128):
        blk, off = divmod(t, bs)
        v = tab[cache[blk, off * D:(off + 1) * D]]
        sc = float(cache[blk, 8192 + 4 * off:8192 + 4 * off + 4].view(np.float32)[0])
        y = x[t] / sc
        # half an e4m3 ulp at |y| (3 mantissa bits, subnormal step 2^-9), plus slack
        # for the f32 division before encoding
        ulp = np.where(np.abs(y) < 2 ** -6, 2.0 ** -9,
                       2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2 ** -6))) - 3))
        assert np.all(np.abs(v - y) <= 0.5 * ulp * (1 + 1e-6) + 1e-12)


# ---------------------------------------------------------------------------
# gather
# ---------------------------------------------------------------------------

def _filled_cache(nb, bs, D, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(nb, bs * (D + 4)), dtype=np.uint8)


def test_gather_identity_table_is_plain_slice():
    bs, D, nb = 64, 128, 5
    cache = _filled_cache(nb, bs, D, 0)
    s = 4 * bs + 17
    bt = np.arange(nb, dtype=np.int32)[None, :]
    cu = np.array([0, s], np.int32)
    out_k = np.zeros((s, D), np.uint8)
    out_s = np.zeros(s, np.float32)
    oracle.gather_k(cache, bs, D, bt, cu, out_k, out_s)
    vals = cache[:, :bs * D].reshape(-1, D)[:s]
    scales = cache[:, bs * D:].reshape(-1, 4).copy().view(np.float32).ravel()[:s]
    assert np.array_equal(out_k, vals)
    assert np.array_equal(out_s.view(np.uint32), scales.view(np.uint32))


def test_gather_ragged_matches_index_formula():
    bs, D, nb = 64, 128, 40
    cache = _filled_cache(nb, bs, D, 1)
    lens = [0, 1, 63, 64, 65, 0, 200, 128]
    rng = np.random.default_rng(2)
    perm = rng.permutation(nb).astype(np.int32)
    maxb = 5
    bt = np.full((len(lens), maxb), 9999, np.int32)  # unused entries are garbage
    o = 0
    for b, s in enumerate(lens):
        nbk = -(-s // bs)
        bt[b, :nbk] = perm[o:o + nbk]
        o += nbk
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    out_k = np.full((T + 3, D), 0xEE, np.uint8)
    out_s = np.full(T + 3, -7.0, np.float32)
    oracle.gather_k(cache, bs, D, bt, cu, out_k, out_s)
    # independent statement: token i of request b is row i%bs of block bt[b, i//bs]
    req = np.repeat(np.arange(len(lens)), lens)
    pos = np.concatenate([np.arange(s) for s in lens])
    blk = bt[req, pos // bs]
    off = pos % bs
    want_k = cache[blk[:, None], off[:, None] * D + np.arange(D)[None, :]]
    sb = cache[blk[:, None], bs * D + off[:, None] * 4 + np.arange(4)[None, :]]
    want_s = np.ascontiguousarray(sb).view(np.float32).ravel()
    assert np.array_equal(out_k[:T], want_k)
    assert np.array_equal(out_s[:T].view(np.uint32), want_s.view(np.uint32))
    assert (out_k[T:] == 0xEE).all() and (out_s[T:] == -7.0).all()


def test_quant_then_gather_round_trip():
    wl = W.build("rt", decode_ctx=[70, 5, 130], next_n=1, topk=16, seed=4, pool_blocks=9)
    cache = np.zeros((wl.num_blocks, 64 * 132), np.uint8)
    oracle.quant_write_k(W.bf16_bits(wl.k_bf16), wl.slot, cache, 64)
    cu = np.concatenate([[0], np.cumsum(wl.req_ctx)]).astype(np.int32)
    T = int(cu[-1])
    out_k = np.zeros((T, 128), np.uint8)
    out_s = np.zeros(T, np.float32)
    oracle.gather_k(cache, 64, 128, wl.block_table, cu, out_k, out_s)
    tab = oracle.e4m3_decode_table()
    deq = tab[out_k] * out_s[:, None].astype(np.float64)
    x = wl.k_bf16.float().numpy()
    # per-token relative error of e4m3 (3 mantissa bits) <= 2^-4 of amax
    err = np.abs(deq - x).max(axis=1) / np.abs(x).max(axis=1)
    assert err.max() <= 2.0 ** -4


# ---------------------------------------------------------------------------
# fp8_ds_mla write
# ---------------------------------------------------------------------------

def test_dsmla_offsets_from_page_arithmetic(golden_dir):
    lay = _layout(golden_dir, "fp8_ds_mla_entry_layout.json")
    kv = lay["kv_dim"]
    # fp32 element index KV_DIM/4 + t -> byte 4*(KV_DIM/4 + t)
    assert 4 * (kv // 4) == lay["scale_offset"]
    # bf16 element index KV_DIM/2 + 8 -> byte 2*(KV_DIM/2 + 8)
    assert 2 * (kv // 2 + 8) == lay["rope_offset"]
    assert lay["scale_offset"] + 4 * lay["num_tiles"] == lay["rope_offset"]
    assert lay["rope_offset"] + 2 * lay["rope_dim"] == lay["entry_bytes"]
    assert lay["num_tiles"] * lay["tile_dim"] == kv


def test_dsmla_write_scale_codes_rope(golden_dir):
    lay = _layout(golden_dir, "fp8_ds_mla_entry_layout.json")
    bs, nb, n = 64, 3, 150
    g = torch.Generator().manual_seed(7)
    nope = torch.randn(n, 512, generator=g)
    out = torch.rand(n, 512, generator=g) < 0.01
    nope = torch.where(out, nope * 20, nope)
    nope[4, :128] = 0.0                   # zero tile
    nope[5, 128:256] *= 1e-35             # tiny tile (scale floor)
    nope = nope.to(torch.bfloat16)
    rope = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    slots = np.random.default_rng(1).permutation(nb * bs)[:n].astype(np.int64)
    cache = np.full((nb, bs, lay["entry_bytes"]), 0x33, np.uint8)
    oracle.dsmla_quant_write(W.bf16_bits(nope), W.bf16_bits(rope), slots, cache, bs)
    x = nope.float().numpy()
    inv = np.float32(1.0 / 448.0)
    floor = np.float32(float(lay["scale_floor"]))
    assert floor == FLT_MIN
    rb = W.bf16_bits(rope)
    for t in range(n):
        blk, off = divmod(int(slots[t]), bs)
        e = cache[blk, off]
        for tile in range(4):
            xt = x[t, tile * 128:(tile + 1) * 128]
            amax = np.float32(np.abs(xt).max())
            want = np.maximum(np.float32(amax * inv), floor)
            got = e[lay["scale_offset"] + 4 * tile:][:4].view(np.float32)[0]
            assert got.view(np.uint32) == np.float32(want).view(np.uint32)
            codes = e[tile * 128:(tile + 1) * 128]
            assert np.array_equal(codes, _torch_e4m3(xt / np.float32(want)))
            if amax > 0:
                assert codes[int(np.argmax(np.abs(xt)))] & 0x7F == 0x7E
        assert np.array_equal(e[lay["rope_offset"]:lay["entry_bytes"]].view(np.uint16), rb[t])
    blk, off = divmod(int(slots[4]), bs)
    assert (cache[blk, off, :128] == 0).all()
    assert cache[blk, off, 512:516].view(np.float32)[0] == FLT_MIN


def test_dsmla_scale_uses_multiply_not_divide():
    # amax * f32(1/448) and amax / 448 differ for some amax; the page's tile
    # scale is the product.  Find such an amax and check the product is written.
    inv = np.float32(1.0 / 448.0)
    cand = None
    for m in range(1, 4000):
        a = np.float32(1.0 + m / 128.0)
        a = np.float32(torch.tensor(float(a)).to(torch.bfloat16).float().item())
        if np.float32(a * inv) != np.float32(a / np.float32(448.0)):
            cand = a
            break
    assert cand is not None
    nope = torch.zeros(1, 512)
    nope[0, 0] = float(cand)
    nope = nope.to(torch.bfloat16)
    cache = np.zeros((1, 64, 656), np.uint8)
    oracle.dsmla_quant_write(W.bf16_bits(nope), W.bf16_bits(torch.zeros(1, 64).to(torch.bfloat16)),
                             np.array([0], np.int64), cache, 64)
    got = cache[0, 0, 512:516].view(np.float32)[0]
    assert got == np.float32(cand * inv)
