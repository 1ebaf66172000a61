"""CPU oracle for the DeepSeek-V3.2 sparse-attention indexer hot path.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports, loads or calls anything here; only the test suite, the
smoke check in ``__graft_entry__`` and the benchmark's CPU-baseline leg do.

The arithmetic lives in ``oracle.c`` (plain C, OpenMP over rows, no fast-math);
this module only marshals numpy arrays into it.  Each C function cites the page
passage it follows; the definitions are:

* fp8 E4M3 codec from the OCP 8-bit floating point spec (bias 7, max 448,
  round-to-nearest-even, saturating).
* ``quant_write_k``: per-token amax/448 scale (floored at FLT_MIN), fp8 codes,
  written into the indexer-K block layout of vLLM PR #25869's
  cp_gather_indexer_k_quant_cache review (block_size x head_dim fp8 values, then
  block_size fp32 scales).
* ``gather_k``: that review's per-request loop (full blocks, then the partial
  last block), into preallocated outputs.
* ``paged_mqa_logits`` / ``mqa_logits``: the lightning-indexer score
  k_scale * sum_h w_h * ReLU(q_h . k), exact dot products, double head sum,
  one rounding to f32; -inf tail when clean (vLLM PR #36250 review).
* ``topk_to_global``: per-row top-k by (value desc, index asc), ascending index
  output, -1 padding, remap to block_table[b, s/bs]*bs + s%bs (ROCm/ATOM PR
  #1094, Technical Details).
* ``dsmla_quant_write``: the fp8_ds_mla 656-byte entry of vLLM PR #47090's
  _fused_norm_rope_kernel snippet.
* ``dsmla_norm_rope_write``: the whole step of that kernel for one token, RMSNorm
  of the NoPE values (exact sum of squares in double, mean square plus eps
  rounded once to f32, reciprocal root and scaling in f32), rotation of the
  interleaved RoPE pairs from a cos/sin table (f32, no fused multiply-add, bf16
  nearest-even), then the same 656-byte entry.
* ``fused_q``: the query side of the sparse MLA attention -- q_pe rotated as the
  cache's RoPE values are, then either the bf16 pair or (quantize_mqa) the
  576-wide MQA query coded to fp8 with one amax/448 scale per (token, head)
  (vLLM PR #47090 prhub summary: fused_q's quantize_mqa flag).
* ``quant_q``: the indexer's fp8 query, one amax/448 scale per (token, head),
  folded into the head weight (a positive scale commutes with the ReLU).
* ``dsmla_sparse_decode``: the consumer of the global top-k indices -- softmax
  attention of the bf16 query (ql_nope, q_pe) over the dequantised 656-byte
  entries each token's index row names (fp8 NoPE times its tile scale, bf16
  RoPE), in double; output and natural-log sum of exponentials per head.

Parity pins live in ``tests/test_oracle_*.py`` (marked ``not gpu``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O3, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quant_write_k.argtypes = [P, I64, I32, P, P, I64, I32]
        lib.oracle_gather_k.argtypes = [P, I64, I32, I32, P, I64, P, I32, P, P]
        lib.oracle_paged_mqa_logits.argtypes = [P, P, P, I64, I32, P, P, I64, I32, I32,
                                                I32, I32, P, I64, I32, P, I64]
        lib.oracle_mqa_logits.argtypes = [P, P, P, P, P, P, I64, I64, I32, I32, P, I64,
                                          I32, P, I64]
        lib.oracle_topk_to_global.argtypes = [P, I64, I64, P, P, P, I64, I32, I32, P, P]
        lib.oracle_dsmla_quant_write.argtypes = [P, P, I64, P, P, I64, I32, I64, I64]
        lib.oracle_dsmla_norm_rope_write.argtypes = [P, P, P, ctypes.c_float, P, P, I64, P, I64, P,
                                                     I64, I32, I64, I64]
        lib.oracle_dsmla_sparse_decode.argtypes = [P, P, P, I64, I32, I64, I64, P, I64, I32, I32,
                                                   ctypes.c_double, P, P]
        lib.oracle_fused_q.argtypes = [P, P, P, P, I64, I64, I32, I32, P, P, P]
        lib.oracle_quant_q.argtypes = [P, P, I64, I32, I32, P, P]
        for name in ("oracle_fused_q", "oracle_quant_q",
                     "oracle_dsmla_sparse_decode", "oracle_quant_write_k", "oracle_gather_k", "oracle_paged_mqa_logits",
                     "oracle_mqa_logits", "oracle_topk_to_global",
                     "oracle_dsmla_quant_write", "oracle_dsmla_norm_rope_write",
                     "oracle_num_threads"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _p(a):
    return None if a is None else a.ctypes.data


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: inconsistent inputs (rc={rc})")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def e4m3_decode(code: int) -> float:
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def e4m3_decode_table() -> np.ndarray:
    """float64 [256]: exact value of every code (NaN for the two NaN codes)."""
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in x], dtype=np.uint8)


def quant_write_k(k_bf16: np.ndarray, slot_mapping: np.ndarray, cache: np.ndarray,
                  block_size: int) -> None:
    """In place on ``cache`` (uint8 [num_blocks, block_size*(head_dim+4)])."""
    k = _c(k_bf16, np.uint16)
    sm = _c(slot_mapping, np.int64)
    assert cache.flags.c_contiguous and cache.dtype == np.uint8
    n, d = k.shape
    rc = _load().oracle_quant_write_k(_p(k), n, d, _p(sm), _p(cache), cache.shape[0], block_size)
    _check(rc, "quant_write_k")


def gather_k(cache: np.ndarray, block_size: int, head_dim: int, block_table: np.ndarray,
             cu_seq_lens: np.ndarray, out_k: np.ndarray, out_scale: np.ndarray) -> None:
    bt = _c(block_table, np.int32)
    cu = _c(cu_seq_lens, np.int32)
    assert out_k.flags.c_contiguous and out_k.dtype == np.uint8
    assert out_scale.flags.c_contiguous and out_scale.dtype == np.float32
    rc = _load().oracle_gather_k(_p(cache), cache.shape[0], block_size, head_dim, _p(bt),
                                 bt.shape[1], _p(cu), len(cu) - 1, _p(out_k), _p(out_scale))
    _check(rc, "gather_k")


def paged_mqa_logits(q_fp8: np.ndarray, w: np.ndarray, cache: np.ndarray, block_size: int,
                     context_lens: np.ndarray, block_table: np.ndarray, ld: int,
                     clean: bool = True, rows=None) -> np.ndarray:
    """q_fp8 uint8 [B, next_n, H, D]; w f32 [B*next_n, H].  Returns f32
    [len(rows) or B*next_n, ld]."""
    q = _c(q_fp8, np.uint8)
    B, next_n, H, D = q.shape
    w = _c(w, np.float32)
    cl = _c(context_lens, np.int32)
    bt = _c(block_table, np.int32)
    r = None if rows is None else _c(np.asarray(rows, dtype=np.int64), np.int64)
    nout = B * next_n if r is None else len(r)
    fill = -np.inf if clean else 0.0
    out = np.full((nout, ld), fill, dtype=np.float32)
    rc = _load().oracle_paged_mqa_logits(_p(q), _p(w), _p(cache), cache.shape[0], block_size,
                                         _p(cl), _p(bt), bt.shape[1], B, next_n, H, D,
                                         _p(out), ld, int(bool(clean)), _p(r),
                                         0 if r is None else len(r))
    _check(rc, "paged_mqa_logits")
    return out


def mqa_logits(q_fp8: np.ndarray, w: np.ndarray, k_fp8: np.ndarray, k_scale: np.ndarray,
               ks: np.ndarray, ke: np.ndarray, ld: int, clean: bool = True,
               rows=None) -> np.ndarray:
    """q_fp8 uint8 [Tq, H, D]; k_fp8 uint8 [Tk, D]; k_scale f32 [Tk]."""
    q = _c(q_fp8, np.uint8)
    tq, H, D = q.shape
    k = _c(k_fp8, np.uint8)
    tk = k.shape[0]
    r = None if rows is None else _c(np.asarray(rows, dtype=np.int64), np.int64)
    nout = tq if r is None else len(r)
    fill = -np.inf if clean else 0.0
    out = np.full((nout, ld), fill, dtype=np.float32)
    ks_ = _c(ks, np.int32)
    ke_ = _c(ke, np.int32)
    sc = _c(k_scale, np.float32)
    w = _c(w, np.float32)
    rc = _load().oracle_mqa_logits(_p(q), _p(w), _p(k), _p(sc), _p(ks_), _p(ke_), tq, tk, H, D,
                                   _p(out), ld, int(bool(clean)), _p(r),
                                   0 if r is None else len(r))
    _check(rc, "mqa_logits")
    return out


def topk_to_global(logits: np.ndarray, row_len: np.ndarray, row_req: np.ndarray,
                   block_table: np.ndarray, block_size: int, k: int):
    """Returns (local int32 [R, k], global int32 [R, k])."""
    lg = _c(logits, np.float32)
    R, ld = lg.shape
    rl = _c(row_len, np.int32)
    rq = _c(row_req, np.int32)
    bt = _c(block_table, np.int32)
    loc = np.empty((R, k), dtype=np.int32)
    glb = np.empty((R, k), dtype=np.int32)
    rc = _load().oracle_topk_to_global(_p(lg), ld, R, _p(rl), _p(rq), _p(bt), bt.shape[1],
                                       block_size, k, _p(loc), _p(glb))
    _check(rc, "topk_to_global")
    return loc, glb


def dsmla_quant_write(nope_bf16: np.ndarray, rope_bf16: np.ndarray, slot_mapping: np.ndarray,
                      cache: np.ndarray, block_size: int) -> None:
    """cache uint8 [num_blocks, block_size, entry_bytes] (dense), in place."""
    nope = _c(nope_bf16, np.uint16)
    rope = _c(rope_bf16, np.uint16)
    sm = _c(slot_mapping, np.int64)
    assert cache.flags.c_contiguous and cache.dtype == np.uint8 and cache.ndim == 3
    nb, bs, entry = cache.shape
    assert bs == block_size
    rc = _load().oracle_dsmla_quant_write(_p(nope), _p(rope), nope.shape[0], _p(sm), _p(cache),
                                          nb, block_size, bs * entry, entry)
    _check(rc, "dsmla_quant_write")


def dsmla_norm_rope_write(kv_bf16: np.ndarray, pe_bf16: np.ndarray, gamma_bf16: np.ndarray,
                          eps: float, positions: np.ndarray, cos_sin: np.ndarray,
                          slot_mapping: np.ndarray, cache: np.ndarray, block_size: int) -> bool:
    """RMSNorm + RoPE + fp8_ds_mla entry write, in place.

    kv_bf16 uint16 [n, 512], pe_bf16 uint16 [n, 64], gamma_bf16 uint16 [512]
    (bf16 bits); positions int64 [n]; cos_sin f32 [max_pos, 64] (cosines, then
    sines); cache uint8 [num_blocks, block_size, entry_bytes].  Returns False
    when a slot or a position was out of range (those tokens are skipped)."""
    kv = _c(kv_bf16, np.uint16)
    pe = _c(pe_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    pos = _c(positions, np.int64)
    cs = _c(cos_sin, np.float32)
    sm = _c(slot_mapping, np.int64)
    assert kv.ndim == 2 and kv.shape[1] == 512 and pe.shape == (kv.shape[0], 64) and g.shape == (512,)
    assert cs.ndim == 2 and cs.shape[1] == 64 and pos.shape == sm.shape == (kv.shape[0],)
    assert cache.flags.c_contiguous and cache.dtype == np.uint8 and cache.ndim == 3
    nb, bs, entry = cache.shape
    assert bs == block_size
    rc = _load().oracle_dsmla_norm_rope_write(_p(kv), _p(pe), _p(g), float(eps), _p(pos), _p(cs),
                                              cs.shape[0], _p(sm), kv.shape[0], _p(cache), nb,
                                              block_size, bs * entry, entry)
    return rc == 0


def dsmla_sparse_decode(q_nope_bf16: np.ndarray, q_pe_bf16: np.ndarray, cache: np.ndarray,
                        block_size: int, indices: np.ndarray, sm_scale: float,
                        block_stride: int = None, entry_stride: int = None):
    """Sparse MLA decode over the fp8_ds_mla cache.

    q_nope uint16 [T, H, 512], q_pe uint16 [T, H, 64] (bf16 bits); cache uint8,
    either [num_blocks, block_size, entry_bytes] (dense) or flat bytes with
    explicit strides; indices int32 [T, topk] global slots (-1: none).
    Returns (out float64 [T, H, 512], lse float64 [T, H], ok)."""
    qn = _c(q_nope_bf16, np.uint16)
    qp = _c(q_pe_bf16, np.uint16)
    idx = _c(indices, np.int32)
    assert qn.ndim == 3 and qn.shape[2] == 512 and qp.shape == qn.shape[:2] + (64,)
    T, H = qn.shape[:2]
    assert idx.ndim == 2 and idx.shape[0] == T
    topk = idx.shape[1]
    cache = np.ascontiguousarray(cache)
    assert cache.dtype == np.uint8
    if cache.ndim == 3:
        nb, bs, entry = cache.shape
        assert bs == block_size
        block_stride = bs * entry if block_stride is None else block_stride
        entry_stride = entry if entry_stride is None else entry_stride
    else:
        assert block_stride is not None and entry_stride is not None
        nb = cache.size // block_stride
    out = np.empty((T, H, 512), dtype=np.float64)
    lse = np.empty((T, H), dtype=np.float64)
    rc = _load().oracle_dsmla_sparse_decode(_p(qn), _p(qp), _p(cache), nb, block_size, block_stride,
                                            entry_stride, _p(idx), T, H, topk, float(sm_scale),
                                            _p(out), _p(lse))
    return out, lse, rc == 0


def fused_q(ql_nope_bf16: np.ndarray, q_pe_bf16: np.ndarray, positions: np.ndarray, cos_sin: np.ndarray,
            quantize_mqa: bool):
    """ql_nope uint16 [T, H, 512], q_pe uint16 [T, H, 64] (bf16 bits); positions
    int64 [T]; cos_sin f32 [max_pos, 64].  Returns (out_pe uint16 [T, H, 64] or
    None, out_mqa uint8 [T, H, 576] or None, out_scale f32 [T, H] or None, ok)."""
    qn = _c(ql_nope_bf16, np.uint16)
    qp = _c(q_pe_bf16, np.uint16)
    pos = _c(positions, np.int64)
    cs = _c(cos_sin, np.float32)
    assert qn.ndim == 3 and qn.shape[2] == 512 and qp.shape == qn.shape[:2] + (64,)
    T, H = qn.shape[:2]
    assert pos.shape == (T,) and cs.ndim == 2 and cs.shape[1] == 64
    out_pe = out_mqa = out_scale = None
    if quantize_mqa:
        out_mqa = np.zeros((T, H, 576), np.uint8)
        out_scale = np.zeros((T, H), np.float32)
    else:
        out_pe = np.zeros((T, H, 64), np.uint16)
    dummy8, dummyf, dummy16 = np.zeros(1, np.uint8), np.zeros(1, np.float32), np.zeros(1, np.uint16)
    rc = _load().oracle_fused_q(_p(qn), _p(qp), _p(pos), _p(cs), cs.shape[0], T, H, int(bool(quantize_mqa)),
                                _p(dummy16 if out_pe is None else out_pe),
                                _p(dummy8 if out_mqa is None else out_mqa),
                                _p(dummyf if out_scale is None else out_scale))
    return out_pe, out_mqa, out_scale, rc == 0


def quant_q(q_bf16: np.ndarray, w: np.ndarray):
    """q uint16 [T, H, D] (bf16 bits), w f32 [T, H].  Returns (q_fp8 uint8
    [T, H, D], w_out f32 [T, H])."""
    q = _c(q_bf16, np.uint16)
    ww = _c(w, np.float32)
    assert q.ndim == 3 and ww.shape == q.shape[:2]
    T, H, D = q.shape
    out_q = np.zeros((T, H, D), np.uint8)
    out_w = np.zeros((T, H), np.float32)
    rc = _load().oracle_quant_q(_p(q), _p(ww), T, H, D, _p(out_q), _p(out_w))
    _check(rc, "quant_q")
    return out_q, out_w
