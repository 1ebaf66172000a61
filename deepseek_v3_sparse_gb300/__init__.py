"""Python binding of libdsix (include/dsix.h): the GB300 DeepSeek-V3.2
sparse-attention indexer hot path.

Argument marshalling only: each function checks dtypes/devices of its torch
tensors, passes their device pointers and sizes to the C entry point of the
same name, and raises ``DsixError`` on a non-zero status.  Every step of the
path runs in the library's CUDA kernels; there is no fallback of any kind --
if ``libdsix.so`` is missing or fails to load, every call raises.

Outputs are caller-allocated tensors (the library allocates nothing).  Calls
are asynchronous on ``stream`` (default: torch's current stream) and never
synchronise, so a sequence of them can be captured in a CUDA graph.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = [
    "DsixError", "load", "ix_status_string", "ix_device_status", "ix_quant_write_k",
    "ix_gather_k", "ix_paged_mqa_logits", "ix_mqa_logits", "ix_topk_to_global",
    "ix_topk_hist_workspace_size", "ix_paged_mqa_logits_topk", "ix_mqa_logits_topk",
    "ix_paged_mqa_logits_hist", "ix_mqa_logits_hist", "ix_topk_from_hist", "dsmla_fused_q", "ix_quant_q",
    "dsmla_quant_write", "dsmla_norm_rope_write", "dsmla_sparse_decode",
    "dsmla_sparse_decode_workspace_size", "dsmla_sparse_decode_noalloc", "MLA_HEADS", "LIB_PATH", "HEADS", "HEAD_DIM", "BLOCK_SIZE",
]

HEADS = 64
HEAD_DIM = 128
BLOCK_SIZE = 64
INDEXER_BLOCK_BYTES = BLOCK_SIZE * (HEAD_DIM + 4)
DSMLA_ENTRY_BYTES = 656

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdsix.so")

_lib = None
_lock = threading.Lock()


class DsixError(RuntimeError):
    pass


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int

_SIGNATURES = {
    "ix_status_string": ([_I32], ctypes.c_char_p),
    "ix_device_status": ([_P], _I32),
    "ix_quant_write_k": ([_P, _I64, _I32, _P, _P, _I64, _I32, _P], _I32),
    "ix_gather_k": ([_P, _I64, _I32, _I32, _P, _I64, _P, _I32, _P, _P, _I64, _P], _I32),
    "ix_paged_mqa_logits": ([_P, _P, _P, _I64, _I32, _P, _P, _I64, _I32, _I32, _I32, _I32, _P,
                             _I64, _I32, _P], _I32),
    "ix_mqa_logits": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _P, _I64, _I32, _P], _I32),
    "ix_topk_to_global": ([_P, _I64, _I64, _P, _P, _P, _I64, _I32, _I32, _P, _P, _P], _I32),
    "ix_topk_hist_workspace_size": ([_I64], ctypes.c_size_t),
    "ix_paged_mqa_logits_topk": ([_P, _P, _P, _I64, _I32, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _I64,
                                  _I32, _P, _P, _P, ctypes.c_size_t, _P], _I32),
    "ix_mqa_logits_topk": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _P, _I64, _P, _P, _I64, _I32,
                            _I32, _P, _P, _P, ctypes.c_size_t, _P], _I32),
    "ix_paged_mqa_logits_hist": ([_P, _P, _P, _I64, _I32, _P, _P, _I64, _I32, _I32, _I32, _I32, _P, _I64,
                                  _I32, _P, ctypes.c_size_t, _P], _I32),
    "ix_mqa_logits_hist": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _P, _I64, _I32, _P,
                            ctypes.c_size_t, _P], _I32),
    "dsmla_fused_q": ([_P, _P, _P, _P, _I64, _I64, _I32, _I32, _P, _P, _P, _P], _I32),
    "ix_quant_q": ([_P, _P, _I64, _I32, _I32, _P, _P, _P], _I32),
    "ix_topk_from_hist": ([_P, _I64, _I64, _P, _P, _P, _I64, _I32, _I32, _P, _P, _P, ctypes.c_size_t, _P],
                          _I32),
    "dsmla_quant_write": ([_P, _P, _I64, _P, _P, _I64, _I32, _I64, _I64, _P], _I32),
    "dsmla_norm_rope_write": ([_P, _P, _P, ctypes.c_float, _P, _P, _I64, _P, _I64, _P, _I64, _I32,
                               _I64, _I64, _P], _I32),
    "dsmla_sparse_decode_workspace_size": ([_I64, _I32, _I32], ctypes.c_size_t),
    "dsmla_sparse_decode": ([_P, _P, _P, _I64, _I32, _I64, _I64, _P, _I64, _I32, _I32, ctypes.c_float,
                             _P, _P, _P, ctypes.c_size_t, _P], _I32),
    "dsmla_sparse_decode_noalloc": ([_P, _P, _P, _I64, _I32, _I64, _I64, _P, _I64, _I32, _I32,
                                     ctypes.c_float, _P, _P, _P], _I32),
}


def load(path: Optional[str] = None):
    """Load libdsix.so (built by ``deepseek_v3_sparse_gb300.build``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise DsixError(f"{p} is missing: build it with `python -m deepseek_v3_sparse_gb300.build` "
                            "(there is no non-CUDA fallback)")
        lib = ctypes.CDLL(p)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        if path is None:
            _lib = lib
        return lib


def ix_status_string(status: int) -> str:
    return load().ix_status_string(int(status)).decode()


def _check(rc: int, name: str):
    if rc != 0:
        raise DsixError(f"{name}: {ix_status_string(rc)} ({rc})")


def ix_device_status() -> int:
    """Synchronously read and clear the device status word (IX_DEV_* bits)."""
    v = ctypes.c_int(0)
    rc = load().ix_device_status(ctypes.byref(v))
    if rc not in (0, -7):
        _check(rc, "ix_device_status")
    return int(v.value)


def _dev(t: torch.Tensor, name: str, dtypes) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise DsixError(f"{name}: must be a CUDA tensor")
    if t.device.index is not None and t.device.index != torch.cuda.current_device():
        # the library launches on the current device: a tensor of another
        # device would hand its pointer to kernels that cannot reach it
        raise DsixError(f"{name}: on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise DsixError(f"{name}: must be contiguous")
    return t.data_ptr()


def _need(ok: bool, what: str):
    """Shape consistency the C ABI cannot see (it receives bare pointers): an
    inconsistent tensor would be read or written past its end."""
    if not ok:
        raise DsixError(what)


def _rows(t, n: int, name: str, cols: Optional[int] = None, dim: int = 2):
    """t has `dim` dimensions, at least n rows, and (if given) exactly `cols` columns."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    _need(t.dim() == dim and t.shape[0] >= n and (cols is None or t.shape[-1] == cols),
          f"{name}: shape {tuple(t.shape)}, expected {dim}-D with >= {n} rows"
          + ("" if cols is None else f" and {cols} columns"))


def _len(t, n: int, name: str):
    """t holds at least n elements."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    _need(t.numel() >= n, f"{name}: {t.numel()} elements, expected >= {n}")


def _opt(t, name, dtypes):
    return None if t is None else _dev(t, name, dtypes)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


_U8 = (torch.uint8, torch.float8_e4m3fn)
_BF16 = (torch.bfloat16,)
_F32 = (torch.float32,)
_I32T = (torch.int32,)
_I64T = (torch.int64,)


def ix_quant_write_k(k_bf16: torch.Tensor, slot_mapping: torch.Tensor, cache: torch.Tensor,
                     block_size: int = BLOCK_SIZE, stream=None) -> None:
    """k_bf16 [n, 128] bf16; slot_mapping [n] int64; cache uint8 [num_blocks, 8448]."""
    _rows(k_bf16, 0, "k_bf16")
    n, d = k_bf16.shape
    _len(slot_mapping, n, "slot_mapping")
    _rows(cache, 0, "cache", block_size * (d + 4))
    rc = load().ix_quant_write_k(_dev(k_bf16, "k_bf16", _BF16), n, d,
                                 _dev(slot_mapping, "slot_mapping", _I64T),
                                 _dev(cache, "cache", (torch.uint8,)), cache.shape[0], block_size,
                                 _stream(stream))
    _check(rc, "ix_quant_write_k")


def ix_gather_k(cache: torch.Tensor, block_table: torch.Tensor, cu_seq_lens: torch.Tensor,
                out_k: torch.Tensor, out_scale: torch.Tensor, block_size: int = BLOCK_SIZE,
                head_dim: int = HEAD_DIM, stream=None) -> None:
    """block_table [B, stride] int32; cu_seq_lens [B+1] int32; out_k [cap, 128] fp8/u8;
    out_scale [cap] f32."""
    _len(cu_seq_lens, 1, "cu_seq_lens")
    _rows(block_table, cu_seq_lens.numel() - 1, "block_table")
    _rows(cache, 0, "cache", block_size * (head_dim + 4))
    _rows(out_k, 0, "out_k", head_dim)
    _len(out_scale, out_k.shape[0], "out_scale")
    rc = load().ix_gather_k(_dev(cache, "cache", (torch.uint8,)), cache.shape[0], block_size,
                            head_dim, _dev(block_table, "block_table", _I32T), block_table.stride(0),
                            _dev(cu_seq_lens, "cu_seq_lens", _I32T), cu_seq_lens.numel() - 1,
                            _dev(out_k, "out_k", _U8), _dev(out_scale, "out_scale", _F32),
                            out_k.shape[0], _stream(stream))
    _check(rc, "ix_gather_k")


def ix_paged_mqa_logits(q_fp8: torch.Tensor, w: torch.Tensor, cache: torch.Tensor,
                        context_lens: torch.Tensor, block_table: torch.Tensor,
                        logits: torch.Tensor, clean_logits: bool = False,
                        block_size: int = BLOCK_SIZE, stream=None) -> None:
    """q_fp8 [B, next_n, 64, 128] e4m3 (or its uint8 bits); w [B*next_n, 64] f32;
    logits [B*next_n, ld] f32 (written in place)."""
    _rows(q_fp8, 0, "q_fp8", dim=4)
    B, next_n, H, D = q_fp8.shape
    _rows(w, B * next_n, "w", H)
    _rows(logits, B * next_n, "logits")
    _len(context_lens, B, "context_lens")
    _rows(block_table, B, "block_table")
    _rows(cache, 0, "cache", block_size * (D + 4))
    rc = load().ix_paged_mqa_logits(
        _dev(q_fp8, "q_fp8", _U8), _dev(w, "w", _F32), _dev(cache, "cache", (torch.uint8,)),
        cache.shape[0], block_size, _dev(context_lens, "context_lens", _I32T),
        _dev(block_table, "block_table", _I32T), block_table.stride(0), B, next_n, H, D,
        _dev(logits, "logits", _F32), logits.shape[1], int(bool(clean_logits)), _stream(stream))
    _check(rc, "ix_paged_mqa_logits")


def ix_mqa_logits(q_fp8: torch.Tensor, w: torch.Tensor, k_fp8: torch.Tensor,
                  k_scale: torch.Tensor, ks: torch.Tensor, ke: torch.Tensor,
                  logits: torch.Tensor, clean_logits: bool = False, stream=None) -> None:
    """q_fp8 [Tq, 64, 128]; w [Tq, 64]; k_fp8 [Tk, 128]; k_scale [Tk]; ks/ke [Tq] int32;
    logits [Tq, ld] f32."""
    _rows(q_fp8, 0, "q_fp8", dim=3)
    tq, H, D = q_fp8.shape
    _rows(w, tq, "w", H)
    _rows(k_fp8, 0, "k_fp8", D)
    _len(k_scale, k_fp8.shape[0], "k_scale")
    _len(ks, tq, "ks")
    _len(ke, tq, "ke")
    _rows(logits, tq, "logits")
    rc = load().ix_mqa_logits(
        _dev(q_fp8, "q_fp8", _U8), _dev(w, "w", _F32), _dev(k_fp8, "k_fp8", _U8),
        _dev(k_scale, "k_scale", _F32), _dev(ks, "ks", _I32T), _dev(ke, "ke", _I32T), tq,
        k_fp8.shape[0], H, D, _dev(logits, "logits", _F32), logits.shape[1],
        int(bool(clean_logits)), _stream(stream))
    _check(rc, "ix_mqa_logits")


def ix_topk_to_global(logits: torch.Tensor, row_len: torch.Tensor, row_req: torch.Tensor,
                      block_table: torch.Tensor, k: int, out_global: torch.Tensor,
                      out_local: Optional[torch.Tensor] = None, block_size: int = BLOCK_SIZE,
                      stream=None) -> None:
    """logits [R, ld] f32; row_len/row_req [R] int32; out_global/out_local [R, k] int32."""
    _rows(logits, 0, "logits")
    R, ld = logits.shape
    _len(row_len, R, "row_len")
    _len(row_req, R, "row_req")
    _rows(block_table, 0, "block_table")
    _len(out_global, R * int(k), "out_global")
    if out_local is not None:
        _len(out_local, R * int(k), "out_local")
    rc = load().ix_topk_to_global(
        _dev(logits, "logits", _F32), ld, R, _dev(row_len, "row_len", _I32T),
        _dev(row_req, "row_req", _I32T), _dev(block_table, "block_table", _I32T),
        block_table.stride(0), block_size, int(k), _opt(out_local, "out_local", _I32T),
        _dev(out_global, "out_global", _I32T), _stream(stream))
    _check(rc, "ix_topk_to_global")


def ix_topk_hist_workspace_size(rows: int) -> int:
    """Bytes of the fused calls' histogram workspace for `rows` logits rows (zero it
    once when it is allocated; every completed call leaves it zero)."""
    return int(load().ix_topk_hist_workspace_size(int(rows)))


def _workspace(ws: torch.Tensor, rows: int):
    _need(isinstance(ws, torch.Tensor) and ws.numel() * ws.element_size() >= ix_topk_hist_workspace_size(rows),
          f"workspace: fewer than {ix_topk_hist_workspace_size(rows)} bytes for {rows} rows")
    return _dev(ws, "workspace", (torch.uint8, torch.int32, torch.float32)), ws.numel() * ws.element_size()


def ix_paged_mqa_logits_topk(q_fp8: torch.Tensor, w: torch.Tensor, cache: torch.Tensor,
                             context_lens: torch.Tensor, block_table: torch.Tensor, logits: torch.Tensor,
                             k: int, out_global: torch.Tensor, workspace: torch.Tensor,
                             out_local: Optional[torch.Tensor] = None, block_size: int = BLOCK_SIZE,
                             stream=None) -> None:
    """Decode logits over the paged cache and the top-k of their rows in one call
    (see ix_paged_mqa_logits and ix_topk_to_global); logits [B*next_n, ld] f32 is
    written and read back; out_global/out_local [B*next_n, k] int32."""
    _rows(q_fp8, 0, "q_fp8", dim=4)
    B, next_n, H, D = q_fp8.shape
    R = B * next_n
    _rows(w, R, "w", H)
    _rows(logits, R, "logits")
    _len(context_lens, B, "context_lens")
    _rows(block_table, B, "block_table")
    _rows(cache, 0, "cache", block_size * (D + 4))
    _len(out_global, R * int(k), "out_global")
    if out_local is not None:
        _len(out_local, R * int(k), "out_local")
    wp, wb = _workspace(workspace, R)
    rc = load().ix_paged_mqa_logits_topk(
        _dev(q_fp8, "q_fp8", _U8), _dev(w, "w", _F32), _dev(cache, "cache", (torch.uint8,)),
        cache.shape[0], block_size, _dev(context_lens, "context_lens", _I32T),
        _dev(block_table, "block_table", _I32T), block_table.stride(0), B, next_n, H, D,
        _dev(logits, "logits", _F32), logits.shape[1], int(k), _opt(out_local, "out_local", _I32T),
        _dev(out_global, "out_global", _I32T), wp, wb, _stream(stream))
    _check(rc, "ix_paged_mqa_logits_topk")


def ix_mqa_logits_topk(q_fp8: torch.Tensor, w: torch.Tensor, k_fp8: torch.Tensor, k_scale: torch.Tensor,
                       ks: torch.Tensor, ke: torch.Tensor, logits: torch.Tensor, row_req: torch.Tensor,
                       block_table: torch.Tensor, k: int, out_global: torch.Tensor, workspace: torch.Tensor,
                       out_local: Optional[torch.Tensor] = None, block_size: int = BLOCK_SIZE,
                       stream=None) -> None:
    """Prefill logits over contiguous K and the top-k of their rows in one call
    (see ix_mqa_logits and ix_topk_to_global); row t has ke[t] - ks[t] keys and is
    remapped through block_table[row_req[t]]."""
    _rows(q_fp8, 0, "q_fp8", dim=3)
    tq, H, D = q_fp8.shape
    _rows(w, tq, "w", H)
    _rows(k_fp8, 0, "k_fp8", D)
    _len(k_scale, k_fp8.shape[0], "k_scale")
    _len(ks, tq, "ks")
    _len(ke, tq, "ke")
    _len(row_req, tq, "row_req")
    _rows(logits, tq, "logits")
    _rows(block_table, 0, "block_table")
    _len(out_global, tq * int(k), "out_global")
    if out_local is not None:
        _len(out_local, tq * int(k), "out_local")
    wp, wb = _workspace(workspace, tq)
    rc = load().ix_mqa_logits_topk(
        _dev(q_fp8, "q_fp8", _U8), _dev(w, "w", _F32), _dev(k_fp8, "k_fp8", _U8),
        _dev(k_scale, "k_scale", _F32), _dev(ks, "ks", _I32T), _dev(ke, "ke", _I32T), tq, k_fp8.shape[0], H, D,
        _dev(logits, "logits", _F32), logits.shape[1], _dev(row_req, "row_req", _I32T),
        _dev(block_table, "block_table", _I32T), block_table.stride(0), block_size, int(k),
        _opt(out_local, "out_local", _I32T), _dev(out_global, "out_global", _I32T), wp, wb, _stream(stream))
    _check(rc, "ix_mqa_logits_topk")


def ix_paged_mqa_logits_hist(q_fp8: torch.Tensor, w: torch.Tensor, cache: torch.Tensor,
                             context_lens: torch.Tensor, block_table: torch.Tensor, logits: torch.Tensor,
                             k: int, workspace: torch.Tensor, block_size: int = BLOCK_SIZE, stream=None) -> None:
    """First half of ix_paged_mqa_logits_topk: the logits and the row histograms."""
    _rows(q_fp8, 0, "q_fp8", dim=4)
    B, next_n, H, D = q_fp8.shape
    R = B * next_n
    _rows(w, R, "w", H)
    _rows(logits, R, "logits")
    _len(context_lens, B, "context_lens")
    _rows(block_table, B, "block_table")
    _rows(cache, 0, "cache", block_size * (D + 4))
    wp, wb = _workspace(workspace, R)
    rc = load().ix_paged_mqa_logits_hist(
        _dev(q_fp8, "q_fp8", _U8), _dev(w, "w", _F32), _dev(cache, "cache", (torch.uint8,)),
        cache.shape[0], block_size, _dev(context_lens, "context_lens", _I32T),
        _dev(block_table, "block_table", _I32T), block_table.stride(0), B, next_n, H, D,
        _dev(logits, "logits", _F32), logits.shape[1], int(k), wp, wb, _stream(stream))
    _check(rc, "ix_paged_mqa_logits_hist")


def ix_mqa_logits_hist(q_fp8: torch.Tensor, w: torch.Tensor, k_fp8: torch.Tensor, k_scale: torch.Tensor,
                       ks: torch.Tensor, ke: torch.Tensor, logits: torch.Tensor, k: int, workspace: torch.Tensor,
                       stream=None) -> None:
    """First half of ix_mqa_logits_topk: the logits and the row histograms."""
    _rows(q_fp8, 0, "q_fp8", dim=3)
    tq, H, D = q_fp8.shape
    _rows(w, tq, "w", H)
    _rows(k_fp8, 0, "k_fp8", D)
    _len(k_scale, k_fp8.shape[0], "k_scale")
    _len(ks, tq, "ks")
    _len(ke, tq, "ke")
    _rows(logits, tq, "logits")
    wp, wb = _workspace(workspace, tq)
    rc = load().ix_mqa_logits_hist(
        _dev(q_fp8, "q_fp8", _U8), _dev(w, "w", _F32), _dev(k_fp8, "k_fp8", _U8),
        _dev(k_scale, "k_scale", _F32), _dev(ks, "ks", _I32T), _dev(ke, "ke", _I32T), tq, k_fp8.shape[0], H, D,
        _dev(logits, "logits", _F32), logits.shape[1], int(k), wp, wb, _stream(stream))
    _check(rc, "ix_mqa_logits_hist")


def ix_topk_from_hist(logits: torch.Tensor, row_len: torch.Tensor, row_req: torch.Tensor,
                      block_table: torch.Tensor, k: int, out_global: torch.Tensor, workspace: torch.Tensor,
                      out_local: Optional[torch.Tensor] = None, block_size: int = BLOCK_SIZE,
                      stream=None) -> None:
    """Second half of the fused calls: the selection from the row histograms."""
    _rows(logits, 0, "logits")
    R, ld = logits.shape
    _len(row_len, R, "row_len")
    _len(row_req, R, "row_req")
    _rows(block_table, 0, "block_table")
    _len(out_global, R * int(k), "out_global")
    if out_local is not None:
        _len(out_local, R * int(k), "out_local")
    wp, wb = _workspace(workspace, R)
    rc = load().ix_topk_from_hist(
        _dev(logits, "logits", _F32), ld, R, _dev(row_len, "row_len", _I32T),
        _dev(row_req, "row_req", _I32T), _dev(block_table, "block_table", _I32T),
        block_table.stride(0), block_size, int(k), _opt(out_local, "out_local", _I32T),
        _dev(out_global, "out_global", _I32T), wp, wb, _stream(stream))
    _check(rc, "ix_topk_from_hist")


def dsmla_fused_q(q_pe_bf16: torch.Tensor, positions: torch.Tensor, cos_sin: torch.Tensor,
                  quantize_mqa: bool, ql_nope_bf16: Optional[torch.Tensor] = None,
                  out_pe: Optional[torch.Tensor] = None, out_mqa: Optional[torch.Tensor] = None,
                  out_scale: Optional[torch.Tensor] = None, stream=None) -> None:
    """q_pe [T, H, 64] bf16; positions [T] int64; cos_sin [max_pos, 64] f32.
    quantize_mqa: ql_nope [T, H, 512] bf16 -> out_mqa [T, H, 576] fp8/u8 and
    out_scale [T, H] f32; else out_pe [T, H, 64] bf16 (the rotated q_pe)."""
    _rows(q_pe_bf16, 0, "q_pe", 64, dim=3)
    T, H, _ = q_pe_bf16.shape
    _len(positions, T, "positions")
    _rows(cos_sin, 0, "cos_sin", 64)
    if quantize_mqa:
        _need(ql_nope_bf16 is not None and out_mqa is not None and out_scale is not None,
              "quantize_mqa: ql_nope, out_mqa and out_scale are required")
        _need(tuple(ql_nope_bf16.shape) == (T, H, 512), f"ql_nope: shape {tuple(ql_nope_bf16.shape)}")
        _len(out_mqa, T * H * 576, "out_mqa")
        _len(out_scale, T * H, "out_scale")
    else:
        _need(out_pe is not None, "out_pe is required when quantize_mqa is False")
        _len(out_pe, T * H * 64, "out_pe")
    rc = load().dsmla_fused_q(
        _opt(ql_nope_bf16, "ql_nope", _BF16) if quantize_mqa else None, _dev(q_pe_bf16, "q_pe", _BF16),
        _dev(positions, "positions", _I64T), _dev(cos_sin, "cos_sin", _F32), cos_sin.shape[0], T, H,
        int(bool(quantize_mqa)), None if quantize_mqa else _dev(out_pe, "out_pe", _BF16),
        _dev(out_mqa, "out_mqa", _U8) if quantize_mqa else None,
        _dev(out_scale, "out_scale", _F32) if quantize_mqa else None, _stream(stream))
    _check(rc, "dsmla_fused_q")


def ix_quant_q(q_bf16: torch.Tensor, w: torch.Tensor, q_fp8: torch.Tensor, w_out: torch.Tensor,
               stream=None) -> None:
    """q [T, H, 128] bf16; w [T, H] f32 -> q_fp8 [T, H, 128] fp8/u8, w_out [T, H] f32."""
    _rows(q_bf16, 0, "q", dim=3)
    T, H, D = q_bf16.shape
    _rows(w, T, "w", H)
    _len(q_fp8, T * H * D, "q_fp8")
    _len(w_out, T * H, "w_out")
    rc = load().ix_quant_q(_dev(q_bf16, "q", _BF16), _dev(w, "w", _F32), T, H, D, _dev(q_fp8, "q_fp8", _U8),
                           _dev(w_out, "w_out", _F32), _stream(stream))
    _check(rc, "ix_quant_q")


def dsmla_quant_write(nope_bf16: torch.Tensor, rope_bf16: torch.Tensor,
                      slot_mapping: torch.Tensor, cache: torch.Tensor, stream=None) -> None:
    """nope [n, 512] bf16; rope [n, 64] bf16; cache uint8 [num_blocks, block_size, 656+]."""
    _rows(nope_bf16, 0, "nope_bf16", 512)
    n = nope_bf16.shape[0]
    _rows(rope_bf16, n, "rope_bf16", 64)
    _len(slot_mapping, n, "slot_mapping")
    _rows(cache, 0, "cache", dim=3)
    nb, bs, entry = cache.shape
    rc = load().dsmla_quant_write(
        _dev(nope_bf16, "nope_bf16", _BF16), _dev(rope_bf16, "rope_bf16", _BF16),
        nope_bf16.shape[0], _dev(slot_mapping, "slot_mapping", _I64T),
        _dev(cache, "cache", (torch.uint8,)), nb, bs, cache.stride(0), cache.stride(1),
        _stream(stream))
    _check(rc, "dsmla_quant_write")


def dsmla_norm_rope_write(kv_bf16: torch.Tensor, pe_bf16: torch.Tensor, gamma_bf16: torch.Tensor,
                          eps: float, positions: torch.Tensor, cos_sin: torch.Tensor,
                          slot_mapping: torch.Tensor, cache: torch.Tensor, stream=None) -> None:
    """kv [n, 512] bf16; pe [n, 64] bf16; gamma [512] bf16; positions [n] int64;
    cos_sin [max_pos, 64] f32; cache uint8 [num_blocks, block_size, 656+]."""
    _rows(kv_bf16, 0, "kv_bf16", 512)
    n = kv_bf16.shape[0]
    _rows(pe_bf16, n, "pe_bf16", 64)
    _len(gamma_bf16, 512, "gamma_bf16")
    _len(positions, n, "positions")
    _rows(cos_sin, 0, "cos_sin", 64)
    _len(slot_mapping, n, "slot_mapping")
    _rows(cache, 0, "cache", dim=3)
    nb, bs, entry = cache.shape
    rc = load().dsmla_norm_rope_write(
        _dev(kv_bf16, "kv_bf16", _BF16), _dev(pe_bf16, "pe_bf16", _BF16),
        _dev(gamma_bf16, "gamma_bf16", _BF16), float(eps), _dev(positions, "positions", _I64T),
        _dev(cos_sin, "cos_sin", _F32), cos_sin.shape[0], _dev(slot_mapping, "slot_mapping", _I64T),
        kv_bf16.shape[0], _dev(cache, "cache", (torch.uint8,)), nb, bs, cache.stride(0),
        cache.stride(1), _stream(stream))
    _check(rc, "dsmla_norm_rope_write")


MLA_HEADS = 128


def _sparse_decode_shapes(q_nope, q_pe, cache, indices, out, lse):
    _rows(q_nope, 0, "q_nope_bf16", 512, dim=3)
    T, H = q_nope.shape[:2]
    _rows(q_pe, T, "q_pe_bf16", 64, dim=3)
    _need(q_pe.shape[1] == H, f"q_pe_bf16: {q_pe.shape[1]} heads, q_nope_bf16 has {H}")
    _rows(indices, T, "indices")
    _rows(out, T, "out", 512, dim=3)
    _need(out.shape[1] == H, f"out: {out.shape[1]} heads, expected {H}")
    _rows(lse, T, "lse", H)
    _rows(cache, 0, "cache", dim=3)
    return T, H, indices.shape[1]


def dsmla_sparse_decode_workspace_size(tokens: int, heads: int, topk: int) -> int:
    """Bytes of scratch dsmla_sparse_decode needs for this shape."""
    return int(load().dsmla_sparse_decode_workspace_size(int(tokens), int(heads), int(topk)))


def dsmla_sparse_decode(q_nope_bf16: torch.Tensor, q_pe_bf16: torch.Tensor, cache: torch.Tensor,
                        indices: torch.Tensor, sm_scale: float, out: torch.Tensor, lse: torch.Tensor,
                        workspace: torch.Tensor, stream=None) -> None:
    """q_nope [T, 128, 512] bf16; q_pe [T, 128, 64] bf16; cache uint8
    [num_blocks, block_size, 656+]; indices int32 [T, topk] global slots (-1:
    none); out [T, 128, 512] bf16 and lse [T, 128] f32 (written); workspace
    uint8 of at least dsmla_sparse_decode_workspace_size(T, 128, topk) bytes."""
    T, H, topk = _sparse_decode_shapes(q_nope_bf16, q_pe_bf16, cache, indices, out, lse)
    nb, bs, entry = cache.shape
    rc = load().dsmla_sparse_decode(
        _dev(q_nope_bf16, "q_nope_bf16", _BF16), _dev(q_pe_bf16, "q_pe_bf16", _BF16),
        _dev(cache, "cache", (torch.uint8,)), nb, bs, cache.stride(0), cache.stride(1),
        _dev(indices, "indices", (torch.int32,)), T, H, topk, float(sm_scale),
        _dev(out, "out", _BF16), _dev(lse, "lse", _F32), _dev(workspace, "workspace", (torch.uint8,)),
        workspace.numel(), _stream(stream))
    _check(rc, "dsmla_sparse_decode")


def dsmla_sparse_decode_noalloc(q_nope_bf16: torch.Tensor, q_pe_bf16: torch.Tensor, cache: torch.Tensor,
                                indices: torch.Tensor, sm_scale: float, out: torch.Tensor, lse: torch.Tensor,
                                stream=None) -> None:
    """dsmla_sparse_decode with the library's own file-scope scratch (no
    workspace argument; tokens * ceil(topk / 256) <= 128)."""
    T, H, topk = _sparse_decode_shapes(q_nope_bf16, q_pe_bf16, cache, indices, out, lse)
    nb, bs, entry = cache.shape
    rc = load().dsmla_sparse_decode_noalloc(
        _dev(q_nope_bf16, "q_nope_bf16", _BF16), _dev(q_pe_bf16, "q_pe_bf16", _BF16),
        _dev(cache, "cache", (torch.uint8,)), nb, bs, cache.stride(0), cache.stride(1),
        _dev(indices, "indices", (torch.int32,)), T, H, topk, float(sm_scale),
        _dev(out, "out", _BF16), _dev(lse, "lse", _F32), _stream(stream))
    _check(rc, "dsmla_sparse_decode_noalloc")
