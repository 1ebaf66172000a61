"""The C ABI library (CPU only: no kernel is launched).

* libdsix.so builds for sm_103a and loads;
* it exports exactly the functions include/dsix.h declares;
* every host-side argument check returns its status code before anything
  touches the GPU.
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsix.h")

IX_OK, IX_ERR_NULL, IX_ERR_SHAPE, IX_ERR_UNSUPPORTED, IX_ERR_ALIGN, IX_ERR_WORKSPACE = 0, -1, -2, -3, -4, -5

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def lib():
    from deepseek_v3_sparse_gb300 import build
    import deepseek_v3_sparse_gb300 as dsix
    build.build()
    return dsix.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"IX_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_exports_match_header(lib):
    names = _declared()
    assert len(names) == 20
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines()
                      if l.split()[-2:-1] == ["T"] and not l.split()[-1].startswith("_"))
    assert exported == names


def test_status_strings(lib):
    import deepseek_v3_sparse_gb300 as dsix
    for code in range(0, -8, -1):
        s = dsix.ix_status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in dsix.ix_status_string(-99)


P = ctypes.c_void_p
A16 = P(0x10000)      # aligned fake device address (never dereferenced by the checks)
A1 = P(0x10001)       # misaligned


def test_quant_write_k_host_checks(lib):
    f = lib.ix_quant_write_k
    assert f(A16, 4, 64, A16, A16, 8, 64, None) == IX_ERR_UNSUPPORTED
    assert f(A16, 4, 128, A16, A16, 8, 32, None) == IX_ERR_UNSUPPORTED
    assert f(A16, -1, 128, A16, A16, 8, 64, None) == IX_ERR_SHAPE
    assert f(None, 4, 128, A16, A16, 8, 64, None) == IX_ERR_NULL
    assert f(A1, 4, 128, A16, A16, 8, 64, None) == IX_ERR_ALIGN
    assert f(None, 0, 128, None, None, 8, 64, None) == IX_OK   # empty: nothing to do


def test_gather_host_checks(lib):
    f = lib.ix_gather_k
    assert f(A16, 8, 64, 64, A16, 4, A16, 2, A16, A16, 100, None) == IX_ERR_UNSUPPORTED
    assert f(A16, 8, 64, 128, A16, 4, A16, -1, A16, A16, 100, None) == IX_ERR_SHAPE
    assert f(A16, 8, 64, 128, None, 4, A16, 2, A16, A16, 100, None) == IX_ERR_NULL
    assert f(A16, 8, 64, 128, A16, 4, A16, 2, A1, A16, 100, None) == IX_ERR_ALIGN
    assert f(A16, 8, 64, 128, A16, 4, A16, 0, A16, A16, 100, None) == IX_OK


def test_paged_logits_host_checks(lib):
    f = lib.ix_paged_mqa_logits
    args = lambda **kw: [kw.get("q", A16), A16, A16, kw.get("nb", 8), kw.get("bs", 64), A16, A16,
                         4, kw.get("batch", 2), kw.get("next_n", 1), kw.get("heads", 64),
                         kw.get("dim", 128), kw.get("logits", A16), kw.get("ld", 64), 0, None]
    assert f(*args(heads=32)) == IX_ERR_UNSUPPORTED
    assert f(*args(next_n=3)) == IX_ERR_UNSUPPORTED
    assert f(*args(bs=16)) == IX_ERR_UNSUPPORTED
    assert f(*args(ld=66)) == IX_ERR_UNSUPPORTED
    assert f(*args(batch=-1)) == IX_ERR_SHAPE
    assert f(*args(nb=0)) == IX_ERR_SHAPE
    assert f(*args(q=None)) == IX_ERR_NULL
    assert f(*args(logits=A1)) == IX_ERR_ALIGN
    assert f(*args(batch=0)) == IX_OK


def test_mqa_logits_host_checks(lib):
    f = lib.ix_mqa_logits
    args = lambda **kw: [kw.get("q", A16), A16, kw.get("k", A16), A16, A16, A16, kw.get("tq", 16),
                         kw.get("tk", 16), kw.get("heads", 64), 128, A16, kw.get("ld", 16), 0, None]
    assert f(*args(heads=16)) == IX_ERR_UNSUPPORTED
    assert f(*args(ld=18)) == IX_ERR_UNSUPPORTED
    assert f(*args(tq=-2)) == IX_ERR_SHAPE
    assert f(*args(k=None)) == IX_ERR_NULL
    assert f(*args(q=A1)) == IX_ERR_ALIGN
    assert f(*args(tq=0)) == IX_OK


def test_topk_host_checks(lib):
    f = lib.ix_topk_to_global
    args = lambda **kw: [kw.get("lg", A16), kw.get("ld", 64), kw.get("rows", 4), A16, A16, A16, 8,
                         64, kw.get("k", 16), None, kw.get("out", A16), None]
    assert f(*args(k=0)) == IX_ERR_UNSUPPORTED
    assert f(*args(ld=62)) == IX_ERR_UNSUPPORTED
    assert f(*args(ld=8 * 32768 + 4)) == IX_ERR_UNSUPPORTED
    assert f(*args(rows=-1)) == IX_ERR_SHAPE
    assert f(*args(out=None)) == IX_ERR_NULL
    assert f(*args(lg=A1)) == IX_ERR_ALIGN
    assert f(*args(rows=0)) == IX_OK


def test_fused_topk_host_checks(lib):
    """The fused logits + top-k calls and their halves check every argument on
    the host (the logits call's checks first, then k / ld / workspace, then the
    top-k outputs) before any CUDA call."""
    ws = lib.ix_topk_hist_workspace_size
    assert ws(3) == 3 * (64 + 2048) * 4 and ws(0) == 0 and ws(-1) == 0
    need = ws(2)
    f = lib.ix_paged_mqa_logits_topk

    def pargs(**kw):
        return [kw.get("q", A16), A16, A16, 8, 64, A16, A16, 4, kw.get("batch", 2), 1, kw.get("heads", 64), 128,
                A16, kw.get("ld", 64), kw.get("k", 16), None, kw.get("out", A16), kw.get("ws", A16),
                kw.get("ws_bytes", need), None]

    assert f(*pargs(heads=32)) == IX_ERR_UNSUPPORTED        # the logits checks come first
    assert f(*pargs(q=None, ws=None)) == IX_ERR_NULL
    assert f(*pargs(k=0)) == IX_ERR_UNSUPPORTED
    assert f(*pargs(ld=262148)) == IX_ERR_UNSUPPORTED
    assert f(*pargs(ws=None)) == IX_ERR_WORKSPACE
    assert f(*pargs(ws_bytes=need - 1)) == IX_ERR_WORKSPACE
    assert f(*pargs(ws=A1)) == IX_ERR_ALIGN
    assert f(*pargs(out=None)) == IX_ERR_NULL
    assert f(*pargs(batch=0, q=None, ws=None, out=None)) == IX_OK
    h = lib.ix_paged_mqa_logits_hist
    hargs = lambda **kw: pargs(**kw)[:15] + [kw.get("ws", A16), kw.get("ws_bytes", need), None]
    assert h(*hargs(k=0)) == IX_ERR_UNSUPPORTED
    assert h(*hargs(ws=None)) == IX_ERR_WORKSPACE
    assert h(*hargs(batch=0, q=None)) == IX_OK

    g = lib.ix_mqa_logits_topk
    need16 = ws(16)

    def cargs(**kw):
        return [kw.get("q", A16), A16, A16, A16, A16, A16, kw.get("tq", 16), 16, 64, 128, A16, kw.get("ld", 16),
                kw.get("req", A16), kw.get("bt", A16), kw.get("bts", 8), kw.get("bs", 64), kw.get("k", 4), None,
                kw.get("out", A16), kw.get("ws", A16), kw.get("ws_bytes", need16), None]

    assert g(*cargs(ld=18)) == IX_ERR_UNSUPPORTED
    assert g(*cargs(k=0)) == IX_ERR_UNSUPPORTED
    assert g(*cargs(ws_bytes=need16 - 4)) == IX_ERR_WORKSPACE
    assert g(*cargs(bts=-1)) == IX_ERR_SHAPE
    assert g(*cargs(bs=0)) == IX_ERR_UNSUPPORTED
    assert g(*cargs(req=None)) == IX_ERR_NULL
    assert g(*cargs(bt=None)) == IX_ERR_NULL
    assert g(*cargs(out=None)) == IX_ERR_NULL
    assert g(*cargs(tq=0)) == IX_OK
    c = lib.ix_mqa_logits_hist
    assert c(A16, A16, A16, A16, A16, A16, 16, 16, 64, 128, A16, 16, 0, A16, need16, None) == IX_ERR_UNSUPPORTED
    assert c(A16, A16, A16, A16, A16, A16, 16, 16, 64, 128, A16, 16, 4, None, need16, None) == IX_ERR_WORKSPACE

    t = lib.ix_topk_from_hist
    targs = lambda **kw: [A16, kw.get("ld", 64), kw.get("rows", 2), A16, A16, A16, 8, 64, kw.get("k", 16), None,
                          kw.get("out", A16), kw.get("ws", A16), kw.get("ws_bytes", need), None]
    assert t(*targs(k=0)) == IX_ERR_UNSUPPORTED
    assert t(*targs(ld=62)) == IX_ERR_UNSUPPORTED
    assert t(*targs(rows=-1)) == IX_ERR_SHAPE
    assert t(*targs(out=None)) == IX_ERR_NULL
    assert t(*targs(ws=None)) == IX_ERR_WORKSPACE
    assert t(*targs(ws=A1)) == IX_ERR_ALIGN
    assert t(*targs(rows=0)) == IX_OK


def test_query_side_host_checks(lib):
    f = lib.dsmla_fused_q
    args = lambda **kw: [kw.get("qn", A16), kw.get("qp", A16), kw.get("pos", A16), A16, kw.get("max_pos", 8),
                         kw.get("T", 4), kw.get("H", 128), kw.get("quant", 1), kw.get("pe", A16),
                         kw.get("mqa", A16), kw.get("sc", A16), None]
    assert f(*args(T=-1)) == IX_ERR_SHAPE
    assert f(*args(max_pos=-1)) == IX_ERR_SHAPE
    assert f(*args(H=0)) == IX_ERR_UNSUPPORTED
    assert f(*args(qp=None)) == IX_ERR_NULL
    assert f(*args(qn=None)) == IX_ERR_NULL                 # read when quantising
    assert f(*args(pe=None, quant=0)) == IX_ERR_NULL
    assert f(*args(mqa=P(0x10004))) == IX_ERR_ALIGN
    assert f(*args(qp=P(0x10002))) == IX_ERR_ALIGN
    assert f(*args(pos=P(0x10004))) == IX_ERR_ALIGN
    assert f(*args(T=0, qn=None, qp=None, pos=None)) == IX_OK
    g = lib.ix_quant_q
    gargs = lambda **kw: [kw.get("q", A16), A16, kw.get("T", 4), kw.get("H", 64), kw.get("D", 128),
                          kw.get("out", A16), A16, None]
    assert g(*gargs(T=-1)) == IX_ERR_SHAPE
    assert g(*gargs(D=64)) == IX_ERR_UNSUPPORTED
    assert g(*gargs(H=0)) == IX_ERR_UNSUPPORTED
    assert g(*gargs(q=None)) == IX_ERR_NULL
    assert g(*gargs(q=P(0x10008))) == IX_ERR_ALIGN
    assert g(*gargs(out=P(0x10004))) == IX_ERR_ALIGN
    assert g(*gargs(T=0)) == IX_OK


def test_dsmla_host_checks(lib):
    f = lib.dsmla_quant_write
    assert f(A16, A16, 4, A16, A16, 8, 64, 64 * 656, 600, None) == IX_ERR_SHAPE
    assert f(A16, A16, 4, A16, A16, 8, 64, 64 * 656, 660, None) == IX_ERR_ALIGN
    assert f(A16, A16, 4, A16, A1, 8, 64, 64 * 656, 656, None) == IX_ERR_ALIGN
    assert f(None, A16, 4, A16, A16, 8, 64, 64 * 656, 656, None) == IX_ERR_NULL
    assert f(None, None, 0, None, None, 8, 64, 64 * 656, 656, None) == IX_OK


def test_dsmla_norm_rope_host_checks(lib):
    f = lib.dsmla_norm_rope_write
    args = lambda **kw: [kw.get("kv", A16), kw.get("pe", A16), kw.get("g", A16), 1e-6,
                         kw.get("pos", A16), A16, kw.get("max_pos", 16), A16, kw.get("n", 4),
                         kw.get("cache", A16), 8, 64, 64 * 656, kw.get("entry", 656), None]
    assert f(*args(entry=600)) == IX_ERR_SHAPE
    assert f(*args(max_pos=-1)) == IX_ERR_SHAPE
    assert f(*args(n=-1)) == IX_ERR_SHAPE
    assert f(*args(entry=660)) == IX_ERR_ALIGN
    assert f(*args(kv=A1)) == IX_ERR_ALIGN
    assert f(*args(g=P(0x10004))) == IX_ERR_ALIGN
    assert f(*args(pos=P(0x10004))) == IX_ERR_ALIGN
    assert f(*args(pe=None)) == IX_ERR_NULL
    assert f(*args(cache=None)) == IX_ERR_NULL
    assert f(*args(kv=None, pe=None, g=None, pos=None, cache=None, n=0)) == IX_OK


def test_dsmla_sparse_decode_host_checks(lib):
    f = lib.dsmla_sparse_decode
    ws = lib.dsmla_sparse_decode_workspace_size
    # 3 tokens x 128 heads x ceil(600 / 256) = 3 splits, 513 floats per (split, head)
    assert ws(3, 128, 600) == 3 * 3 * 128 * 513 * 4
    assert ws(0, 128, 600) == 0 and ws(3, 128, 0) == 0
    need = ws(3, 128, 600)

    def args(**kw):
        return [kw.get("qn", A16), kw.get("qp", A16), kw.get("cache", A16), 8, 64, kw.get("bstride", 64 * 656),
                kw.get("entry", 656), kw.get("idx", A16), kw.get("tokens", 3), kw.get("heads", 128),
                kw.get("topk", 600), kw.get("scale", 0.07), kw.get("out", A16), kw.get("lse", A16),
                kw.get("ws", A16), kw.get("ws_bytes", need), None]

    assert f(*args(tokens=-1)) == IX_ERR_SHAPE
    assert f(*args(heads=64)) == IX_ERR_UNSUPPORTED
    assert f(*args(topk=0)) == IX_ERR_UNSUPPORTED
    assert f(*args(topk=65537)) == IX_ERR_UNSUPPORTED
    assert f(*args(scale=0.0)) == IX_ERR_UNSUPPORTED
    assert f(*args(scale=float("inf"))) == IX_ERR_UNSUPPORTED
    assert f(*args(qn=None)) == IX_ERR_NULL
    assert f(*args(idx=None)) == IX_ERR_NULL
    assert f(*args(entry=640)) == IX_ERR_SHAPE
    assert f(*args(bstride=63 * 656)) == IX_ERR_SHAPE
    assert f(*args(entry=664, bstride=64 * 664)) == IX_ERR_ALIGN
    assert f(*args(qp=A1)) == IX_ERR_ALIGN
    assert f(*args(out=P(0x10008))) == IX_ERR_ALIGN
    assert f(*args(idx=P(0x10002))) == IX_ERR_ALIGN
    assert f(*args(ws=None)) == IX_ERR_WORKSPACE
    assert f(*args(ws_bytes=need - 1)) == IX_ERR_WORKSPACE
    assert f(*args(tokens=0, qn=None, qp=None, cache=None, idx=None, out=None, lse=None, ws=None)) == IX_OK


def test_binding_fails_loudly_without_library(tmp_path):
    import deepseek_v3_sparse_gb300 as dsix
    with pytest.raises(dsix.DsixError):
        dsix.load(str(tmp_path / "missing.so"))
