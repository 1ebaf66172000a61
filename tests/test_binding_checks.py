"""Host-side shape checks of the Python binding (CPU only: no kernel runs).

The C entry points receive bare pointers, so a tensor whose shape disagrees
with the others would be read or written past its end.  The binding refuses
such calls before touching a pointer.  With CPU tensors of consistent shapes a
call gets past the shape checks and stops at the device check ("must be a
CUDA tensor"); each inconsistent shape stops earlier, naming the tensor.
"""
import os
import shutil

import pytest
import torch

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def dsix():
    from deepseek_v3_sparse_gb300 import build
    import deepseek_v3_sparse_gb300 as m
    build.build()
    m.load()
    return m


def u8(*s):
    return torch.zeros(*s, dtype=torch.uint8)


def bf(*s):
    return torch.zeros(*s, dtype=torch.bfloat16)


def f32(*s):
    return torch.zeros(*s, dtype=torch.float32)


def i32(*s):
    return torch.zeros(*s, dtype=torch.int32)


def i64(*s):
    return torch.zeros(*s, dtype=torch.int64)


def passes_shape_checks(fn, *args, **kw):
    with pytest.raises(Exception) as e:
        fn(*args, **kw)
    return "must be a CUDA tensor" in str(e.value)


def refused(fn, name, *args, **kw):
    with pytest.raises(Exception) as e:
        fn(*args, **kw)
    msg = str(e.value)
    return name in msg and "CUDA tensor" not in msg


def test_quant_write_and_gather(dsix):
    f = dsix.ix_quant_write_k
    assert passes_shape_checks(f, bf(5, 128), i64(5), u8(3, 8448))
    assert refused(f, "slot_mapping", bf(5, 128), i64(4), u8(3, 8448))
    assert refused(f, "cache", bf(5, 128), i64(5), u8(3 * 8448))
    assert refused(f, "cache", bf(5, 128), i64(5), u8(3, 8192))
    g = dsix.ix_gather_k
    assert passes_shape_checks(g, u8(3, 8448), i32(2, 3), i32(3), u8(10, 128), f32(10))
    assert refused(g, "block_table", u8(3, 8448), i32(1, 3), i32(3), u8(10, 128), f32(10))
    assert refused(g, "out_scale", u8(3, 8448), i32(2, 3), i32(3), u8(10, 128), f32(9))
    assert refused(g, "out_k", u8(3, 8448), i32(2, 3), i32(3), u8(10, 64), f32(10))


def test_logits(dsix):
    p = dsix.ix_paged_mqa_logits
    args = [u8(4, 2, 64, 128), f32(8, 64), u8(3, 8448), i32(4), i32(4, 3), f32(8, 256)]
    assert passes_shape_checks(p, *args)
    for i, name, bad in [(1, "w", f32(7, 64)), (1, "w", f32(8, 32)), (5, "logits", f32(7, 256)),
                         (3, "context_lens", i32(3)), (4, "block_table", i32(3, 3)),
                         (0, "q_fp8", u8(8, 64, 128))]:
        a = list(args)
        a[i] = bad
        assert refused(p, name, *a), name
    m = dsix.ix_mqa_logits
    args = [u8(6, 64, 128), f32(6, 64), u8(40, 128), f32(40), i32(6), i32(6), f32(6, 40)]
    assert passes_shape_checks(m, *args)
    for i, name, bad in [(1, "w", f32(5, 64)), (3, "k_scale", f32(39)), (4, "ks", i32(5)),
                         (5, "ke", i32(5)), (6, "logits", f32(5, 40)), (2, "k_fp8", u8(40, 64))]:
        a = list(args)
        a[i] = bad
        assert refused(m, name, *a), name


def test_topk(dsix):
    t = dsix.ix_topk_to_global
    assert passes_shape_checks(t, f32(4, 100), i32(4), i32(4), i32(4, 2), 16, i32(4, 16))
    assert passes_shape_checks(t, f32(4, 100), i32(4), i32(4), i32(4, 2), 16, i32(4, 16), i32(4, 16))
    assert refused(t, "row_len", f32(4, 100), i32(3), i32(4), i32(4, 2), 16, i32(4, 16))
    assert refused(t, "row_req", f32(4, 100), i32(4), i32(3), i32(4, 2), 16, i32(4, 16))
    assert refused(t, "out_global", f32(4, 100), i32(4), i32(4), i32(4, 2), 16, i32(4, 15))
    assert refused(t, "out_local", f32(4, 100), i32(4), i32(4), i32(4, 2), 16, i32(4, 16), i32(3, 16))


def test_dsmla_writes(dsix):
    w = dsix.dsmla_quant_write
    assert passes_shape_checks(w, bf(5, 512), bf(5, 64), i64(5), u8(2, 64, 656))
    assert refused(w, "rope_bf16", bf(5, 512), bf(4, 64), i64(5), u8(2, 64, 656))
    assert refused(w, "nope_bf16", bf(5, 500), bf(5, 64), i64(5), u8(2, 64, 656))
    assert refused(w, "slot_mapping", bf(5, 512), bf(5, 64), i64(4), u8(2, 64, 656))
    assert refused(w, "cache", bf(5, 512), bf(5, 64), i64(5), u8(2 * 64, 656))
    n = dsix.dsmla_norm_rope_write
    args = [bf(5, 512), bf(5, 64), bf(512), 1e-6, i64(5), f32(9, 64), i64(5), u8(2, 64, 656)]
    assert passes_shape_checks(n, *args)
    for i, name, bad in [(1, "pe_bf16", bf(5, 32)), (2, "gamma_bf16", bf(256)), (4, "positions", i64(4)),
                         (5, "cos_sin", f32(9, 32)), (6, "slot_mapping", i64(2))]:
        a = list(args)
        a[i] = bad
        assert refused(n, name, *a), name


def test_sparse_decode(dsix):
    for fn, extra in ((dsix.dsmla_sparse_decode, [u8(64)]), (dsix.dsmla_sparse_decode_noalloc, [])):
        args = [bf(3, 128, 512), bf(3, 128, 64), u8(4, 64, 656), i32(3, 300), 0.07, bf(3, 128, 512),
                f32(3, 128)] + extra
        assert passes_shape_checks(fn, *args)
        for i, name, bad in [(1, "q_pe_bf16", bf(2, 128, 64)), (1, "q_pe_bf16", bf(3, 64, 64)),
                             (3, "indices", i32(2, 300)), (5, "out", bf(3, 128, 256)),
                             (5, "out", bf(2, 128, 512)), (6, "lse", f32(3, 64)),
                             (2, "cache", u8(4, 64 * 656)), (0, "q_nope_bf16", bf(3, 128, 576))]:
            a = list(args)
            a[i] = bad
            assert refused(fn, name, *a), (fn.__name__, name)


def test_step_calls_pass_the_checks(dsix, monkeypatch):
    # Every call one indexer step makes (decode, MTP decode, mixed decode +
    # prefill) satisfies the shape checks: the step is built on the CPU and run
    # against a stand-in library that accepts any call.
    import workloads as W
    from workloads.device import make_step

    seen = []

    class AnyCall:
        def __getattr__(self, name):
            return lambda *a: seen.append(name) or 0

    def dev(t, name, dtypes):
        assert t.dtype in dtypes and t.is_contiguous(), name
        return 0

    monkeypatch.setattr(dsix, "_dev", dev)
    monkeypatch.setattr(dsix, "load", lambda path=None: AnyCall())
    monkeypatch.setattr(dsix, "_stream", lambda s: 0)
    for wl in (W.tiny_decode(), W.build("mtp", decode_ctx=[300, 700], next_n=2, topk=64, seed=1),
               W.build("mix", decode_ctx=[500], next_n=1, prefill=[(900, 300), (400, 400)], topk=128, seed=2)):
        seen.clear()
        make_step(wl, "cpu").run()
        assert "ix_paged_mqa_logits" in seen and "ix_topk_to_global" in seen


def test_tensor_on_another_device_is_refused(dsix, monkeypatch):
    """The library launches on the current device; a tensor that lives on
    another one is refused before its pointer is taken (a CUDA tensor is faked
    on the CPU: nothing is launched)."""
    class OnCuda1(torch.Tensor):
        @property
        def is_cuda(self):
            return True

        @property
        def device(self):
            return torch.device("cuda", 1)

    t = torch.zeros(16, dtype=torch.float32).as_subclass(OnCuda1)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(dsix.DsixError, match="current device"):
        dsix._dev(t, "logits", (torch.float32,))
