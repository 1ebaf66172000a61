"""dsmla_sparse_decode_noalloc: the sparse MLA decode without a caller
workspace, its split outputs held in the library's file-scope device scratch.

CPU: the entry point is exported and refuses a call larger than its scratch
before any CUDA call.  GPU: the results are bit-identical to the workspace
entry point (same kernels), agree with the oracle, and the call leaves torch's
allocator untouched.
"""
import ctypes
import os
import shutil

import numpy as np
import pytest

IX_OK, IX_ERR_SHAPE, IX_ERR_UNSUPPORTED, IX_ERR_WORKSPACE = 0, -2, -3, -5
A16 = ctypes.c_void_p(0x10000)

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def lib():
    from deepseek_v3_sparse_gb300 import build
    import deepseek_v3_sparse_gb300 as dsix
    build.build()
    return dsix.load()


@needs_nvcc
def test_noalloc_is_exported_and_checks_capacity_on_the_host(lib):
    f = lib.dsmla_sparse_decode_noalloc

    def call(tokens, topk, heads=128):
        return f(A16, A16, A16, 8, 64, 64 * 656, 656, A16, tokens, heads, topk, 0.07, A16, A16, None)

    assert call(17, 2048) == IX_ERR_WORKSPACE      # 17 tokens x 8 splits > 128
    assert call(129, 1) == IX_ERR_WORKSPACE
    assert call(1, 65536) == IX_ERR_WORKSPACE      # 256 splits of one token > 128
    assert call(9, 3840) == IX_ERR_WORKSPACE       # 9 x 15 = 135
    assert call(-1, 64) == IX_ERR_SHAPE
    assert call(2, 64, heads=64) == IX_ERR_UNSUPPORTED
    assert call(0, 64) == IX_OK


@needs_nvcc
def test_noalloc_runs_the_workspace_calls_checks_first(lib):
    """An oversized call with a bad argument reports the same error as the
    workspace entry point would: the capacity check takes the place of the
    workspace check, after every other host check."""
    f = lib.dsmla_sparse_decode_noalloc
    big, unaligned = 17, ctypes.c_void_p(0x10008)
    # NULL query: IX_ERR_NULL, not IX_ERR_WORKSPACE
    assert f(None, A16, A16, 8, 64, 64 * 656, 656, A16, big, 128, 2048, 0.07, A16, A16, None) == -1
    # entry stride below 656: IX_ERR_SHAPE
    assert f(A16, A16, A16, 8, 64, 64 * 656, 640, A16, big, 128, 2048, 0.07, A16, A16, None) == IX_ERR_SHAPE
    # misaligned output: IX_ERR_ALIGN
    assert f(A16, A16, A16, 8, 64, 64 * 656, 656, A16, big, 128, 2048, 0.07, unaligned, A16, None) == -4
    # sm_scale not positive: IX_ERR_UNSUPPORTED
    assert f(A16, A16, A16, 8, 64, 64 * 656, 656, A16, big, 128, 2048, 0.0, A16, A16, None) == IX_ERR_UNSUPPORTED
    # block_size < 1: IX_ERR_UNSUPPORTED
    assert f(A16, A16, A16, 8, 0, 64 * 656, 656, A16, big, 128, 2048, 0.07, A16, A16, None) == IX_ERR_UNSUPPORTED
    # the same calls through the workspace entry point give the same codes
    g = lib.dsmla_sparse_decode
    assert g(None, A16, A16, 8, 64, 64 * 656, 656, A16, big, 128, 2048, 0.07, A16, A16, A16, 1 << 40, None) == -1
    assert g(A16, A16, A16, 8, 64, 64 * 656, 640, A16, big, 128, 2048, 0.07, A16, A16, A16, 1 << 40,
             None) == IX_ERR_SHAPE


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_and_oracle():
    from tests._helpers import require_gpu
    require_gpu()
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import deepseek_v3_sparse_gb300 as dsix
    import oracle
    import workloads as W

    x = W.sparse_decode_inputs(16, 2048, 4096, seed=23)
    dense = np.zeros((x.num_blocks, 64, 656), np.uint8)
    oracle.dsmla_quant_write(W.bf16_bits(x.nope_bf16), W.bf16_bits(x.rope_bf16), x.slots, dense, 64)
    cache = torch.from_numpy(dense).cuda()
    qn, qp, idx = x.q_nope.cuda(), x.q_pe.cuda(), torch.from_numpy(x.indices).cuda()
    out_a = torch.empty(16, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse_a = torch.empty(16, 128, dtype=torch.float32, device="cuda")
    out_b, lse_b = torch.empty_like(out_a), torch.empty_like(lse_a)
    ws = torch.empty(dsix.dsmla_sparse_decode_workspace_size(16, 128, 2048), dtype=torch.uint8, device="cuda")
    dsix.dsmla_sparse_decode(qn, qp, cache, idx, x.sm_scale, out_a, lse_a, ws)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    dsix.dsmla_sparse_decode_noalloc(qn, qp, cache, idx, x.sm_scale, out_b, lse_b)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    assert dsix.ix_device_status() == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)
    ref_o, ref_l, ok = oracle.dsmla_sparse_decode(W.bf16_bits(x.q_nope), W.bf16_bits(x.q_pe), dense, 64,
                                                  x.indices, x.sm_scale)
    assert ok
    named = dense.reshape(-1, 656)[x.indices.reshape(-1)]
    vmax = float((torch.from_numpy(named[:, :512].copy()).view(torch.float8_e4m3fn).double() *
                  torch.from_numpy(named[:, 512:528].copy()).view(torch.float32).double()
                  .repeat_interleave(128, dim=1)).abs().max())
    got = out_b.double().cpu().numpy()
    assert np.all(np.abs(got - ref_o) <= 2.0 ** -8 * np.abs(ref_o) + 2.0 ** -7 * vmax)
    assert np.all(np.abs(lse_b.double().cpu().numpy() - ref_l) <= 2.0 ** -7 + 2.0 ** -9 * np.abs(ref_l))
    # a second call in a row, on other inputs (4 tokens, top-1024): the scratch
    # keeps the first call's contents, none of which may leak into this result
    y = W.sparse_decode_inputs(4, 1024, 2048, seed=29)
    dense_y = np.zeros((y.num_blocks, 64, 656), np.uint8)
    oracle.dsmla_quant_write(W.bf16_bits(y.nope_bf16), W.bf16_bits(y.rope_bf16), y.slots, dense_y, 64)
    cache_y = torch.from_numpy(dense_y).cuda()
    qn_y, qp_y, idx_y = y.q_nope.cuda(), y.q_pe.cuda(), torch.from_numpy(y.indices).cuda()
    out_c = torch.empty(4, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse_c = torch.empty(4, 128, dtype=torch.float32, device="cuda")
    out_d, lse_d = torch.empty_like(out_c), torch.empty_like(lse_c)
    ws_y = torch.empty(dsix.dsmla_sparse_decode_workspace_size(4, 128, 1024), dtype=torch.uint8, device="cuda")
    dsix.dsmla_sparse_decode(qn_y, qp_y, cache_y, idx_y, y.sm_scale, out_c, lse_c, ws_y)
    dsix.dsmla_sparse_decode_noalloc(qn_y, qp_y, cache_y, idx_y, y.sm_scale, out_d, lse_d)
    torch.cuda.synchronize()
    assert dsix.ix_device_status() == 0
    assert torch.equal(out_c.view(torch.int16), out_d.view(torch.int16))
    assert torch.equal(lse_c, lse_d)
    with pytest.raises(dsix.DsixError):      # 17 tokens x 8 splits do not fit the scratch
        dsix.dsmla_sparse_decode_noalloc(torch.cat([qn, qn[:1]]), torch.cat([qp, qp[:1]]), cache,
                                         torch.cat([idx, idx[:1]]), x.sm_scale,
                                         torch.empty(17, 128, 512, dtype=torch.bfloat16, device="cuda"),
                                         torch.empty(17, 128, dtype=torch.float32, device="cuda"))
