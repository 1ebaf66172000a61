"""Benchmark of the DeepSeek-V3.2 sparse-attention indexer hot path on GB300.

One step = the whole hot path over one batch of the long-context mixed
workload (16 decode requests at context 131072 + 4 prefill chunks of 2048
query tokens on 8192-token contexts; top_k 2048):
  indexer-K quant-write and fp8_ds_mla write of the 8208 new tokens, paged
  gather of the prefill contexts, prefill FP8 logits (tcgen05), decode FP8
  logits over the paged cache (tcgen05), top-k + remap of all 8208 rows.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

value = query tokens (decode + prefill rows) per second over all ranks.
Multi-GPU runs are independent replicas (one process per GPU, no collective on
the data path; barrier + max-over-ranks timing only).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "indexer decode query-tokens/s and prefill TFLOP/s; HBM GB/s & FP8 roofline fraction"
UNIT = "query-tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DECODE_BYTES_PER_KEY = 132        # 128 fp8 values + one fp32 scale
PREFILL_FLOP_PER_PAIR = 2 * 64 * 128
NORM_ROPE_BYTES_PER_TOKEN = 1024 + 128 + 8 + 8 + 256 + 656  # fused norm/RoPE ds_mla write
SPARSE_DECODE_ENTRY = 656  # bytes of one fp8_ds_mla entry read by the sparse MLA decode
# the query side, per query token: dsmla_fused_q with quantize_mqa over 128 heads
# (1024 + 128 B read, 576 + 4 B written per head; 8 B position + 256 B table row
# per token) and ix_quant_q over 64 heads (256 + 4 B read, 128 + 4 B written)
QUERY_BYTES_PER_TOKEN = {
    "dsmla_fused_q": (128 * (1024 + 128 + 576 + 4) + 8 + 256,
                      "128 heads x (1152 B bf16 in + 580 B fp8 query and scale out) + 264 B position and table row"),
    "ix_quant_q": (64 * (256 + 4 + 128 + 4), "64 heads x (260 B in + 132 B out)"),
}


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "traffic_mixed_long.txt")
KERNEL_SOURCES = {
    "mqa_logits": ("deepseek_v3_sparse_gb300/csrc/logits.cu", "deepseek_v3_sparse_gb300/csrc/common.cuh"),
    "paged_mqa_logits": ("deepseek_v3_sparse_gb300/csrc/logits.cu", "deepseek_v3_sparse_gb300/csrc/common.cuh"),
    "topk_decode": ("deepseek_v3_sparse_gb300/csrc/topk.cu", "deepseek_v3_sparse_gb300/csrc/common.cuh"),
    "topk_prefill": ("deepseek_v3_sparse_gb300/csrc/topk.cu", "deepseek_v3_sparse_gb300/csrc/common.cuh"),
}


def measured_traffic(workload_name):
    """DRAM bytes per launch from the committed ncu capture, per kernel, for the
    kernels whose sources still hash to the captured build (others: None)."""
    import hashlib
    out = {}
    if not os.path.exists(TRAFFIC_PROFILE):
        return out
    sources, kernels, wl = {}, {}, None
    with open(TRAFFIC_PROFILE) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "workload":
                wl = t[1]
            elif t[0] == "source":
                sources[t[1]] = t[2]
            elif t[0] == "kernel":
                kv = dict(zip(t[2::2], t[3::2]))
                kernels[t[1]] = int(kv["read"]) + int(kv["write"])
    if wl != workload_name:
        return out
    def current(path):
        with open(os.path.join(ROOT, path), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()
    for name, nbytes in kernels.items():
        srcs = KERNEL_SOURCES.get(name, ())
        if srcs and all(sources.get(src) == current(src) for src in srcs):
            out[name] = nbytes
    return out


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def sparse_decode_line(d, pk):
    """Bench entry of the sparse MLA decode: tokens/s and both rooflines.
    Per token (128 heads, topk indices, all valid): 2 * 128 * topk * (576 + 512)
    flop; bytes = topk * (656 entry + 4 index) + 128 * (576 * 2 query + 512 * 2
    output + 4 lse)."""
    T, topk, ms = d["units"], d["topk"], d["ms"]
    flop = 2.0 * 128 * d["valid"] * (576 + 512)
    byts = T * (topk * (SPARSE_DECODE_ENTRY + 4) + 128 * (576 * 2 + 512 * 2 + 4))
    tfs = flop / (ms / 1e3) / 1e12
    gbs = byts / (ms / 1e3) / 1e9
    return {"ms": ms, "tokens_per_s": T / (ms / 1e3), "units": T, "topk": topk, "heads": 128,
            "tensor": {"achieved": tfs, "unit": "TFLOP/s", "peak": pk["bf16_tflops"],
                       "frac": tfs / pk["bf16_tflops"], "per_unit": "2*128*topk*(576+512) flop per token"},
            "hbm": {"achieved": gbs, "unit": "GB/s", "peak": pk["hbm_gbs"], "frac": gbs / pk["hbm_gbs"],
                    "per_unit": "topk*660 + 128*(1152+1024+4) B per token"},
            "bound": "tensor" if flop / (pk["bf16_tflops"] * 1e12) > byts / (pk["hbm_gbs"] * 1e9) else "hbm",
            "l2": "flushed between launches (256 MB read)"}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, rows_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job rows per second: every rank runs the same per-rank workload
    (weak scaling), and the elapsed time is the slowest rank's."""
    return world * rows_per_step * steps / (elapsed_ms / 1e3)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = str(device_index)
        try:  # nvidia-smi numbering can differ from CUDA's; the UUID cannot
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self.dev = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def workload_config(wl):
    return {"workload": wl.name, "decode_requests": wl.n_decode,
            "decode_context": int(wl.context_lens.max()) if wl.n_decode else 0,
            "next_n": wl.next_n, "prefill_chunks": len(wl.prefill_req),
            "prefill_chunk_len": wl.chunk_len[0] if wl.chunk_len else 0,
            "prefill_context": int(wl.req_ctx[wl.prefill_req[0]]) if wl.prefill_req else 0,
            "top_k": wl.topk, "block_size": wl.block_size, "heads": wl.heads,
            "head_dim": wl.head_dim, "new_tokens": int(wl.is_new.sum()),
            "l2": "no flush: inputs larger than L2 (about 0.6 GB touched per step)"}


def algorithmic(wl):
    dec_keys = int(wl.decode_rows()[0].astype(np.int64).sum()) if wl.n_decode else 0
    if wl.n_decode and wl.next_n > 1:  # keys are read once per request
        dec_keys = int(wl.context_lens.astype(np.int64).sum())
    pairs = int(wl.prefill_rows()[2].astype(np.int64).sum()) if wl.prefill_req else 0
    return dec_keys, pairs


def spread(ms_list):
    """min / median / max (ms) of per-launch event times, and the launch count."""
    v = np.asarray(ms_list, dtype=np.float64)
    return {"min": float(v.min()), "median": float(np.median(v)), "max": float(v.max()), "n": int(v.size)}


NOMINAL_FP8_TFLOPS = 4500.0  # dense FP8 tensor peak of a GB300 (nominal)
NOMINAL_HBM_GBS = 8000.0     # HBM3e, the round figure the targets are stated against
L2_BYTES = 129 << 20  # GB300 L2 (129 MB; about 126 MB usable)


def config_entries(dev, stream, n_launch=60, n_graph=20, replays=8):
    """The three single-kernel configurations (batch-32 decode, next_n=2 MTP
    decode over 128 requests, 8192-token causal prefill), the fused call's two
    kernels and the unfused pair.  Main figures: CUDA-graph replays of n_graph
    back-to-back launches with L2-cold operands (copies in rotation); also, under
    `single_launch`, one launch at a time after an L2 flush with events around
    each kernel.  Per configuration: per-kernel mean and min/median/max, the
    algorithmic rate (132 B per key, keys read once per request; 16384 flop per
    visible (query, key) pair) and its fraction of the measured and of the
    nominal peak; query tokens per second of logits + top-k."""
    import deepseek_v3_sparse_gb300 as dsix
    import workloads as W
    from workloads.device import make_step
    pk, pk_kind = peaks()
    fp8_meas = 2.0 * pk["bf16_tflops"]
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    out = {}
    for name, fn in (("decode_b32", W.decode_b32), ("decode_mtp2_b128", W.decode_mtp2_b128),
                     ("prefill_8k", W.prefill_8k)):
        wl = fn(seed=0)
        st = make_step(wl, dev, fused=True)
        st.run(stream=stream)
        # each call takes the copy of its streamed operand (the cache for decode,
        # the query rows and weights for prefill) and the stream to issue on
        if wl.n_decode:
            d = st.decode
            rows = wl.n_decode * wl.next_n
            ws = st.dec_ws
            operand = st.cache
            hist_c = lambda c, s_: dsix.ix_paged_mqa_logits_hist(d.q, d.w, c, d.context_lens, st.block_table,
                                                                 st.dec_logits, wl.topk, ws, stream=s_)
            sel_c = lambda s_: dsix.ix_topk_from_hist(st.dec_logits, d.row_len, d.row_req, st.block_table, wl.topk,
                                                      st.dec_global, ws, stream=s_)
            logits_c = lambda c, s_: dsix.ix_paged_mqa_logits(d.q, d.w, c, d.context_lens, st.block_table,
                                                              st.dec_logits, stream=s_)
            topk_c = lambda s_: dsix.ix_topk_to_global(st.dec_logits, d.row_len, d.row_req, st.block_table,
                                                       wl.topk, st.dec_global, None, stream=s_)
        else:
            p = st.prefill
            rows = wl.n_prefill_rows
            ws = st.pf_ws
            operand = (p.q, p.w)
            hist_c = lambda c, s_: dsix.ix_mqa_logits_hist(c[0], c[1], st.k_fp8, st.k_scale, p.ks, p.ke,
                                                           st.pf_logits, wl.topk, ws, stream=s_)
            sel_c = lambda s_: dsix.ix_topk_from_hist(st.pf_logits, p.row_len, p.row_req, st.block_table, wl.topk,
                                                      st.pf_global, ws, stream=s_)
            logits_c = lambda c, s_: dsix.ix_mqa_logits(c[0], c[1], st.k_fp8, st.k_scale, p.ks, p.ke, st.pf_logits,
                                                        stream=s_)
            topk_c = lambda s_: dsix.ix_topk_to_global(st.pf_logits, p.row_len, p.row_req, st.block_table,
                                                       wl.topk, st.pf_global, None, stream=s_)
        hist = lambda: hist_c(operand, stream)
        sel = lambda: sel_c(stream)
        logits = lambda: logits_c(operand, stream)
        topk = lambda: topk_c(stream)
        for _ in range(3):
            hist()
            sel()
            logits()
            topk()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_launch)]
        for e in evs:
            torch.sum(flush, 0, out=sink)
            e[0].record(stream)
            hist()
            e[1].record(stream)
            sel()
            e[2].record(stream)
            torch.sum(flush, 0, out=sink)
            e[3].record(stream)
            logits()
            e[4].record(stream)
            topk()
            e[5].record(stream)
        torch.cuda.synchronize()
        if dsix.ix_device_status() != 0:
            raise RuntimeError(f"device status set in the {name} timing")
        t = lambda i, j: [e[i].elapsed_time(e[j]) for e in evs]
        dec_keys, pairs = algorithmic(wl)

        def kern(ms_list):
            return {"ms": float(np.mean(ms_list)), **{f"ms_{k}": v for k, v in spread(ms_list).items()}}

        def rate(kd):
            ms = kd["ms"]
            if wl.n_decode:
                gbs = dec_keys * DECODE_BYTES_PER_KEY / (ms / 1e3) / 1e9
                gbs_med = dec_keys * DECODE_BYTES_PER_KEY / (kd["ms_median"] / 1e3) / 1e9
                kd.update(achieved=gbs, unit="GB/s", units=dec_keys,
                          per_unit=f"{DECODE_BYTES_PER_KEY} B per key, read once per request",
                          peak=pk["hbm_gbs"], peak_kind=f"{pk_kind} copy bandwidth",
                          frac=gbs / pk["hbm_gbs"], frac_at_median=gbs_med / pk["hbm_gbs"],
                          frac_of_8tbs=gbs / NOMINAL_HBM_GBS, target=0.70)
            else:
                tfs = pairs * PREFILL_FLOP_PER_PAIR / (ms / 1e3) / 1e12
                tfs_med = pairs * PREFILL_FLOP_PER_PAIR / (kd["ms_median"] / 1e3) / 1e12
                kd.update(achieved=tfs, unit="TFLOP/s", units=pairs,
                          per_unit=f"{PREFILL_FLOP_PER_PAIR} flop per visible (query, key) pair",
                          peak=fp8_meas, peak_kind=f"{pk_kind}: fp8 = 2 x cuBLAS bf16 burst {pk['bf16_tflops']}",
                          frac=tfs / fp8_meas, frac_at_median=tfs_med / fp8_meas,
                          frac_of_nominal_fp8=tfs / NOMINAL_FP8_TFLOPS, target=0.50)
            return kd

        # ---- graph timing: each call sequence as one CUDA graph of n_graph back-to-back
        # launches (the way the step is replayed), cycling through copies of the
        # streamed operand that total more than twice L2, so no launch finds it in
        # L2; per launch = replay time / n_graph, over `replays` replays (L2
        # flushed before each).  A top-k's time is its pair's minus its logits'.
        op_bytes = (operand.numel() * operand.element_size() if wl.n_decode
                    else sum(x.numel() * x.element_size() for x in operand))
        n_copies = max(2, int(np.ceil(2 * L2_BYTES / op_bytes)))
        copies = [operand] + [operand.clone() if wl.n_decode else tuple(x.clone() for x in operand)
                              for _ in range(n_copies - 1)]

        def graph_ms(body, clears_ws):
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    for j in range(n_graph):
                        body(copies[j % n_copies], side)
            stream.wait_stream(side)
            times = []
            for rep in range(replays + 1):
                torch.sum(flush, 0, out=sink)
                b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                b0.record(stream)
                g.replay()
                b1.record(stream)
                torch.cuda.synchronize()
                if not clears_ws:
                    ws.zero_()  # histogram kernels alone leave their counts behind
                if rep > 0:  # the first replay is a warm-up
                    times.append(b0.elapsed_time(b1) / n_graph)
            del g
            return times

        g_hist = graph_ms(lambda c, s_: hist_c(c, s_), False)
        g_fpair = graph_ms(lambda c, s_: (hist_c(c, s_), sel_c(s_)), True)
        g_plain = graph_ms(lambda c, s_: logits_c(c, s_), True)
        g_upair = graph_ms(lambda c, s_: (logits_c(c, s_), topk_c(s_)), True)
        if dsix.ix_device_status() != 0:
            raise RuntimeError(f"device status set in the {name} graph timing")
        del copies

        def pair_entry(ms_list):
            ms = float(np.mean(ms_list))
            return {"ms": ms, **{f"ms_{k}": v for k, v in spread(ms_list).items()},
                    "query_tokens_per_s": rows / (ms / 1e3),
                    "query_tokens_per_s_at_median": rows / (float(np.median(ms_list)) / 1e3)}

        fused_pair = [a + b for a, b in zip(t(0, 1), t(1, 2))]
        unfused_pair = [a + b for a, b in zip(t(3, 4), t(4, 5))]
        e = {"workload": wl.name, "rows": rows, "top_k": wl.topk,
             "timing": f"CUDA graph of {n_graph} back-to-back launches, {replays} replays, L2 flushed before "
                       f"each replay, {n_copies} copies of the streamed operand in rotation (more than twice L2)",
             "logits": rate(kern(g_hist)),
             "topk": kern([b - a for a, b in zip(g_hist, g_fpair)]),
             "logits_plus_topk": pair_entry(g_fpair),
             "unfused": {"logits": rate(kern(g_plain)),
                         "topk": kern([b - a for a, b in zip(g_plain, g_upair)]),
                         "logits_plus_topk": pair_entry(g_upair)},
             "single_launch": {
                 "timing": f"{n_launch} launches one at a time, L2 flushed (256 MB read) before each logits "
                           "launch, events around each kernel (launch and completion latency included)",
                 "logits": rate(kern(t(0, 1))), "topk": kern(t(1, 2)),
                 "logits_plus_topk": {"ms": float(np.mean(fused_pair)),
                                      "query_tokens_per_s": rows / (float(np.mean(fused_pair)) / 1e3)},
                 "unfused": {"logits": rate(kern(t(3, 4))), "topk": kern(t(4, 5)),
                             "logits_plus_topk": {"ms": float(np.mean(unfused_pair)),
                                                  "query_tokens_per_s": rows / (float(np.mean(unfused_pair)) / 1e3)}}},
             "note": "logits / topk: the two kernels of the fused call (histogram logits kernel, selection "
                     "from the histograms); unfused: the standalone logits kernel and top-k"}
        out[name] = e
        del st
        torch.cuda.empty_cache()
    return out


def kernel_event_pass(step, names, n_ev, stream, graph):
    """Per-kernel times of `n_ev` steps: events around each logits / top-k
    launch (a fused call issued as its two halves).  With `graph` the step and
    its events are one CUDA graph, replayed n_ev times as the timed steps are;
    otherwise the kernels are launched one by one.  Returns name -> list of ms."""
    if graph:
        try:
            ev = {n: (torch.cuda.Event(enable_timing=True, external=True),
                      torch.cuda.Event(enable_timing=True, external=True)) for n in names}
        except TypeError:  # no event nodes in graphs in this torch: launch one by one
            graph = False
    if graph:
        side = torch.cuda.Stream(device=stream.device)
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                step.run(stream=side, events=ev, split=True)
        stream.wait_stream(side)
        out = {n: [] for n in names}
        for _ in range(n_ev):
            g.replay()
            torch.cuda.synchronize()
            for n in names:
                out[n].append(ev[n][0].elapsed_time(ev[n][1]))
        del g
        return out, "events inside one CUDA graph of the step, replayed per sample"
    evl = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_ev)] for n in names}
    for i in range(n_ev):
        step.run(stream=stream, events={n: evl[n][i] for n in names}, split=True)
    torch.cuda.synchronize()
    return {n: [a.elapsed_time(b) for a, b in evl[n]] for n in names}, "events around eager launches"


def gpu_arm(args, world, rank, local):
    import deepseek_v3_sparse_gb300 as dsix
    from deepseek_v3_sparse_gb300 import build as libbuild
    import workloads as W
    from workloads.device import make_step

    libbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.NAMED[args.workload](seed=rank)
    fused = () if args.unfused else tuple(args.fused.split(","))
    step = make_step(wl, dev, fused=fused)
    stream = torch.cuda.current_stream(dev)
    names = []
    if wl.prefill_req:
        names += ["mqa_logits", "topk_prefill"]
    if wl.n_decode:
        names += ["paged_mqa_logits", "topk_decode"]
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if dsix.ix_device_status() != 0:
        raise RuntimeError("device status set during warm-up")
    # by default every timed step is one replay of the step's CUDA graph (the
    # same kernels as the eager launches, without a launch per kernel)
    run_step = (lambda st: st.run(stream=stream)) if args.eager else (lambda st: st.graph().replay())
    for _ in range(2):
        run_step(step)
    torch.cuda.synchronize()

    # the timed steps carry no per-kernel events (they would add gaps); the
    # per-kernel breakdown comes from a separate pass of the same steps after it
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(args.steps):
            run_step(step)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    elapsed_ms = t0.elapsed_time(t1)
    clk = clocks.summary()
    n_ev = min(args.steps, 200)
    samples, kern_mode = kernel_event_pass(step, names, n_ev, stream, graph=not args.eager)
    kern_ms = {n: float(np.mean(samples[n])) for n in names}
    kern_spread = {n: spread(samples[n]) for n in names}
    status = dsix.ix_device_status()

    # ---- the next row beyond the step: fused RMSNorm + RoPE + fp8_ds_mla write of
    # the step's new tokens at their own positions, timed launch by launch with
    # L2 flushed between launches (its inputs are far smaller than L2).  The flush
    # reads 256 MB: L2 is left full of clean lines, so the timed launch does not
    # also pay for writing back the flush's own data.
    next_rows = {}
    if wl.nope_bf16 is not None:
        pos = wl.new_positions()
        gamma, table = W.norm_rope_params(int(pos.max()) + 1)
        nr_in = dict(kv=wl.nope_bf16.to(dev), pe=wl.rope_bf16.to(dev), gamma=gamma.to(dev),
                     pos=torch.from_numpy(pos).to(dev), table=table.to(dev))
        nr_cache = torch.zeros(wl.num_blocks, 64, 656, dtype=torch.uint8, device=dev)
        nr_slots = step.new_slot
        flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)  # 256 MB > L2
        sink = torch.empty((), dtype=torch.float32, device=dev)
        nr = lambda: dsix.dsmla_norm_rope_write(nr_in["kv"], nr_in["pe"], nr_in["gamma"], 1e-6,
                                                nr_in["pos"], nr_in["table"], nr_slots, nr_cache,
                                                stream=stream)
        for _ in range(3):
            nr()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(50)]
        for a, b in evs:
            torch.sum(flush, 0, out=sink)
            a.record(stream)
            nr()
            b.record(stream)
        torch.cuda.synchronize()
        nr_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        next_rows["dsmla_norm_rope_write"] = dict(ms=nr_ms, units=int(len(pos)))
        del flush, nr_cache, nr_in
        if dsix.ix_device_status() != 0:
            raise RuntimeError("device status set by the fused norm/rope write")

    # ---- the query side of the step's query tokens (decode and prefill rows):
    # dsmla_fused_q with quantize_mqa (128 heads: RoPE, 576-wide fp8 MQA query)
    # and ix_quant_q (64 indexer heads: fp8 query, folded head weights), each
    # timed launch by launch with L2 flushed in between.
    if wl.nope_bf16 is not None:
        pos = torch.from_numpy(wl.new_positions()).to(dev)
        T = int(pos.numel())
        _, table = W.norm_rope_params(int(pos.max()) + 1)
        qi = W.query_inputs(T, seed=rank)
        qd = dict(qn=qi.ql_nope.to(dev), qp=qi.q_pe.to(dev), iq=qi.index_q.to(dev), iw=qi.index_w.to(dev),
                  table=table.to(dev), mqa=torch.empty(T, 128, 576, dtype=torch.uint8, device=dev),
                  sc=torch.empty(T, 128, dtype=torch.float32, device=dev),
                  qf=torch.empty(T, 64, 128, dtype=torch.uint8, device=dev),
                  wo=torch.empty(T, 64, dtype=torch.float32, device=dev))
        flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        sink = torch.empty((), dtype=torch.float32, device=dev)
        calls = {
            "dsmla_fused_q": lambda: dsix.dsmla_fused_q(qd["qp"], pos, qd["table"], True, ql_nope_bf16=qd["qn"],
                                                        out_mqa=qd["mqa"], out_scale=qd["sc"], stream=stream),
            "ix_quant_q": lambda: dsix.ix_quant_q(qd["iq"], qd["iw"], qd["qf"], qd["wo"], stream=stream)}
        for name, fn in calls.items():
            for _ in range(3):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
            for a, b in evs:
                torch.sum(flush, 0, out=sink)
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            ms_list = [a.elapsed_time(b) for a, b in evs]
            next_rows[name] = dict(ms=float(np.mean(ms_list)), spread=spread(ms_list), units=T)
        del flush, qd
        if dsix.ix_device_status() != 0:
            raise RuntimeError("device status set by the query side")

    # ---- the consumer of the decode indices: sparse MLA decode attention of the
    # decode tokens (128 heads) over top-k entries of the fp8_ds_mla cache, each
    # token's indices drawn from its own 131072-position context; entries written
    # by dsmla_quant_write.  Timed like the row above (L2 flushed per launch).
    if wl.n_decode > 0:
        T = wl.n_decode * wl.next_n
        ctx = int(wl.context_lens.max())
        x = W.sparse_decode_inputs(T, wl.topk, ctx, seed=17)
        mla_cache = torch.zeros(x.num_blocks, 64, 656, dtype=torch.uint8, device=dev)
        dsix.dsmla_quant_write(x.nope_bf16.to(dev), x.rope_bf16.to(dev), torch.from_numpy(x.slots).to(dev),
                               mla_cache, stream=stream)
        sd = dict(qn=x.q_nope.to(dev), qp=x.q_pe.to(dev), idx=torch.from_numpy(x.indices).to(dev),
                  out=torch.empty(T, 128, 512, dtype=torch.bfloat16, device=dev),
                  lse=torch.empty(T, 128, dtype=torch.float32, device=dev),
                  ws=torch.empty(dsix.dsmla_sparse_decode_workspace_size(T, 128, wl.topk), dtype=torch.uint8,
                                 device=dev))
        flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        sink = torch.empty((), dtype=torch.float32, device=dev)
        sdc = lambda: dsix.dsmla_sparse_decode(sd["qn"], sd["qp"], mla_cache, sd["idx"], x.sm_scale, sd["out"],
                                               sd["lse"], sd["ws"], stream=stream)
        for _ in range(3):
            sdc()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
        for a, b in evs:
            torch.sum(flush, 0, out=sink)
            a.record(stream)
            sdc()
            b.record(stream)
        torch.cuda.synchronize()
        next_rows["dsmla_sparse_decode"] = dict(ms=float(np.mean([a.elapsed_time(b) for a, b in evs])), units=T,
                                                topk=wl.topk, valid=int((x.indices >= 0).sum()))
        del flush, mla_cache, sd
        if dsix.ix_device_status() != 0:
            raise RuntimeError("device status set by the sparse MLA decode")

    # ---- end to end through the public API: pinned host inputs in, indices out.
    # Two step instances alternate, so the host-to-device copy of step i+1's
    # inputs and the device-to-host copy of step i-1's indices (each on a copy
    # stream of its own) overlap step i's kernels, as a serving loop would run
    # them; every step's copies lie inside the timed region, and events order
    # each buffer's reuse (a set's inputs are rewritten only after the step that
    # read them ran, its indices only after they were copied out).
    e2e_steps = min(args.steps, 200)
    steps = [step, make_step(wl, dev, fused=fused)]
    host_src = {
        "new_k": wl.new_k.pin_memory(),
        "new_slot": torch.from_numpy(wl.new_slot.copy()).pin_memory(),
        "bt": torch.from_numpy(wl.block_table.copy()).pin_memory(),
    }
    if wl.n_decode:
        host_src["q_dec"] = wl.q_decode.pin_memory()
        host_src["w_dec"] = wl.w_decode.pin_memory()
        host_src["ctx"] = torch.from_numpy(wl.context_lens.copy()).pin_memory()
    if wl.prefill_req:
        host_src["q_pf"] = wl.q_prefill.pin_memory()
        host_src["w_pf"] = wl.w_prefill.pin_memory()
    if wl.nope_bf16 is not None:
        host_src["nope"] = wl.nope_bf16.pin_memory()
        host_src["rope"] = wl.rope_bf16.pin_memory()

    def device_inputs(st):
        d = {"new_k": st.new_k, "new_slot": st.new_slot, "bt": st.block_table}
        if wl.n_decode:
            d.update(q_dec=st.decode.q, w_dec=st.decode.w, ctx=st.decode.context_lens)
        if wl.prefill_req:
            d.update(q_pf=st.prefill.q, w_pf=st.prefill.w)
        if wl.nope_bf16 is not None:
            d.update(nope=st.nope, rope=st.rope)
        return d

    def device_outputs(st):
        return ([st.dec_global] if wl.n_decode else []) + ([st.pf_global] if wl.prefill_req else [])

    host_in = [[(host_src[n], d) for n, d in device_inputs(st).items()] for st in steps]
    host_out = [[(d, torch.empty(d.shape, dtype=d.dtype).pin_memory()) for d in device_outputs(st)]
                for st in steps]
    h2d = sum(h.numel() * h.element_size() for h, _ in host_in[0])
    d2h = sum(h.numel() * h.element_size() for _, h in host_out[0])
    for st in steps:  # both instances warm (and captured)
        st.run(stream=stream)
        run_step(st)
    cp_in, cp_out = torch.cuda.Stream(), torch.cuda.Stream()
    mk = lambda: [torch.cuda.Event(), torch.cuda.Event()]
    in_done, run_done, out_done = mk(), mk(), mk()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    cp_in.wait_event(e0)
    cp_out.wait_event(e0)
    for i in range(e2e_steps):
        b = i & 1
        if i >= 2:
            cp_in.wait_event(run_done[b])
        with torch.cuda.stream(cp_in):
            for h, d in host_in[b]:
                d.copy_(h, non_blocking=True)
        in_done[b].record(cp_in)
        stream.wait_event(in_done[b])
        if i >= 2:
            stream.wait_event(out_done[b])
        run_step(steps[b])
        run_done[b].record(stream)
        cp_out.wait_event(run_done[b])
        with torch.cuda.stream(cp_out):
            for d, h in host_out[b]:
                h.copy_(d, non_blocking=True)
        out_done[b].record(cp_out)
    stream.wait_stream(cp_in)
    stream.wait_stream(cp_out)
    e1.record(stream)
    torch.cuda.synchronize()
    wall_e2e = time.perf_counter() - w0
    barrier(world)
    e2e_ms = max(e0.elapsed_time(e1), wall_e2e * 1e3)
    print(f"e2e: {e2e_steps} steps, device {e0.elapsed_time(e1):.2f} ms, host wall {wall_e2e * 1e3:.2f} ms",
          file=sys.stderr)
    del steps[1]

    dec_keys, pairs = algorithmic(wl)
    rows = int(wl.n_decode * wl.next_n + wl.n_prefill_rows)
    configs = {} if args.no_configs else config_entries(dev, stream)
    return dict(wl=wl, step=step, elapsed_ms=elapsed_ms, kern_ms=kern_ms, kern_spread=kern_spread,
                kern_mode=kern_mode,
                configs=configs, clocks=clk,
                status=status, e2e_ms=e2e_ms, e2e_steps=e2e_steps, h2d=h2d, d2h=d2h,
                dec_keys=dec_keys, pairs=pairs, rows=rows, next_rows=next_rows)


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg / reference arm)
# ---------------------------------------------------------------------------
class OracleSampler:
    """The oracle on whole-row samples of the workload, every figure measured
    (nothing is extrapolated).  One sample step runs the oracle, as it stands,
    on one decode row with all its keys and on the prefill rows that go with it
    in the step's own decode:prefill proportion (8192 / 16 = 512 rows for the
    mixed workload), and on the matching share of the fixed work: the cache
    writes (indexer K and fp8_ds_mla) of exactly those rows' new tokens, and a
    gather of the same share of the prefill contexts.  value = rows processed /
    time taken.  Set-up (the cache of already-cached positions, the gathered K
    the prefill rows read) is done once and not timed."""

    def __init__(self, wl):
        import oracle
        import workloads as W
        self.W, self.o, self.wl = W, oracle, wl
        oracle.build()
        self.cache = np.zeros((wl.num_blocks, 64 * 132), np.uint8)
        hist = ~wl.is_new
        oracle.quant_write_k(W.bf16_bits(wl.k_bf16[torch.from_numpy(hist)]), wl.slot[hist],
                             self.cache, 64)
        oracle.quant_write_k(W.bf16_bits(wl.new_k), wl.new_slot, self.cache, 64)
        cu = wl.prefill_gather()
        self.cu = cu
        self.kf = np.zeros((int(cu[-1]), 128), np.uint8)
        self.ksc = np.zeros(int(cu[-1]), np.float32)
        oracle.gather_k(self.cache, 64, 128, wl.prefill_block_table(), cu, self.kf, self.ksc)
        self.ks, self.ke, self.rl, self.rq = wl.prefill_rows()
        self.n_dec = wl.n_decode * wl.next_n
        self.dec_len, self.dec_req = wl.decode_rows()
        self.pf_per_dec = max(1, wl.n_prefill_rows // max(1, self.n_dec))
        # new tokens: flat index (request-major over cached positions) -> rank among new tokens
        self.new_rank = np.cumsum(wl.is_new) - 1
        self.req_off = np.concatenate([[0], np.cumsum(wl.req_ctx)]).astype(np.int64)
        # the fp8_ds_mla pool is written to before the clock starts, so the timed
        # writes do not also pay for the first touch of its pages
        self.dcache = np.ones((wl.num_blocks, 64, 656), np.uint8)
        self.gather_share = int(cu[-1]) * self.pf_per_dec // max(1, wl.n_prefill_rows)
        self.kf_share = np.zeros((max(1, self.gather_share), 128), np.uint8)
        self.ksc_share = np.zeros(max(1, self.gather_share), np.float32)
        self.rows = self.steps = 0
        self.t = 0.0
        self.n = 0

    def reset(self):
        self.rows = self.steps = 0
        self.t = 0.0

    def _new_of(self, req, pos):
        """Rank among the new tokens of request req's cached position pos."""
        return int(self.new_rank[self.req_off[req] + pos])

    def sample(self):
        wl, o, W = self.wl, self.o, self.W
        d = self.n % max(1, self.n_dec)
        T = len(self.ks)
        pf = np.array(sorted({int((self.n * self.pf_per_dec + j) * 0.6180339887 * T) % T
                              for j in range(self.pf_per_dec)}), dtype=np.int64) if T else np.zeros(0, np.int64)
        self.n += 1
        # the new tokens of these rows: the decode row's own token, and each prefill
        # row's token (row i of a chunk is position ctx - chunk_len + i of its request)
        toks = []
        if self.n_dec:
            b, j = d // wl.next_n, d % wl.next_n
            toks.append(self._new_of(b, int(wl.req_ctx[b]) - wl.next_n + j))
        for t in pf:
            r = int(self.rq[t])
            toks.append(self._new_of(r, int(self.rl[t]) - 1))
        toks = np.array(toks, dtype=np.int64)
        new_k = wl.new_k[torch.from_numpy(toks)]
        slots = wl.new_slot[toks]
        t0 = time.perf_counter()
        o.quant_write_k(W.bf16_bits(new_k), slots, self.cache, 64)
        if wl.nope_bf16 is not None:
            sel = torch.from_numpy(toks)
            o.dsmla_quant_write(W.bf16_bits(wl.nope_bf16[sel]), W.bf16_bits(wl.rope_bf16[sel]), slots,
                                self.dcache, 64)
        if len(pf) and self.gather_share > 0:
            c = int(np.searchsorted(self.cu, int(self.ks[pf[0]]), side="right") - 1)
            o.gather_k(self.cache, 64, 128, wl.prefill_block_table()[c:c + 1],
                       np.array([0, self.gather_share], np.int32), self.kf_share, self.ksc_share)
        if self.n_dec:
            L = int(self.dec_len[d])
            lg = o.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), self.cache, 64,
                                    wl.context_lens, wl.block_table, ld=max(4, (L + 3) // 4 * 4),
                                    clean=False, rows=[d])
            o.topk_to_global(lg, self.dec_len[d:d + 1], self.dec_req[d:d + 1], wl.block_table, 64, wl.topk)
        if len(pf):
            plg = o.mqa_logits(W.u8(wl.q_prefill), wl.w_prefill.numpy(), self.kf, self.ksc, self.ks,
                               self.ke, ld=int(self.rl[pf].max() + 3) // 4 * 4, clean=False, rows=pf)
            o.topk_to_global(plg, self.rl[pf], self.rq[pf], wl.block_table, 64, wl.topk)
        self.t += time.perf_counter() - t0
        self.rows += (1 if self.n_dec else 0) + len(pf)
        self.steps += 1

    def value(self) -> float:
        return self.rows / self.t

    def describe(self) -> str:
        return (f"oracle on the host cores, measured on {self.steps} sample steps of whole rows "
                f"({self.rows} rows in {self.t:.2f} s): each step 1 decode row with all its keys + "
                f"{self.pf_per_dec} prefill rows (the step's decode:prefill mix), the cache writes of "
                f"those rows' new tokens and a gather of {self.gather_share} cached tokens (the same "
                f"share of the step's prefill contexts); value = rows / time")


def next_row_cpu_baselines(wl, rows):
    """The oracle timed on the inputs of the rows timed beside the step (the
    same draws as the GPU lines): the fused norm/RoPE write of all the step's
    new tokens, and the sparse MLA decode of the whole decode batch.  Each
    is small enough to time whole.  Returns name -> cpu_baseline entry."""
    import oracle
    import workloads as W
    oracle.build()
    out = {}
    if "dsmla_norm_rope_write" in rows and wl.nope_bf16 is not None:
        pos = wl.new_positions()
        gamma, table = W.norm_rope_params(int(pos.max()) + 1)
        n = len(pos)
        dense = np.ones((-(-n // 64), 64, 656), np.uint8)  # a compact pool, pages touched up front
        t = time.perf_counter()
        oracle.dsmla_norm_rope_write(W.bf16_bits(wl.nope_bf16), W.bf16_bits(wl.rope_bf16),
                                     W.bf16_bits(gamma), 1e-6, pos, table.numpy(),
                                     np.arange(n, dtype=np.int64), dense, 64)
        dt = time.perf_counter() - t
        out["dsmla_norm_rope_write"] = {
            "value": n / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"all {n} new tokens into a compact pool, timed whole ({dt:.3f} s)"}
    if ("dsmla_fused_q" in rows or "ix_quant_q" in rows) and wl.nope_bf16 is not None:
        pos = wl.new_positions()
        _, table = W.norm_rope_params(int(pos.max()) + 1)
        n = 512  # a bounded sample of the step's query tokens
        qi = W.query_inputs(n, seed=0)
        t = time.perf_counter()
        oracle.fused_q(W.bf16_bits(qi.ql_nope), W.bf16_bits(qi.q_pe), pos[:n], table.numpy(), True)
        dt = time.perf_counter() - t
        out["dsmla_fused_q"] = {
            "value": n / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of the step's {len(pos)} query tokens x 128 heads, quantize_mqa, timed whole ({dt:.3f} s)"}
        t = time.perf_counter()
        oracle.quant_q(W.bf16_bits(qi.index_q), qi.index_w.numpy())
        dt = time.perf_counter() - t
        out["ix_quant_q"] = {
            "value": n / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of the step's {len(pos)} query tokens x 64 heads, timed whole ({dt:.3f} s)"}
    if "dsmla_sparse_decode" in rows and wl.n_decode > 0:
        T = wl.n_decode * wl.next_n
        x = W.sparse_decode_inputs(T, wl.topk, int(wl.context_lens.max()), seed=17)
        dense = np.zeros((x.num_blocks, 64, 656), np.uint8)
        oracle.dsmla_quant_write(W.bf16_bits(x.nope_bf16), W.bf16_bits(x.rope_bf16), x.slots, dense, 64)
        t = time.perf_counter()
        oracle.dsmla_sparse_decode(W.bf16_bits(x.q_nope), W.bf16_bits(x.q_pe), dense, 64, x.indices,
                                   x.sm_scale)
        dt = time.perf_counter() - t
        out["dsmla_sparse_decode"] = {
            "value": T / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the whole batch of {T} tokens x 128 heads x top-{wl.topk}, timed whole ({dt:.3f} s)"}
    return out


def reference_arm(args, world, rank):
    import oracle
    import workloads as W
    if rank != 0:
        return
    wl = W.mixed_long(seed=0)
    s = OracleSampler(wl)
    for _ in range(args.warmup):
        s.sample()
    s.reset()
    # each sample step takes about a second on the host cores: the timed steps
    # stop early (and the line says how many ran) once two minutes have passed
    w0 = time.perf_counter()
    for _ in range(args.steps):
        s.sample()
        if time.perf_counter() - w0 > 120.0:
            break
    wall = time.perf_counter() - w0
    value = s.value()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": s.steps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": s.t / s.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (exact fp8 products, double head sum)",
            "data": "synthetic (seeded; no dataset, no weights)",
            "config": {**workload_config(wl), "parallelism": "replicas x1 (rank 0 only)",
                       "step": "one sample step: 1 decode row + its share of prefill rows, whole rows"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": s.describe()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="dsix", choices=["dsix", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="run every logits call and its top-k as separate calls")
    ap.add_argument("--fused", default="decode",
                    help="parts whose logits and top-k run as one fused call: decode, prefill or decode,prefill "
                         "(default decode: for the prefill rows the histogram costs the logits kernel more than "
                         "it saves the selection)")
    ap.add_argument("--eager", action="store_true",
                    help="launch each step's kernels one by one instead of replaying the step's CUDA graph")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration timing of the decode, MTP and prefill kernels")
    ap.add_argument("--workload", default="mixed_long",
                    help="named workload; the benchmark line is mixed_long, the others are "
                         "for profiling single kernels")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_init()
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return
    r = gpu_arm(args, world, rank, local)
    elapsed = max_over_ranks(r["elapsed_ms"], world)
    e2e_ms = max_over_ranks(r["e2e_ms"], world)
    if rank != 0:
        return
    wl, step = r["wl"], r["step"]
    pk, pk_kind = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"]
    value = job_throughput(world, r["rows"], args.steps, elapsed)
    km = r["kern_ms"]
    pf_tflops = (r["pairs"] * PREFILL_FLOP_PER_PAIR / (km["mqa_logits"] / 1e3) / 1e12
                 if "mqa_logits" in km else None)
    dec_gbs = (r["dec_keys"] * DECODE_BYTES_PER_KEY / (km["paged_mqa_logits"] / 1e3) / 1e9
               if "paged_mqa_logits" in km else None)
    kernels = {}
    if "mqa_logits" in km:
        kernels["mqa_logits"] = {
            "ms": km["mqa_logits"], "achieved": pf_tflops, "unit": "TFLOP/s", "peak": fp8_peak,
            "frac": pf_tflops / fp8_peak, "units": r["pairs"],
            "per_unit": f"{PREFILL_FLOP_PER_PAIR} flop per visible (query, key) pair"}
    if "paged_mqa_logits" in km:
        kernels["paged_mqa_logits"] = {
            "ms": km["paged_mqa_logits"], "achieved": dec_gbs, "unit": "GB/s",
            "peak": pk["hbm_gbs"], "frac": dec_gbs / pk["hbm_gbs"], "frac_of_8tbs": dec_gbs / 8000.0,
            "per_unit": f"{DECODE_BYTES_PER_KEY} B per key", "units": r["dec_keys"]}
    for n in ("topk_decode", "topk_prefill"):
        if n in km:
            kernels[n] = {"ms": km[n]}
    for n, kd in kernels.items():
        sp = r["kern_spread"][n]
        kd.update({f"ms_{k}": v for k, v in sp.items()})
        if "frac" in kd:  # the fraction at the median launch time too
            kd["frac_at_median"] = kd["frac"] * kd["ms"] / sp["median"]
    if "mqa_logits" in kernels:
        kernels["mqa_logits"]["frac_of_nominal_fp8"] = pf_tflops / NOMINAL_FP8_TFLOPS
    traffic = measured_traffic(workload_config(wl)["workload"])
    for n, kd in kernels.items():
        kd["traffic"] = traffic.get(n)
    dominant = max((n for n in ("mqa_logits", "paged_mqa_logits") if n in km), key=lambda n: km[n])
    kd = kernels[dominant]
    roofline = {"bound": "tensor" if dominant == "mqa_logits" else "hbm",
                "kernel": dominant, "achieved": kd["achieved"], "peak": kd["peak"],
                "unit": kd["unit"], "frac": kd["frac"], "traffic": kd["traffic"],
                "traffic_unit": "bytes per launch (ncu dram read + write; null once the kernel changed)",
                "peak_kind": (f"{pk_kind}: fp8 = 2 x cuBLAS bf16 burst {pk['bf16_tflops']} TFLOP/s"
                              if dominant == "mqa_logits" else f"{pk_kind} copy bandwidth"),
                "frac_of_nominal": (kd["achieved"] / NOMINAL_FP8_TFLOPS if dominant == "mqa_logits"
                                    else kd["achieved"] / NOMINAL_HBM_GBS),
                "nominal_peak": NOMINAL_FP8_TFLOPS if dominant == "mqa_logits" else NOMINAL_HBM_GBS}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8_e4m3 x fp8_e4m3 -> f32 (logits); u8/bf16 cache writes",
            "data": "synthetic (seeded; random-init inputs of the indexer shapes; no dataset)",
            "config": {**workload_config(wl), "parallelism": f"replicas x{world}",
                       "fused_logits_topk": [] if args.unfused else args.fused.split(","),
                       "step_issue": "eager launches" if args.eager else
                       "one CUDA graph replay per step (the step's kernels, captured once)"},
            "roofline": roofline, "kernels": kernels,
            "prefill_tflops": pf_tflops, "decode_hbm_gbs": dec_gbs,
            "e2e": {"value": job_throughput(world, r["rows"], r["e2e_steps"], e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": step.kernels_per_step() * args.steps,
            "kernel_timing": r["kern_mode"],
            "clocks": r["clocks"], "device_status": r["status"]}
    if r["configs"]:
        line["configs"] = r["configs"]
    for n, d in r["next_rows"].items():  # rows beyond the step, timed on their own
        if n == "dsmla_sparse_decode":
            line.setdefault("next_rows", {})[n] = sparse_decode_line(d, pk)
            continue
        if n in QUERY_BYTES_PER_TOKEN:
            per, what = QUERY_BYTES_PER_TOKEN[n]
            gbs = d["units"] * per / (d["ms"] / 1e3) / 1e9
            line.setdefault("next_rows", {})[n] = {
                "ms": d["ms"], **{f"ms_{k}": v for k, v in d["spread"].items()}, "achieved": gbs, "unit": "GB/s",
                "peak": pk["hbm_gbs"], "frac": gbs / pk["hbm_gbs"], "units": d["units"],
                "per_unit": f"{per} B per query token ({what})", "bound": "hbm",
                "l2": "flushed between launches (256 MB read)"}
            continue
        gbs = d["units"] * NORM_ROPE_BYTES_PER_TOKEN / (d["ms"] / 1e3) / 1e9
        line.setdefault("next_rows", {})[n] = {
            "ms": d["ms"], "achieved": gbs, "unit": "GB/s", "peak": pk["hbm_gbs"],
            "frac": gbs / pk["hbm_gbs"], "units": d["units"],
            "per_unit": f"{NORM_ROPE_BYTES_PER_TOKEN} B per token (1024 NoPE + 128 RoPE in, "
                        "8 position + 8 slot + 256 table row read, 656 entry out)",
            "l2": "flushed between launches (256 MB read)"}
    if not args.no_cpu_baseline:
        import oracle
        s = OracleSampler(wl)
        s.sample()  # warm-up (page faults, thread pool)
        s.reset()
        while s.t < 10.0 or s.steps < 3:
            s.sample()
        line["cpu_baseline"] = {"value": s.value(), "unit": UNIT,
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": s.describe(), "sample_seconds": s.t}
        for n, cb in next_row_cpu_baselines(wl, set(line.get("next_rows", {}))).items():
            line["next_rows"][n]["cpu_baseline"] = cb
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
