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


def gpu_arm(args, world, rank, local):
    import deepseek_v3_sparse_gb300 as dsix
    from deepseek_v3_sparse_gb300 import build as libbuild
    import workloads as W
    from workloads.device import make_step

    libbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.NAMED[args.workload](seed=rank)
    step = make_step(wl, dev)
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

    # the timed steps carry no per-kernel events (they would add gaps); the
    # per-kernel breakdown comes from a separate pass of the same steps after it
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(args.steps):
            step.run(stream=stream)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    elapsed_ms = t0.elapsed_time(t1)
    clk = clocks.summary()
    n_ev = min(args.steps, 200)
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_ev)] for n in names}
    for i in range(n_ev):
        step.run(stream=stream, events={n: ev[n][i] for n in names})
    torch.cuda.synchronize()
    kern_ms = {n: float(np.mean([a.elapsed_time(b) for a, b in ev[n]])) for n in names}
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
    steps = [step, make_step(wl, dev)]
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
    for st in steps:  # both instances warm
        st.run(stream=stream)
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
        steps[b].run(stream=stream)
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
    return dict(wl=wl, step=step, elapsed_ms=elapsed_ms, kern_ms=kern_ms, clocks=clk,
                status=status, e2e_ms=e2e_ms, e2e_steps=e2e_steps, h2d=h2d, d2h=d2h,
                dec_keys=dec_keys, pairs=pairs, rows=rows, next_rows=next_rows)


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg / reference arm)
# ---------------------------------------------------------------------------
class OracleSampler:
    """The oracle timed on bounded samples of the workload.  Set-up (the cache
    of already-cached positions) is done once; each sample times a slice of a
    decode row and whole prefill rows (logits + top-k), rotating over rows;
    per-key / per-pair costs extrapolate to one whole step."""

    def __init__(self, wl):
        import oracle
        import workloads as W
        self.W, self.o, self.wl = W, oracle, wl
        oracle.build()
        self.cache = np.zeros((wl.num_blocks, 64 * 132), np.uint8)
        hist = ~wl.is_new
        oracle.quant_write_k(W.bf16_bits(wl.k_bf16[torch.from_numpy(hist)]), wl.slot[hist],
                             self.cache, 64)
        # the fp8_ds_mla pool is written to before the clock starts, so the timed
        # write does not also pay for the first touch of its pages
        dcache = np.ones((wl.num_blocks, 64, 656), np.uint8)
        t = time.perf_counter()  # whole-step cache writes and gather, timed once
        oracle.quant_write_k(W.bf16_bits(wl.new_k), wl.new_slot, self.cache, 64)
        oracle.dsmla_quant_write(W.bf16_bits(wl.nope_bf16), W.bf16_bits(wl.rope_bf16),
                                 wl.new_slot, dcache, 64)
        cu = wl.prefill_gather()
        self.kf = np.zeros((int(cu[-1]), 128), np.uint8)
        self.ksc = np.zeros(int(cu[-1]), np.float32)
        oracle.gather_k(self.cache, 64, 128, wl.prefill_block_table(), cu, self.kf, self.ksc)
        self.t_fixed = time.perf_counter() - t
        del dcache
        self.ks, self.ke, self.rl, self.rq = wl.prefill_rows()
        self.full_keys = int(wl.context_lens.astype(np.int64).sum())
        self.full_pairs = int(self.rl.astype(np.int64).sum())
        self.keys = self.pairs = 0
        self.t_keys = self.t_pairs = 0.0
        self.n = 0

    def sample(self, dec_keys: int = 2048, pf_rows: int = 0):
        wl, o, W = self.wl, self.o, self.W
        pf_rows = pf_rows or o.num_threads()  # one row per thread: rows run in parallel
        ctx = wl.context_lens.copy()
        ctx[0] = dec_keys
        t = time.perf_counter()
        lg = o.paged_mqa_logits(W.u8(wl.q_decode), wl.w_decode.numpy(), self.cache, 64, ctx,
                                wl.block_table, ld=dec_keys, clean=False, rows=[0])
        o.topk_to_global(lg, np.array([dec_keys], np.int32), np.zeros(1, np.int32),
                         wl.block_table, 64, wl.topk)
        self.t_keys += time.perf_counter() - t
        self.keys += dec_keys
        T = len(self.ks)
        rows = np.array([(int((self.n + j) * 0.6180339887 * T)) % T for j in range(pf_rows)],
                        dtype=np.int64)
        self.n += pf_rows
        t = time.perf_counter()
        plg = o.mqa_logits(W.u8(wl.q_prefill), wl.w_prefill.numpy(), self.kf, self.ksc, self.ks,
                           self.ke, ld=int(self.rl[rows].max()), clean=False, rows=rows)
        o.topk_to_global(plg, self.rl[rows], self.rq[rows], wl.block_table, 64, wl.topk)
        self.t_pairs += time.perf_counter() - t
        self.pairs += int(self.rl[rows].astype(np.int64).sum())

    def step_seconds(self) -> float:
        return (self.t_fixed + self.t_keys / self.keys * self.full_keys
                + self.t_pairs / self.pairs * self.full_pairs)

    def describe(self) -> str:
        return (f"oracle on the host cores: new-token cache writes, fp8_ds_mla write and gather "
                f"timed whole; decode logits+top-k over {self.keys} keys and prefill logits+top-k "
                f"over {self.n} rows ({self.pairs} pairs) spread over the chunks, extrapolated "
                f"per key / per pair to one step ({self.full_keys} decode keys, "
                f"{self.full_pairs} prefill pairs)")


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
    rows = int(wl.n_decode * wl.next_n + wl.n_prefill_rows)
    s = OracleSampler(wl)
    for _ in range(args.warmup):
        s.sample()
    s.keys = s.pairs = 0
    s.t_keys = s.t_pairs = 0.0
    w0 = time.perf_counter()
    for _ in range(args.steps):
        s.sample()
    wall = time.perf_counter() - w0
    est = s.step_seconds()
    value = rows / est
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": est * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (exact fp8 products, double head sum)",
            "data": "synthetic (seeded; no dataset, no weights)",
            "config": workload_config(wl),
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
                              if dominant == "mqa_logits" else f"{pk_kind} copy bandwidth")}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8_e4m3 x fp8_e4m3 -> f32 (logits); u8/bf16 cache writes",
            "data": "synthetic (seeded; random-init inputs of the indexer shapes; no dataset)",
            "config": {**workload_config(wl), "parallelism": f"replicas x{world}"},
            "roofline": roofline, "kernels": kernels,
            "prefill_tflops": pf_tflops, "decode_hbm_gbs": dec_gbs,
            "e2e": {"value": job_throughput(world, r["rows"], r["e2e_steps"], e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": step.kernels_per_step() * args.steps,
            "clocks": r["clocks"], "device_status": r["status"]}
    for n, d in r["next_rows"].items():  # rows beyond the step, timed on their own
        if n == "dsmla_sparse_decode":
            line.setdefault("next_rows", {})[n] = sparse_decode_line(d, pk)
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
        w0 = time.perf_counter()
        while time.perf_counter() - w0 < 12.0 or s.n < 8:
            s.sample(dec_keys=8192)
        line["cpu_baseline"] = {"value": r["rows"] / s.step_seconds(), "unit": UNIT,
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": s.describe(),
                                "sample_seconds": time.perf_counter() - w0 + s.t_fixed}
        for n, cb in next_row_cpu_baselines(wl, set(line.get("next_rows", {}))).items():
            line["next_rows"][n]["cpu_baseline"] = cb
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
