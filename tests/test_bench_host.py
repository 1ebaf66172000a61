"""Host logic of bench.py, on CPU: replica timing over gloo ranks, whole-job
throughput, the reference arm's rank rule and the traffic lookup."""
import multiprocessing as mp
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench as b
    world, r, local = b.dist_init()
    b.barrier(world)
    elapsed = b.max_over_ranks(10.0 + 5.0 * rank, world)  # rank 1 is the slow one
    q.put((r, world, local, elapsed, b.job_throughput(world, 100, 4, elapsed)))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for rank, world, local, elapsed, value in out:
        assert world == 2 and local == rank
        assert elapsed == 15.0                      # max over ranks, on every rank
        assert value == pytest.approx(2 * 100 * 4 / 0.015)  # all ranks' rows / slowest time


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.job_throughput(1, 8208, 10, 9.7) == pytest.approx(8208 * 10 / 0.0097)


def test_reference_arm_prints_nothing_off_rank_zero(capsys):
    class A:
        steps = warmup = gpus = 2
    assert bench.reference_arm(A(), 2, 1) is None
    assert capsys.readouterr().out == ""


def _profile(tmp_path, lines):
    p = tmp_path / "traffic.txt"
    p.write_text("\n".join(lines) + "\n")
    return str(p)


def test_traffic_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    import hashlib
    def h(rel):
        with open(os.path.join(bench.ROOT, rel), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()
    logits, common, topk = (f"deepseek_v3_sparse_gb300/csrc/{n}" for n in ("logits.cu", "common.cuh", "topk.cu"))
    prof = _profile(tmp_path, [
        "# comment", "workload wl_a",
        f"source {logits} {h(logits)}", f"source {common} {h(common)}", f"source {topk} {'0' * 64}",
        "kernel mqa_logits read 100 write 20 ncu_ns 1",
        "kernel topk_prefill read 7 write 3 ncu_ns 1"])
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", prof)
    t = bench.measured_traffic("wl_a")
    assert t == {"mqa_logits": 120}          # the top-k source no longer matches: no figure
    assert bench.measured_traffic("wl_b") == {}  # another workload: no figure
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(tmp_path / "missing.txt"))
    assert bench.measured_traffic("wl_a") == {}


def test_committed_traffic_profile_parses():
    t = bench.measured_traffic("mixed_16x131072dec_4x2048pf")
    assert set(t) <= set(bench.KERNEL_SOURCES)
    assert all(isinstance(v, int) and v > 0 for v in t.values())


def test_next_row_cpu_baselines_small_workload():
    # the oracle legs beside the next rows run on the host alone
    import workloads as W
    wl = W.build("mix", decode_ctx=[500, 700], next_n=1, prefill=[(900, 300)], topk=128, seed=2,
                 dsmla=True)
    out = bench.next_row_cpu_baselines(wl, {"dsmla_norm_rope_write", "dsmla_sparse_decode"})
    assert set(out) == {"dsmla_norm_rope_write", "dsmla_sparse_decode"}
    for v in out.values():
        assert v["value"] > 0 and v["unit"] == "tokens/s" and v["kind"] == "oracle" and v["cores"] >= 1
    assert "2 tokens" in out["dsmla_sparse_decode"]["sample"]
    assert bench.next_row_cpu_baselines(wl, set()) == {}


def test_oracle_sampler_counts_whole_rows_it_measured():
    """The CPU baseline is measured, not extrapolated: a sample step runs whole
    rows (one decode row, its share of prefill rows) and the value is the rows
    it ran over the time it took."""
    import workloads as W
    wl = W.build("small_mixed", decode_ctx=[300, 200], next_n=1, prefill=[(256, 64), (128, 64)],
                 topk=64, seed=3, dsmla=True)
    s = bench.OracleSampler(wl)
    assert s.pf_per_dec == 64  # 128 prefill rows for 2 decode rows
    s.sample()
    s.reset()
    for _ in range(3):
        s.sample()
    assert s.steps == 3
    assert 3 <= s.rows <= 3 * 65
    assert s.value() == pytest.approx(s.rows / s.t)
    assert "3 sample steps" in s.describe()
