"""Host logic of bench.py at N > 1, on CPU: two gloo ranks.

The benchmark runs independent replicas (the ring collective on one GPU has no
exchange between GPUs); the job time is the slowest replica's, and the value
is the sum of every replica's work over that time.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [10.0 + 5 * rank, 1.0 + rank]  # the second rank is slower
    got = bench.combine_ranks(dist, local)
    value = bench.job_throughput(world, 1 << 20, got[0])
    # only rank 0 of the reference arm does work and prints
    buf = io.StringIO()
    with redirect_stdout(buf):
        if rank != 0:
            bench.run_reference(type("A", (), dict(warmup=3, steps=1, msg_mib=512, ref_sample_mib=1))())
    q.put((rank, got, value, buf.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value, out in results:
        assert got == [15.0, 2.0]  # max over ranks, element-wise
        assert value == pytest.approx(2 * (1 << 20) / 15e-3 / 1e9)
        if rank != 0:
            assert out == ""


def test_single_process_combine_is_identity():
    assert bench.combine_ranks(None, [3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_throughput(1, 512 << 20, 1.0) == pytest.approx((512 << 20) / 1e-3 / 1e9)


def test_reference_arm_prints_one_json_line(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    args = type("A", (), dict(warmup=3, steps=2, msg_mib=512, ref_sample_mib=1))()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_clock_summary_flags_throttling():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(1.0, ["1900", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Active"]),
                 (1.2, ["1950", "2070", "950", "0x0", "Not Active", "Active", "Not Active", "Not Active"]),
                 (5.0, ["300", "2070", "100", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"])]
    c = s.summary(0.9, 1.3)
    assert c["samples"] == 2 and c["sm_mhz"] == 1925.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_kernel_digest_ignores_comments_only():
    import bench

    src = 'int f(int x) { // add one\n  return x + 1; /* done */ }\nconst char *s = "a//b /* c */";\n'
    same = 'int f(int x) {\n  return x + 1;\n}\nconst char *s = "a//b /* c */"; // note\n'
    other = 'int f(int x) { return x + 2; }\nconst char *s = "a//b /* c */";\n'
    assert bench.code_only(src) == bench.code_only(same)
    assert bench.code_only(src) != bench.code_only(other)
    assert '"a//b /* c */"' in bench.code_only(src)


def test_gpus_flag_launches_replicas_itself(tmp_path):
    """`bench.py --gpus 2` started without a launcher starts two ranks under
    torch.distributed.run by itself; rank 0 alone prints one JSON line, which
    reports both ranks.  (The reference arm runs here: it needs no GPU.)"""
    import subprocess

    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3", "--ref-sample-mib", "1"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=str(tmp_path))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_replica_launch_command():
    cmd = bench.replica_launch_command(4, ["--gpus", "4", "--steps", "5"], 29511)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--master-addr=127.0.0.1" in cmd and "--master-port=29511" in cmd
    assert cmd[-4:] == ["--gpus", "4", "--steps", "5"] and cmd[-5].endswith("bench.py")


def test_path_choice_table_marks_the_planner():
    """The sweep's table lists both paths per point and whether the planner's
    pick is within 5 % of the faster."""
    def row(variant, path, us, R=4):
        return {"op": "allreduce", "R": R, "count": 1 << 20, "msg_bytes": 2 << 20, "off_grid": False,
                "variant": variant, "path": path, "us": us}

    rows = [row("auto", "direct", 10.0), row("bulk", "bulk", 12.0), row("direct", "direct", 10.0),
            row("auto", "bulk", 20.0, R=2), row("bulk", "bulk", 20.0, R=2), row("direct", "direct", 15.0, R=2)]
    args = type("A", (), dict(sweep_ops="ar", sweep_ranks="2,4", sweep_mib="2", sweep_dtype="f16", sweep_layouts=1,
                              sweep_off_grid="no"))()
    text = bench.path_choice_table(rows, args)
    lines = [ln for ln in text.splitlines() if ln.startswith("| allreduce")]
    assert lines[0].split("|")[6:10] == [" 12.0 ", " 10.0 ", " direct ", " yes "]
    assert lines[1].split("|")[6:10] == [" 20.0 ", " 15.0 ", " bulk ", " NO "]
    assert "--sweep-table FILE" in text
