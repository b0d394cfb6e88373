"""Benchmark of libringred's ring AllReduce on one GB300 (or N independent replicas).

Workload (the ring AllReduce sweep): R = 8 virtual ranks, binary16 storage and
wire (a rounding after every hop), values normal with sigma 1e-3, per-rank
message of 512 MiB (268,435,456 elements).  One step = one ring_allreduce call
through the C ABI over all 8 rank buffers (partition, reduce-scatter fold and
allgather copies fused in one kernel).  The step's inputs (4 GiB) and outputs
(4 GiB) are far larger than L2, so no flush is needed between timed steps.

Printed value: algbw = per-rank message bytes / step time (GB/s, 1e9), the
whole job's aggregate over replicas at N > 1 (weak scaling: every GPU runs its
own full workload; the path has no exchange between GPUs).

Also reported: the roofline of the kernel (2 R msg bytes per launch over its
CUDA-event time against the measured HBM copy bandwidth), the sweep over 1,
16, 128 and 512 MiB and a table of the other workloads (AllReduce /
ReduceScatter / AllGather at R = 4, the bfloat16 wire, the two-level ring, a
fusion bucket), each timed by CUDA-graph replay over rotating buffer sets of
at least 3x the L2 size so no launch finds its inputs in L2, an end-to-end
figure through the C ABI's host-buffer entry point (ring_allreduce_host_ex:
page-locked inputs copied in and all R outputs copied back inside the timed
region, pipelined in pieces, with the copy schedule the link measured just
before favours), the CPU oracle's throughput on a bounded sample, and the SM
clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --path-sweep [--sweep-ops ar,rs,ag] [--sweep-ranks ...] [--sweep-mib ...]
                  [--sweep-off-grid no|only|both] [--sweep-variants]
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "allreduce algbw GB/s and % of HBM roofline vs message size at R ranks, 1 GB300"
UNIT = "GB/s"
MIB = 1 << 20
R = 8
MSG_MIB = 512
SWEEP_MIB = (1, 16, 128, 512)
CPU_SAMPLE_MIB = 64
REF_SAMPLE_MIB = 64
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


DEVICE_SOURCES = ("rr_kernels.cuh", "rr_device.cuh", "rr_params.h", "rr_inst_one.cu", "rr_dispatch.cu",
                  "rr_hd_direct.cuh", "rr_inst_hd_f32.cu", "rr_inst_hd_f16.cu", "rr_inst_hd_bf16.cu")


def code_only(text):
    """C / C++ source without its comments and with runs of whitespace folded,
    so that a comment edit does not count as a change of the code."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':  # string literals (the inline PTX) are code
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_sources_digest():
    """Digest of the device code (the kernels, not the host-side planner;
    comments and layout do not count)."""
    h = hashlib.sha256()
    for name in DEVICE_SOURCES:
        with open(os.path.join(ROOT, "ring_allreduce_reducescatter_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(digest):
    """DRAM bytes per launch of the AllReduce kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        with open(p) as f:
            text = f.read()
        m = re.search(r"traffic_per_launch_bytes:\s*(\d+)\s*\(kernel sources ([0-9a-f]+)\)", text)
        if m and m.group(2) == digest:
            return int(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples (every PERIOD_MS) with host
    timestamps; short timed regions (tens of milliseconds) still get samples."""

    PERIOD_MS = 25

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_id), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        source = "timed region"
        if not inside:  # region shorter than the sampling period: nearest samples
            inside = [p for (t, p) in self.samples if t0 - 1.0 <= t <= t1 + 1.0]
            source = "within 1 s of the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "none"}
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for p in inside for k in range(4) if p[4 + k].lower().startswith("active")})
        pw = [num(p[2]) for p in inside if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "source": source,
                "power_w_max": max(pw) if pw else None}


def combine_ranks(pg, local_ms, device=None):
    """Max over ranks of each timing (ms), the slowest replica sets the job time."""
    if pg is None:
        return list(local_ms)
    import torch

    t = torch.tensor(list(local_ms), dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world, msg_bytes, ms_per_step):
    """Whole-job algbw (GB/s): every replica moves msg_bytes per rank per step."""
    return world * msg_bytes / (ms_per_step * 1e-3) / 1e9


def parse_cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def bind_to_gpu_local_cpus(props, gpu_id):
    """Run this process on the CPUs attached to the GPU's PCI root, so that
    page-locked host buffers land in the memory next to the GPU's host link.
    Returns a short description, or None when the topology is not readable."""
    addr = None
    if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
        addr = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    else:
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(gpu_id), "--query-gpu=pci.bus_id",
                                  "--format=csv,noheader"], capture_output=True, text=True, timeout=30).stdout
            bus = out.strip().lower()
            if bus:
                dom, rest = bus.split(":", 1)
                addr = f"{int(dom, 16) & 0xffff:04x}:{rest}"
        except (OSError, ValueError, subprocess.SubprocessError):
            return None
    if not addr:
        return None
    base = f"/sys/bus/pci/devices/{addr}"
    try:
        with open(f"{base}/local_cpulist") as f:
            cpus = parse_cpulist(f.read())
        node = open(f"{base}/numa_node").read().strip() if os.path.exists(f"{base}/numa_node") else "?"
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return f"{len(cpus)} CPUs local to GPU {addr} (NUMA node {node})"
    except (OSError, ValueError):
        return None


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def free_port():
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def replica_launch_command(n, argv, port):
    """The command that starts n ranks of this script, one per GPU, through
    torch.distributed.run on this node (rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]


def launch_replicas(n, argv):
    """`--gpus N` (N > 1) started without a launcher: run N ranks of this
    script under torch.distributed.run and return its exit status.  Each rank
    runs its own replica of the workload on GPU LOCAL_RANK; rank 0 prints the
    JSON line.  NCCL's initialisation log stays on (unless NCCL_DEBUG is set),
    so the communicator lines show N ranks."""
    env = dict(os.environ)
    env.setdefault("NCCL_DEBUG", "INFO")
    env.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
    return subprocess.call(replica_launch_command(n, argv, free_port()), env=env)


# --------------------------------------------------------------------------
# CPU oracle timing (the baseline, and the reference arm)
# --------------------------------------------------------------------------

def oracle_inputs(msg_mib, seed0):
    import numpy as np

    n = int(msg_mib * MIB) // 2
    rng = np.random.default_rng(seed0)
    return [(rng.standard_normal(n, dtype=np.float32) * np.float32(1e-3)).astype(np.float16).view(np.uint16)
            for _ in range(R)], n


def time_oracle(msg_mib, seed0=2000):
    import oracle

    oracle.build()
    xs, n = oracle_inputs(msg_mib, seed0)
    t0 = time.perf_counter()
    res = oracle.allreduce(xs, "f16")
    dt = time.perf_counter() - t0
    assert res.status == oracle.OK
    return n * 2 / dt / 1e9, dt, n


def staggered_inputs(rr, wl, w, dev, in_lens=None, out_lens=None):
    """Workload w's inputs and room for its outputs, each side R vectors in
    one allocation, staggered (rank_buffers) so that the ranks' concurrent
    accesses do not all fall on the same memory channels."""
    in_lens = in_lens or [w.count] * w.R
    out_lens = out_lens or [w.count] * w.R
    ins = rr.rank_buffers(w.R, in_lens, w.dtype, dev)
    for r in range(w.R):
        wl.rank_values(w.wid, r, in_lens[r], w.dtype, w.dist, dev, out=ins[r])
    return ins, rr.rank_buffers(w.R, out_lens, w.dtype, dev)


REPLAYS, REPLAY_WARMUP = 20, 5


def time_replays(dev, sets, call, launches):
    """Per-call time (ms) of `call` by CUDA-graph replay: one graph of
    `launches` back-to-back calls cycling through the buffer sets, REPLAY_WARMUP
    untimed replays, then REPLAYS replays each timed with CUDA events on the
    replay stream.  Returns (median, min, max) over the replays of the replay
    time / launches (a replay's events sit on the stream replay() launches on)."""
    import torch

    for ins, outs in sets:  # warm up outside capture (first-call set-up)
        call(ins, outs)
    torch.cuda.synchronize(dev)
    s = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for k in range(launches):
                ins, outs = sets[k % len(sets)]
                call(ins, outs, s)
    for _ in range(REPLAY_WARMUP):
        g.replay()
    torch.cuda.synchronize(dev)
    cur = torch.cuda.current_stream(dev)  # replay() launches on the current stream
    times = []
    for _ in range(REPLAYS):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        g.replay()
        b.record(cur)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b) / launches)
    del g
    return statistics.median(times), min(times), max(times)


def graph_row(rr, wl, w, dev, l2_bytes, peak, launches, algo="ring", cfg=None):
    """Time workload w: CUDA-graph replay of `launches` back-to-back calls over
    rotating buffer sets (>= 3x L2 in total).  Returns one table row."""
    import torch

    op = {"allreduce": rr.OP_ALLREDUCE, "reduce_scatter": rr.OP_REDUCE_SCATTER, "allgather": rr.OP_ALLGATHER}[w.op]
    E = torch.tensor([], dtype=w.dtype).element_size()
    N, R_ = w.count, w.R
    msg = N * E
    lens = [rr.chunk_count(N, R_, c) for c in range(R_)]
    in_lens = lens if op == rr.OP_ALLGATHER else [N] * R_
    out_lens = lens if op == rr.OP_REDUCE_SCATTER else [N] * R_
    set_bytes = (sum(in_lens) + sum(out_lens)) * E
    nsets = max(1, min(16, -(-3 * l2_bytes // set_bytes)))
    sets = []
    for k in range(nsets):
        if k == 0:
            sets.append(staggered_inputs(rr, wl, w, dev, in_lens, out_lens))
        else:
            ins = rr.rank_buffers(R_, in_lens, w.dtype, dev)
            for a, b in zip(ins, sets[0][0]):
                a.copy_(b)
            sets.append((ins, rr.rank_buffers(R_, out_lens, w.dtype, dev)))
    def call(ins, outs, stream=None):
        if algo == "ring":
            rr.collective(op, ins, outs, N, w.wire, w.group_size, stream, cfg)
        else:
            rr.allreduce_algo(ins, outs, w.wire, algo, stream, cfg)

    t_ms, t_min, t_max = time_replays(dev, sets, call, launches)
    alg = (2 * R_ if op == rr.OP_ALLREDUCE else R_ + 1) * msg
    busbw = msg / t_ms / 1e6 * ((2 if op == rr.OP_ALLREDUCE else 1) * (R_ - 1) / R_)
    row = {"workload": w.name if algo == "ring" else f"{w.name}, {algo} order", "op": w.op, "algo": algo,
           "R": R_, "group_size": w.group_size or R_, "count": N,
           "msg_bytes": msg, "ms": round(t_ms, 5), "ms_min": round(t_min, 5), "ms_max": round(t_max, 5),
           "replays": REPLAYS, "algbw_gbs": round(msg / t_ms / 1e6, 2),
           "busbw_gbs": round(busbw, 2), "hbm_gbs": round(alg / t_ms / 1e6, 1),
           "roofline_frac": round(alg / t_ms / 1e6 / peak, 4), "buffer_sets": nsets,
           "plan": rr.plan(op, sets[0][0], sets[0][1], N, w.wire, w.group_size, cfg)}
    del sets
    return row


def bucket_set_row(rr, wl, dev, peak):
    """Workload 5 whole: the 49 gradient buckets of the decoder, all resident
    (one flat in-place vector per rank, about 104 GB), reduced bucket by bucket
    in place as data-parallel training does; timed over one pass."""
    import torch

    counts = wl.decoder_bucket_counts()
    total = sum(counts)
    R_ = 8
    flat = [torch.empty(total, dtype=torch.bfloat16, device=dev) for _ in range(R_)]
    for r in range(R_):  # seeded per rank and bucket (workload 5's recipe)
        off = 0
        for b, n in enumerate(counts):
            wl.rank_values(5, r, n, torch.bfloat16, "grad1e-2", dev, bucket=b, out=flat[r][off:off + n])
            off += n
    views, off = [], 0
    for n in counts:
        views.append([f[off:off + n] for f in flat])
        off += n

    def one_pass():
        for v in views:
            rr.allreduce(v, outs=v)

    one_pass()  # warm-up (and in place: the values grow, the timing does not care)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    one_pass()
    b.record()
    torch.cuda.synchronize(dev)
    t_ms = a.elapsed_time(b)
    msg = total * 2
    row = {"workload": f"fusion buckets: {len(counts)} bf16 buckets of a 32-layer 4096-hidden decoder, "
                       f"R=8, in place, all resident", "op": "allreduce", "R": R_, "count": total,
           "buckets": len(counts), "msg_bytes": msg, "ms": round(t_ms, 3),
           "algbw_gbs": round(msg / t_ms / 1e6, 2), "hbm_gbs": round(2 * R_ * msg / t_ms / 1e6, 1),
           "roofline_frac": round(2 * R_ * msg / t_ms / 1e6 / peak, 4), "gpu_launches": len(counts)}
    del views, flat
    torch.cuda.empty_cache()
    return row


def host_link_speeds(dev, host_in, host_out, dev_src):
    """The host link alone, on the e2e step's own page-locked buffers: the R
    inputs copied to the device, the R results copied back, each alone and
    both at once (one stream each way), median of 3.  Tells a slow host-buffer
    pipeline from a slow link."""
    import torch

    nbytes = sum(t.numel() * t.element_size() for t in host_in)
    dst = [torch.empty_like(t, device=dev) for t in host_in]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(h2d, d2h):
        cur = torch.cuda.current_stream(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(cur)
        up.wait_stream(cur)
        down.wait_stream(cur)
        if h2d:
            with torch.cuda.stream(up):
                for d, h in zip(dst, host_in):
                    d.copy_(h, non_blocking=True)
        if d2h:
            with torch.cuda.stream(down):
                for h, d in zip(host_out, dev_src):
                    h.copy_(d, non_blocking=True)
        cur.wait_stream(up)
        cur.wait_stream(down)
        t1.record(cur)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    def med(h2d, d2h):
        run(h2d, d2h)
        return statistics.median(run(h2d, d2h) for _ in range(3))

    h, d, both = med(True, False), med(False, True), med(True, True)
    del dst
    return {"h2d_ms": round(h, 3), "d2h_ms": round(d, 3), "both_ms": round(both, 3),
            "h2d_gbs": round(nbytes / h / 1e6, 1), "d2h_gbs": round(nbytes / d / 1e6, 1)}


def overlap_rows(rr, wl, dev, pieces=8, rounds=5):
    """Chunked AllReduce overlapped with compute (the pattern of the page
    bjdmk.com.cn/news/5966809, sections 4.2-4.3): `pieces` bf16 GEMMs run on the
    compute stream; after each one an event releases one range of a 512 MiB
    fp16 AllReduce (R = 8) on a communication stream.  For each grid setting
    of the AllReduce (uncapped; capped at a share of the SMs; the library's
    own cap, beside_compute) the two streams are timed alone and together;
    the settings take turns over `rounds` rounds and each row reports medians.
    On one GPU the "communication" is itself HBM traffic that SMs drive, so
    the figure of merit is the time together against the time one after the
    other."""
    import torch

    w = wl.config2(512)
    xs, outs = staggered_inputs(rr, wl, w, dev)
    N = w.count
    step = -(-N // pieces) // 256 * 256
    n = 8192
    A = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    B = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    C = torch.empty(n, n, device=dev, dtype=torch.bfloat16)
    comp, comm = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    evs = [torch.cuda.Event() for _ in range(pieces)]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    settings = [("uncapped", rr.LaunchCfg())]
    for eighths in (7, 6, 5, 4, 3):
        settings.append((f"max_ctas={sms * eighths // 8}", rr.LaunchCfg(0, 0, 0, 0, 0, sms * eighths // 8)))
    settings.append(("beside_compute", rr.LaunchCfg(0, 0, 0, 0, 0, 0, 0, 0, 1)))

    def ranges(k):
        a = k * step
        return a, min(N, a + step)

    def compute_only(cfg):
        with torch.cuda.stream(comp):
            for _ in range(pieces):
                torch.matmul(A, B, out=C)

    def comm_only(cfg):
        for k in range(pieces):
            a, b = ranges(k)
            rr.allreduce_range([x[a:b] for x in xs], [o[a:b] for o in outs], N, a, stream=comm, cfg=cfg)

    def both(cfg):
        for k in range(pieces):
            with torch.cuda.stream(comp):
                torch.matmul(A, B, out=C)
                evs[k].record(comp)
            comm.wait_event(evs[k])
            a, b = ranges(k)
            rr.allreduce_range([x[a:b] for x in xs], [o[a:b] for o in outs], N, a, stream=comm, cfg=cfg)

    def timed(fn, cfg):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        t0.record(cur)
        comp.wait_stream(cur)
        comm.wait_stream(cur)
        fn(cfg)
        cur.wait_stream(comp)
        cur.wait_stream(comm)
        t1.record(cur)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    for _, cfg in settings:  # warm up every setting
        timed(both, cfg)
    times = {name: {"compute": [], "allreduce": [], "together": []} for name, _ in settings}
    for _ in range(rounds):
        for name, cfg in settings:
            times[name]["compute"].append(timed(compute_only, cfg))
            times[name]["allreduce"].append(timed(comm_only, cfg))
            times[name]["together"].append(timed(both, cfg))
    rows = []
    for name, cfg in settings:
        t = {k: statistics.median(v) for k, v in times[name].items()}
        serial = t["compute"] + t["allreduce"]
        grid = rr.plan(rr.OP_ALLREDUCE, [x[:step] for x in xs], [o[:step] for o in outs], step, cfg=cfg)["max_ctas"]
        rows.append({"what": f"{pieces} bf16 GEMMs {n}^3 on a compute stream; after each, one of {pieces} ranges "
                             f"of the 512 MiB R=8 fp16 AllReduce on a communication stream", "setting": name,
                     "allreduce_grid": grid, "compute_ms": round(t["compute"], 3),
                     "allreduce_ms": round(t["allreduce"], 3), "together_ms": round(t["together"], 3),
                     "serial_ms": round(serial, 3), "saved_of_serial": round((serial - t["together"]) / serial, 3),
                     "rounds": rounds})
    del xs, outs, A, B, C
    torch.cuda.empty_cache()
    return rows


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    pg = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import __graft_entry__

    if local == 0:
        __graft_entry__.build()
    if pg:
        pg.barrier()
    import ring_allreduce_reducescatter_gb300 as rr
    from ring_allreduce_reducescatter_gb300 import workloads as wl

    props = torch.cuda.get_device_properties(dev)
    l2_bytes = int(getattr(props, "L2_cache_size", 128 * MIB))
    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (uuid or local)
    affinity = bind_to_gpu_local_cpus(props, gpu_id)
    w = wl.config2(args.msg_mib)
    N = w.count
    msg = N * 2
    xs, outs = staggered_inputs(rr, wl, w, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        rr.allreduce(xs, outs=outs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if rr.device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    sampler = ClockSampler(gpu_id) if local == 0 else None
    time.sleep(0.5 if sampler else 0)

    # timed region: exactly K steps, barrier + synchronize on both sides.  One
    # ring kernel per step and nothing else on the stream, so the kernel's
    # average launch duration is the region's time over K (events between the
    # launches would also stop each launch from overlapping the one before).
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    region0.record(stream)
    for k in range(args.steps):
        step()
    region1.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    if pg:
        pg.barrier()
    region_ms = region0.elapsed_time(region1)
    kern_ms = region_ms / args.steps
    if rr.device_status() != 0:
        raise RuntimeError("device status set during the timed region")
    gpu_launches = args.steps  # one ring_allreduce kernel per step

    region_ms, kern_ms = combine_ranks(pg, [region_ms, kern_ms], dev)
    ms_per_step = region_ms / args.steps
    value = job_throughput(world, msg, ms_per_step)
    peak, peak_kind = measured_hbm_peak()
    achieved = 2 * R * msg / (kern_ms * 1e-3) / 1e9
    digest = kernel_sources_digest()
    traffic = recorded_traffic(digest)
    if sampler:  # only the timed region's samples are used; nvidia-smi polling costs host time
        time.sleep(0.3)
        sampler.stop()
    clocks = sampler.summary(t_host0, t_host1) if sampler else None

    # the size sweep and the other workloads: CUDA-graph replay of back-to-back
    # launches over rotating buffer sets at least 3x the L2 size, so every
    # launch reads inputs that are not in L2 and no host time is included
    sweep, table, overlap, rsag = [], [], None, []
    if not args.no_sweep and world == 1:  # per-GPU tables: every replica would measure the same
        del outs
        torch.cuda.empty_cache()
        for mib in SWEEP_MIB:
            sweep.append(graph_row(rr, wl, wl.config2(mib), dev, l2_bytes, peak, args.sweep_iters))
        torch.cuda.empty_cache()
        if not args.no_workloads:
            for wk in (wl.config1("allreduce"), wl.config1("reduce_scatter"), wl.config1("allgather"), wl.config3(),
                       wl.config4(), wl.config5(0), wl.config2(512, wire="f32")):
                table.append(graph_row(rr, wl, wk, dev, l2_bytes, peak, args.sweep_iters))
                torch.cuda.empty_cache()
            for algo in ("hd", "naive"):
                table.append(graph_row(rr, wl, wl.config2(512), dev, l2_bytes, peak, args.sweep_iters, algo=algo))
                torch.cuda.empty_cache()
            del xs
            torch.cuda.empty_cache()
            table.append(bucket_set_row(rr, wl, dev, peak))
            # ReduceScatter / AllGather over few ranks, chunk boundaries on and off
            # the 16-byte grid (binary16, the planner's choice)
            for op_ in (1, 2):
                for R_ in (2, 3, 4, 8):
                    for mib in (16, 256):
                        for off in (False, True):
                            rsag.extend(path_sweep_point(rr, dev, l2_bytes, peak, op_, R_, mib, torch.float16, None,
                                                         off, False, only_auto=True))
            overlap = overlap_rows(rr, wl, dev)
            xs, outs = staggered_inputs(rr, wl, w, dev)
        else:
            outs = rr.rank_buffers(R, N, torch.float16, dev)

    # end to end through the C ABI's host-buffer entry point (ring_allreduce_host):
    # inputs in page-locked host memory, every output copied back to the host,
    # all inside the timed region; the copies of piece k+1 and k-1 overlap the
    # fold of piece k
    e2e = None
    if not args.no_e2e:
        del outs
        torch.cuda.empty_cache()
        host_in = [torch.empty(N, dtype=torch.float16, pin_memory=True) for _ in range(R)]
        host_out = [torch.empty(N, dtype=torch.float16, pin_memory=True) for _ in range(R)]
        for r in range(R):
            host_in[r].copy_(xs[r])
        piece = args.e2e_piece_mib * MIB // 2
        ws = torch.empty(rr.host_workspace_bytes(R, piece, torch.float16), dtype=torch.uint8, device=dev)
        # the host link on these buffers: where both directions at once are
        # slower than one after the other, the copies take turns
        link = host_link_speeds(dev, host_in, host_out, xs)
        one_way = link["both_ms"] > link["h2d_ms"] + link["d2h_ms"]
        mode = rr.HOST_COPIES_ONE_WAY if one_way else rr.HOST_COPIES_OVERLAP

        def e2e_step():
            rr.allreduce_host(host_in, host_outs=host_out, workspace=ws, copy_mode=mode)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
        if pg:
            pg.barrier()
        marks[0].record(stream)
        for k in range(args.e2e_steps):
            e2e_step()
            marks[k + 1].record(stream)
        torch.cuda.synchronize(dev)
        step_ms = [marks[k].elapsed_time(marks[k + 1]) for k in range(args.e2e_steps)]
        e_ms = combine_ranks(pg, [marks[0].elapsed_time(marks[-1]) / args.e2e_steps], dev)[0]
        e2e = {"value": round(job_throughput(world, msg, e_ms), 3), "unit": UNIT,
               "h2d_bytes_per_step": R * msg, "d2h_bytes_per_step": R * msg, "ms_per_step": round(e_ms, 4),
               "step_ms_min": round(min(step_ms), 3), "step_ms_median": round(statistics.median(step_ms), 3),
               "step_ms_max": round(max(step_ms), 3), "step_ms_all": [round(t, 3) for t in step_ms],
               "steps": args.e2e_steps, "api": "ring_allreduce_host_ex",
               "copy_mode": "one_way" if one_way else "overlap",
               "piece_mib_per_rank": args.e2e_piece_mib, "host_affinity": affinity, "link": link}
        del host_in, host_out, ws
        outs = rr.rank_buffers(R, N, torch.float16, dev)


    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, n = time_oracle(args.cpu_sample_mib)
        cpu = {"value": round(v, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the same workload at {args.cpu_sample_mib} MiB per rank ({n} fp16 elements x {R} "
                         f"ranks), one literal ring simulation, {dt:.2f} s on 1 host core"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"ring allreduce R={R} fp16 per-hop fp16, {args.msg_mib} MiB per rank, "
                                   f"N(0,1e-3)", "R": R, "count": N, "msg_bytes": msg,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (2 x R x msg bytes per step)"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
                         "kernel_ms": round(kern_ms, 5), "algorithmic_bytes_per_launch": 2 * R * msg},
            "busbw_gbs": round(value / world * 2 * (R - 1) / R, 3),
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks, "gpu_launches": gpu_launches,
            "sweep": sweep, "workloads": table, "reduce_scatter_allgather": rsag, "overlap": overlap,
            "kernel_sources": digest,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


# --------------------------------------------------------------------------
# path sweep: the measurements behind the planner's choices
# --------------------------------------------------------------------------

SWEEP_OPS = {"ar": 0, "rs": 1, "ag": 2}


def sweep_variants(rr, op, wide, shifted, all_variants, prefetch=False, explicit=""):
    """(label, cfg) pairs to time at one point: the planner's choice, the tile
    pipeline and the direct path (each forced); with prefetch the direct path
    under each L2-prefetch mode; with all_variants every direct kernel the
    library builds (vectors a thread x register budget)."""
    out = [("auto", None), ("bulk", rr.LaunchCfg(rr.PATH_BULK)), ("direct", rr.LaunchCfg(rr.PATH_DIRECT))]
    if explicit:
        out = [("auto", None)]
        for item in explicit.split(";"):
            vals = [int(v) for v in item.split(",")]
            path, u, occ, pf = vals[:4]
            cap, threads, early, tile, stages = (vals[4:] + [0, 0, 0, 0, 0])[:5]
            label = f"path={path} U={u} occ={occ} prefetch={pf}" + (f" max_ctas={cap}" if cap else "")
            label += (f" threads={threads}" if threads else "") + (f" early={early}" if early else "")
            label += (f" tile={tile}" if tile else "") + (f" stages={stages}" if stages else "")
            out.append((label, rr.LaunchCfg(path, tile, stages, occ, threads, cap, early, u, 0, pf)))
        return out
    if prefetch and not shifted:
        for pf, name in ((1, "none"), (2, "head"), (3, "ahead"), (4, "head+ahead")):
            out.append((f"direct prefetch={name}", rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 0, 0, 0, 0, 0, pf)))
    if all_variants:
        if shifted:
            rows = (1, 2, 4) if op == 2 else ((1, 2) if wide else (1, 2, 3, 4))
            pairs = [(u, 0) for u in rows]
        elif op == 2:
            pairs = [(1, 2), (2, 2), (4, 2)]
        elif wide:
            pairs = [(1, 2), (2, 2)]
        else:
            pairs = [(1, 2), (1, 3), (2, 2), (2, 3), (3, 2), (4, 2)]
        for u, occ in pairs:
            out.append((f"direct U={u} occ={occ or 'auto'}", rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, occ, 0, 0, 0, u)))
    return out


SWEEP_STAGGERS = ((2 << 20), (2 << 20) + (640 << 10) + 256, (5 << 20) + 4096, (1 << 20) + (320 << 10) + 768)


def path_sweep_point(rr, dev, l2_bytes, peak, op, R_, mib, dtype, wire, off_grid, all_variants, prefetch=False,
                     only_auto=False, layouts=1, explicit=""):
    """Time every variant of one (collective, ranks, size) point.  Chunks are
    whole multiples of the 16-byte vector (or, off_grid, one element more, so
    chunk boundaries fall off the 16-byte grid).  With layouts > 1 every
    variant is timed on that many buffer layouts (rank vectors staggered by
    different distances; where the ranks sit in HBM moves some points by up
    to ~10 %) and the row reports the median over layouts.  Returns JSON rows."""
    rows = None
    for j in range(layouts):
        part = path_sweep_layout(rr, dev, l2_bytes, peak, op, R_, mib, dtype, wire, off_grid, all_variants, prefetch,
                                 only_auto, SWEEP_STAGGERS[j % len(SWEEP_STAGGERS)], explicit)
        if rows is None:
            rows = part
            for r in rows:
                r["us_layouts"] = [r["us"]]
        else:
            for r, q in zip(rows, part):
                r["us_layouts"].append(q["us"])
    for r in rows or []:
        if layouts > 1:
            med = statistics.median(r["us_layouts"])
            r["frac"] = round(r["frac"] * r["us"] / med, 4)
            r["us"] = round(med, 3)
    return rows or []


def path_sweep_layout(rr, dev, l2_bytes, peak, op, R_, mib, dtype, wire, off_grid, all_variants, prefetch, only_auto,
                      stagger, explicit=""):
    import torch

    E = torch.tensor([], dtype=dtype).element_size()
    V = 16 // E
    base = max(V, (int(mib * MIB) // E) // R_ // V * V) + (1 if off_grid else 0)
    N = R_ * base
    lens = [rr.chunk_count(N, R_, c) for c in range(R_)]
    in_lens = lens if op == 2 else [N] * R_
    out_lens = lens if op == 1 else [N] * R_
    set_bytes = (sum(in_lens) + sum(out_lens)) * E
    nsets = max(1, min(16, -(-3 * l2_bytes // set_bytes)))
    sets = []
    for k in range(nsets):
        ins = rr.rank_buffers(R_, in_lens, dtype, dev, stagger_bytes=stagger)
        for x in ins:
            x.copy_(torch.randn(x.numel(), device=dev).mul_(1e-2).to(dtype))
        sets.append((ins, rr.rank_buffers(R_, out_lens, dtype, dev, stagger_bytes=stagger)))
    msg = N * E
    alg = (2 * R_ if op == 0 else R_ + 1) * msg
    # about 2 ms of work per replay, 4 to 40 launches
    launches = max(4, min(40, int(2e-3 * 6.5e12 / alg) + 1))
    wide = dtype != torch.float32 and wire == "f32"
    shifted = off_grid and op != 0
    rows = []
    variants = [("auto", None)] if only_auto else sweep_variants(rr, op, wide, shifted, all_variants, prefetch,
                                                                 explicit)
    for label, cfg in variants:
        try:
            plan = rr.plan(op, sets[0][0], sets[0][1], N, wire, 0, cfg)
        except rr.RingError:
            continue  # a path these buffers do not allow
        if label != "auto" and plan["path"] == rr.PATH_SIMPLE:
            continue

        def call(ins, outs, stream=None, cfg=cfg):
            rr.collective(op, ins, outs, N, wire, 0, stream, cfg)

        med, lo, hi = time_replays(dev, sets, call, launches)
        rows.append({"op": {0: "allreduce", 1: "reduce_scatter", 2: "allgather"}[op], "R": R_, "count": N,
                     "msg_bytes": msg, "off_grid": off_grid, "variant": label,
                     "path": {1: "bulk", 2: "simple", 3: "direct"}[plan["path"]], "vectors": plan["vectors"],
                     "ctas_per_sm": plan["ctas_per_sm"], "prefetch": plan["prefetch"], "grid": plan["max_ctas"],
                     "us": round(med * 1e3, 3), "us_min": round(lo * 1e3, 3), "us_max": round(hi * 1e3, 3),
                     "frac": round(alg / (med * 1e-3) / 1e9 / peak, 4), "replays": REPLAYS, "launches": launches})
    del sets
    torch.cuda.empty_cache()
    return rows


def run_path_sweep(args):
    """--path-sweep: one JSON line per (point, variant) on stdout; the planner's
    rules in the library cite these measurements."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import ring_allreduce_reducescatter_gb300 as rr

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = int(getattr(props, "L2_cache_size", 128 * MIB))
    peak, _ = measured_hbm_peak()
    dtype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[args.sweep_dtype]
    wire = args.sweep_wire or None
    all_rows = []
    for op_name in args.sweep_ops.split(","):
        op = SWEEP_OPS[op_name]
        for R_ in (int(v) for v in args.sweep_ranks.split(",")):
            for mib in (float(v) for v in args.sweep_mib.split(",")):
                for off_grid in ((False, True) if args.sweep_off_grid == "both" else
                                 ((True,) if args.sweep_off_grid == "only" else (False,))):
                    if off_grid and op == 0:
                        continue
                    for row in path_sweep_point(rr, dev, l2_bytes, peak, op, R_, mib, dtype, wire, off_grid,
                                                args.sweep_variants, args.sweep_prefetch,
                                                layouts=args.sweep_layouts, explicit=args.sweep_cfg):
                        print(json.dumps(row), flush=True)
                        all_rows.append(row)
    if args.sweep_table:
        with open(args.sweep_table, "w") as f:
            f.write(path_choice_table(all_rows, args))


def path_choice_table(rows, args):
    """Markdown table of the tile pipeline against the direct path at every
    point (the planner's path and whether it is within 5 % of the faster),
    from path-sweep rows; tests/test_abi_cpu.py checks the planner against
    the committed copy."""
    pts = {}
    for r in rows:
        pts.setdefault((r["op"], r["R"], r["count"], r["msg_bytes"], r["off_grid"]), {})[r["variant"]] = r
    cmd = "python bench.py --path-sweep " + " ".join(
        f"--{k.replace('_', '-')} {v}" for k, v in (("sweep_ops", args.sweep_ops), ("sweep_ranks", args.sweep_ranks),
                                                   ("sweep_mib", args.sweep_mib), ("sweep_dtype", args.sweep_dtype),
                                                   ("sweep_layouts", args.sweep_layouts),
                                                   ("sweep_off_grid", args.sweep_off_grid))) + " --sweep-table FILE"
    out = ["# Path choice: tile pipeline against direct path", "",
           "Made by (one GB300; microseconds per call, CUDA-graph replay over buffer sets of at least 3x the",
           f"L2, median of {REPLAYS} replays; with several layouts the median over layouts):", "", "```", cmd, "```",
           "", "| op | R | count | msg bytes | off grid | bulk us | direct us | planner | planner ok |",
           "|---|---|---|---|---|---|---|---|---|"]
    for (op, R_, count, msg, off), v in pts.items():
        if "auto" not in v or "direct" not in v:
            continue
        b = v["bulk"]["us"] if "bulk" in v else None
        d = v["direct"]["us"]
        planner = v["auto"]["path"]
        best = min(x for x in (b, d) if x is not None)
        mine = b if planner == "bulk" else d if planner == "direct" else None
        ok = mine is not None and mine <= 1.05 * best
        out.append(f"| {op} | {R_} | {count} | {msg} | {int(off)} | {b if b is not None else '-'} | {d} | {planner} | "
                   f"{'yes' if ok else 'NO'} |")
    return "\n".join(out) + "\n"


# --------------------------------------------------------------------------
# reference arm: the CPU oracle, timed as it stands
# --------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    # size each step's sample so the whole run stays within about two minutes
    _, dt_cal, n_cal = time_oracle(0.25, seed0=1999)
    per_elem = dt_cal / n_cal
    budget = min(2.0, 120.0 / (args.warmup + args.steps))
    n = max(2048, int(budget / per_elem) // 256 * 256)
    if args.ref_sample_mib:
        n = min(n, args.ref_sample_mib * MIB // 2)
    mib = n * 2 / MIB
    times = []
    for k in range(args.warmup + args.steps):
        v, dt, n = time_oracle(mib, seed0=2000 + k)
        if k >= args.warmup:
            times.append(dt)
    ms = statistics.mean(times) * 1e3
    value = n * 2 / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"ring allreduce R={R} fp16 per-hop fp16, {args.msg_mib} MiB per rank, "
                               f"N(0,1e-3)", "R": R, "count": args.msg_mib * MIB // 2,
                   "sample_elements_per_rank": n},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step: the workload at {n} fp16 elements per rank x {R} ranks "
                                   f"({mib:.3f} MiB per rank), one literal ring simulation on 1 host core"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--msg-mib", type=int, default=MSG_MIB)
    ap.add_argument("--sweep-iters", type=int, default=40)
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--e2e-piece-mib", type=int, default=32)
    ap.add_argument("--cpu-sample-mib", type=int, default=CPU_SAMPLE_MIB)
    ap.add_argument("--ref-sample-mib", type=int, default=REF_SAMPLE_MIB)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--overlap-only", action="store_true",
                    help="print only the compute-overlap table (JSON lines) of the chunked AllReduce")
    ap.add_argument("--path-sweep", action="store_true",
                    help="time the planner's choice against the forced tile pipeline and direct path instead")
    ap.add_argument("--sweep-ops", default="ar,rs,ag")
    ap.add_argument("--sweep-ranks", default="2,3,4,5,8,9,12,16,32")
    ap.add_argument("--sweep-mib", default="1,4,16,64,256")
    ap.add_argument("--sweep-dtype", default="f16", choices=["f32", "f16", "bf16"])
    ap.add_argument("--sweep-wire", default="", choices=["", "f32", "f16", "bf16"])
    ap.add_argument("--sweep-off-grid", default="no", choices=["no", "only", "both"],
                    help="chunk boundaries off the 16-byte grid (ReduceScatter / AllGather)")
    ap.add_argument("--sweep-variants", action="store_true", help="every direct kernel variant too")
    ap.add_argument("--sweep-prefetch", action="store_true", help="the direct path under each L2-prefetch mode too")
    ap.add_argument("--sweep-layouts", type=int, default=1, help="buffer layouts per point (median reported)")
    ap.add_argument("--sweep-table", default="", help="also write the tile-vs-direct table (markdown) to this file")
    ap.add_argument("--sweep-cfg", default="",
                    help="explicit launch configurations "
                         "'path,vectors,ctas_per_sm,prefetch[,max_ctas[,threads[,early_launch[,tile_bytes"
                         "[,stages]]]]];...' "
                         "(with auto)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if "WORLD_SIZE" in os.environ and int(os.environ["WORLD_SIZE"]) != args.gpus:
        ap.error(f"--gpus {args.gpus} but the launcher started WORLD_SIZE={os.environ['WORLD_SIZE']} ranks")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]))
    if args.overlap_only:
        import torch

        import __graft_entry__

        __graft_entry__.build()
        import ring_allreduce_reducescatter_gb300 as rr
        from ring_allreduce_reducescatter_gb300 import workloads as wl

        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        for row in overlap_rows(rr, wl, dev):
            print(json.dumps(row), flush=True)
    elif args.path_sweep:
        run_path_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
