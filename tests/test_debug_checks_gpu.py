"""The debug build: every device access checked against its buffer.

libringred_debug.so is the same library compiled with RR_DEBUG_CHECKS: each
load, store, bulk copy and prefetch a kernel makes of a rank buffer is
checked against that buffer's extent in the launch, and one outside it is
skipped and recorded in the device status word instead of being made.

test_edge_grids_under_the_debug_build builds it and reruns the edge-case
grids of tests/test_parity_gpu.py against it in a child process (the library
is chosen by RINGRED_LIBRARY before the binding loads it), where every test
also checks that the status word stays clear: no kernel index leaves its
buffer, on any path, format, rank count or ragged size of those grids.  The
child also runs the tests below, which need the debug build: with the checks
told that every buffer is 16 bytes shorter than it is, each path reports the
accesses to the last 16 bytes (which are valid, so nothing faults), and with
the true extents the results are bit-exact.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EDGE_GRIDS = ("edge_grid or maximum_rank_counts or two_level_grid or reduce_scatter_grid or allgather_grid or "
              "shifted or misaligned or outputs_do_not_write_outside or vectors_over_chunk_boundaries or "
              "every_direct_variant or capped_grids or algorithm_grid or ranges_concatenate or "
              "direct_occupancy_variants or algorithm_occupancy_variants or workload1_full or allreduce_rows or "
              "allgather_rows or chunk_by_chunk")


def test_edge_grids_under_the_debug_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_allreduce_reducescatter_gb300 import _build

    oracle.build()
    debug_lib = _build.build(debug=True)
    env = dict(os.environ, RINGRED_LIBRARY=debug_lib)
    probe = subprocess.run([sys.executable, "-c", "import ring_allreduce_reducescatter_gb300 as rr; "
                            "print(rr.LIB_PATH, rr.debug_checks())"],
                           capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.split() == [debug_lib, "True"], probe.stdout
    # one -k for both files; never this test itself (the child would recurse)
    select = f"(({EDGE_GRIDS}) or checks_fire or true_extents) and not under_the_debug_build"
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_parity_gpu.py"),
                        os.path.join(ROOT, "tests", "test_debug_checks_gpu.py"), "-k", select],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=3000)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    summary = [ln for ln in r.stdout.splitlines() if " passed" in ln]
    assert summary and "skipped" not in summary[-1], tail


@pytest.fixture(scope="module")
def drr():
    """The debug build, when this process loaded it (the child process above)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ring_allreduce_reducescatter_gb300 as rr

    if not os.environ.get("RINGRED_LIBRARY") or not rr.debug_checks():
        pytest.skip("runs in the debug build's child process")
    torch.cuda.set_device(0)
    return rr


def host(t):
    t = t.detach().cpu().contiguous()
    return t.numpy().view(np.uint32) if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)


def cases(rr):
    """(what, op, ins, outs, count, wire, cfg, algo) on every path: tile
    pipeline, direct (aligned, shifted, halving-doubling, the chunk-by-chunk
    rows on aligned chunks), one element."""
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    out = []
    for R, N, dtype in ((4, 4 * 8192, torch.float32), (3, 3 * (8 * 700 + 1), torch.float16)):
        xs = [torch.randn(N, generator=g, device="cuda").to(dtype) for _ in range(R)]
        lens = [rr.chunk_count(N, R, c) for c in range(R)]
        for path in (rr.PATH_BULK, rr.PATH_DIRECT, rr.PATH_SIMPLE):
            cfg = rr.LaunchCfg(path)
            out.append((f"AR R={R} path={path}", rr.OP_ALLREDUCE, xs, [torch.empty_like(x) for x in xs], N, None, cfg,
                        "ring"))
            if path == rr.PATH_BULK and (N // R * xs[0].element_size()) % 16:
                continue  # the tile pipeline needs chunk offsets on 16 bytes
            out.append((f"RS R={R} path={path}", rr.OP_REDUCE_SCATTER, xs,
                        [torch.empty(n, dtype=dtype, device="cuda") for n in lens], N, None, cfg, "ring"))
            chunks = [x[:n].clone() for x, n in zip(xs, lens)]
            out.append((f"AG R={R} path={path}", rr.OP_ALLGATHER, chunks,
                        [torch.empty(N, dtype=dtype, device="cuda") for _ in range(R)], N, None, cfg, "ring"))
        out.append((f"AR R={R} halving-doubling", rr.OP_ALLREDUCE, xs, [torch.empty_like(x) for x in xs], N, None,
                    rr.LaunchCfg(rr.PATH_DIRECT), "hd"))
    # the chunk-by-chunk rows on chunks on the grid: AllReduce over two ranks
    # from 16 MiB, AllGather over four from 12 MiB, ReduceScatter over two
    # from 64 MiB (binary16; ragged last chunks)
    for what, op, R, N in (("AR rows", rr.OP_ALLREDUCE, 2, 2 * (4 << 20) + 1),
                           ("AG rows", rr.OP_ALLGATHER, 4, 4 * (3 << 19) + 3),
                           ("RS rows", rr.OP_REDUCE_SCATTER, 2, 2 * (16 << 20) + 1)):
        xs = [torch.randn(N, generator=g, device="cuda").to(torch.float16) for _ in range(R)]
        lens = [rr.chunk_count(N, R, c) for c in range(R)]
        if op == rr.OP_ALLGATHER:
            ins, outs = [x[:n].clone() for x, n in zip(xs, lens)], [torch.empty(N, dtype=torch.float16,
                                                                               device="cuda") for _ in range(R)]
        elif op == rr.OP_REDUCE_SCATTER:
            ins, outs = xs, [torch.empty(n, dtype=torch.float16, device="cuda") for n in lens]
        else:
            ins, outs = xs, [torch.empty_like(x) for x in xs]
        out.append((f"{what} R={R} N={N}", op, ins, outs, N, None, rr.LaunchCfg(rr.PATH_DIRECT), "ring"))
    return out


def run(rr, case):
    what, op, ins, outs, N, wire, cfg, algo = case
    if algo == "ring":
        rr.collective(op, ins, outs, N, wire, 0, None, cfg)
    else:
        rr.allreduce_algo(ins, outs, wire, algo, None, cfg)
    torch.cuda.synchronize()
    return outs


def test_checks_fire_on_every_path(drr):
    try:
        drr.debug_set_margin(16)
        for case in cases(drr):
            run(drr, case)
            assert drr.device_status() == 2, f"{case[0]}: the checks did not report the last 16 bytes"
    finally:
        drr.debug_set_margin(0)
    assert drr.device_status() == 0


def test_true_extents_are_clean_and_exact(drr):
    names = {torch.float32: "f32", torch.float16: "f16"}
    for case in cases(drr):
        what, op, ins, outs, N, wire, cfg, algo = case
        run(drr, case)
        assert drr.device_status() == 0, what
        hin = [host(x) for x in ins]
        dt = names[ins[0].dtype]
        if dt == "f32":
            hin = [h.view(np.float32) for h in hin]
        if op == drr.OP_ALLREDUCE:
            ref = oracle.allreduce(hin, dt) if algo == "ring" else oracle.allreduce_algo(hin, dt, None, algo)
        elif op == drr.OP_REDUCE_SCATTER:
            ref = oracle.reduce_scatter(hin, dt)
        else:
            ref = oracle.allgather(hin, N, dt)
        for r, o in enumerate(outs):
            want = np.asarray(ref.outs[r])
            want = want.view(np.uint32) if want.dtype == np.float32 else want
            assert np.array_equal(host(o), want), f"{what} output {r}"
