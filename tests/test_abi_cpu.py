"""Host-side tests of the C ABI: no GPU needed, no kernel launched.

The library must load, export every function include/ringred.h declares, and
reject bad arguments before it makes any CUDA call (the validation runs on the
host), so fake device addresses are enough here.
"""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringred.h")

OK, EINVAL, EUNSUP, EALIAS, ECUDA, ETIMEOUT = range(6)
AR, RS, AG = 0, 1, 2
F32, F16, BF16 = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    from ring_allreduce_reducescatter_gb300 import _build

    _build.build()
    import ring_allreduce_reducescatter_gb300 as rr

    return rr.lib()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:rr_status|size_t|const char|int)\s*\**\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_collectives():
    names = declared_functions()
    for want in ("ring_allreduce", "ring_reduce_scatter", "ring_allgather", "ring_allreduce_ex",
                 "ring_reduce_scatter_ex", "ring_collective", "ring_plan", "ring_chunk_count",
                 "ring_chunk_offset", "ring_status_string", "ring_device_status",
                 "ring_selftest_bounded_wait", "ring_abi_version"):
        assert want in names


def test_header_is_c_and_links_from_c(L, tmp_path):
    """include/ringred.h compiles as C11 (no CUDA or C++ headers) and a C
    program links libringred.so and gets the documented answers."""
    import subprocess

    import ring_allreduce_reducescatter_gb300 as rr

    exe = tmp_path / "abi_from_c"
    libdir = os.path.dirname(rr.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "csrc", "abi_from_c.c"), "-o", str(exe), "-L", libdir, "-lringred",
                    f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    lines = dict(l.split(" ", 1) for l in out if l)
    assert lines["abi"] == "3"
    assert out[1:5] == ["chunk 0 2 0", "chunk 1 2 2", "chunk 2 2 4", "chunk 3 4 6"]
    assert lines["bad_rank_count"] == str(EINVAL) and lines["bad_dtype"] == str(EINVAL)
    assert lines["unsupported_pair"] == str(EUNSUP) and lines["alias"] == str(EALIAS)
    assert lines["empty"] == str(OK)
    assert "alias" in lines["status"].lower() or "overlap" in lines["status"].lower()


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_last_cuda_error_is_recorded(L):
    """Without a GPU a valid call fails in the runtime: RR_ERR_CUDA, and the
    runtime error behind it is kept for the calling thread."""
    import ring_allreduce_reducescatter_gb300 as rr

    rr.lib()
    ins, outs = fake(4, 100, 4)
    st = call(L, AR, ins, outs, 4, 100, F32)
    assert st == ECUDA
    assert L.ring_last_cuda_error() != 0
    assert L.ring_last_cuda_error_string() not in (b"", b"no CUDA error")
    err = rr.RingError(rr.ERR_CUDA, "probe")
    assert err.cuda_error == L.ring_last_cuda_error() and "CUDA error" in str(err)


def test_abi_version(L):
    assert L.ring_abi_version() == 3


def test_status_strings(L):
    for s in range(6):
        assert L.ring_status_string(s)
    assert b"unknown" in L.ring_status_string(77)


def test_chunk_table_agrees_with_oracle(L):
    for R in range(1, 17):
        for N in list(range(0, 70)) + [1_048_576, 50_000_017, 16_777_216, 2 ** 33 + 7]:
            for c in range(R):
                assert L.ring_chunk_count(N, R, c) == oracle.chunk_len(N, R, c)
                assert L.ring_chunk_offset(N, R, c) == oracle.chunk_off(N, R, c)
    assert L.ring_chunk_count(10, 0, 0) == 0
    assert L.ring_chunk_count(10, 4, 4) == 0
    assert L.ring_chunk_offset(10, 4, -1) == 0


def ptrs(vals):
    arr = (ctypes.c_void_p * len(vals))()
    for k, v in enumerate(vals):
        arr[k] = v
    return arr


BASE = 0x7F0000000000  # fake, never dereferenced


def fake(R, count, E, gap=1 << 24):
    ins = [BASE + r * gap for r in range(R)]
    outs = [BASE + (R + r) * gap for r in range(R)]
    return ins, outs


def call(L, op, ins, outs, R, count, dtype, wire=None, group=0, cfg=None):
    import ring_allreduce_reducescatter_gb300 as rr

    wire = dtype if wire is None else wire
    c = None
    if cfg is not None:
        c = ctypes.byref(rr.LaunchCfg(*cfg))
    return L.ring_collective(op, ptrs(ins) if ins is not None else None,
                             ptrs(outs) if outs is not None else None, R, count, dtype, wire, group, c, None)


def test_bad_rank_counts(L):
    ins, outs = fake(64, 100, 4)
    assert call(L, AR, ins[:0], outs[:0], 0, 100, F32) == EINVAL
    assert call(L, AR, ins + [BASE], outs + [BASE], 65, 100, F32) == EINVAL


def test_bad_dtypes_and_pairs(L):
    ins, outs = fake(4, 100, 4)
    assert call(L, AR, ins, outs, 4, 100, 3) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F16, F32) not in (EINVAL, EUNSUP, EALIAS)  # binary32 accumulation
    assert call(L, AR, ins, outs, 4, 100, F16, BF16) == EUNSUP
    assert call(L, AR, ins, outs, 4, 100, BF16, F16) == EUNSUP
    assert call(L, AG, ins, outs, 4, 100, F32, BF16) == EUNSUP


def test_bad_group_sizes(L):
    ins, outs = fake(8, 100, 4)
    assert call(L, AR, ins, outs, 8, 100, F32, group=3) == EINVAL
    assert call(L, AR, ins, outs, 8, 100, F32, group=16) == EINVAL
    assert call(L, AR, ins, outs, 8, 100, F32, group=-1) == EINVAL
    assert call(L, RS, ins, outs, 8, 100, F32, group=4) == EINVAL
    assert call(L, AG, ins, outs, 8, 100, F32, group=2) == EINVAL


def test_null_and_misaligned_pointers(L):
    ins, outs = fake(4, 100, 4)
    assert call(L, AR, None, outs, 4, 100, F32) == EINVAL
    assert call(L, AR, ins, None, 4, 100, F32) == EINVAL
    assert call(L, AR, [0] + ins[1:], outs, 4, 100, F32) == EINVAL
    assert call(L, AR, ins, outs[:3] + [0], 4, 100, F32) == EINVAL
    assert call(L, AR, [ins[0] + 2] + ins[1:], outs, 4, 100, F32) == EINVAL  # not 4-byte aligned
    assert call(L, AR, ins, [outs[0] + 1] + outs[1:], 4, 100, F16) == EINVAL
    # zero-length buffers may be NULL: AllGather with N < R has empty chunks 0..R-2
    r = call(L, AG, [0, 0, 0, ins[3]], outs, 4, 3, F32)
    assert r not in (EINVAL, EALIAS, EUNSUP)


def test_count_zero_is_a_no_op(L):
    assert call(L, AR, [0] * 4, [0] * 4, 4, 0, F32) == OK
    assert call(L, RS, [0] * 4, [0] * 4, 4, 0, F16) == OK
    assert call(L, AG, [0] * 4, [0] * 4, 4, 0, BF16) == OK


def test_huge_count_and_address_wrap(L):
    ins, outs = fake(2, 100, 4)
    assert call(L, AR, ins, outs, 2, 2 ** 62, F32) == EINVAL
    top = (1 << 64) - 64
    assert call(L, AR, [top, ins[1]], outs, 2, 100, F32) == EINVAL


def test_aliasing(L):
    R, N, E = 4, 1000, 4
    ins, outs = fake(R, N, E)
    # outputs overlapping each other
    assert call(L, AR, ins, [outs[0], outs[0] + 400] + outs[2:], R, N, F32) == EALIAS
    # an output overlapping another rank's input
    assert call(L, AR, ins, [ins[1] + 16] + outs[1:], R, N, F32) == EALIAS
    # partial overlap with its own input
    assert call(L, AR, ins, [ins[0] + 16] + outs[1:], R, N, F32) == EALIAS
    # in place is allowed for AllReduce (validation passes; the call then needs a device)
    assert call(L, AR, ins, list(ins), R, N, F32) not in (EALIAS, EINVAL, EUNSUP)
    # ... but not for ReduceScatter / AllGather
    assert call(L, RS, ins, list(ins), R, N, F32) == EALIAS
    assert call(L, AG, ins, list(ins), R, N, F32) == EALIAS
    # inputs may overlap one another (they are only read)
    assert call(L, AR, [ins[0]] * R, outs, R, N, F32) not in (EALIAS, EINVAL, EUNSUP)
    # ReduceScatter outputs are chunk-sized: back to back is fine, one byte more is not
    rs_len = N // R * E
    packed = [outs[0] + k * rs_len for k in range(R)]
    assert call(L, RS, ins, packed, R, N, F32) not in (EALIAS, EINVAL, EUNSUP)
    assert call(L, RS, ins, [packed[0], packed[1] - 4] + packed[2:], R, N, F32) == EALIAS


def test_bad_launch_cfg(L):
    ins, outs = fake(4, 100, 4)
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(4, 0, 0, 0, 0)) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(1, 24, 0, 0, 0)) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(1, 0, 17, 0, 0)) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(1, 0, 1, 0, 0)) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(1, 0, 0, 5, 0)) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(1, 0, 0, 0, 1000)) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(0, 0, 0, 0, 0, 0, 3)) == EINVAL
    assert call(L, AR, ins, outs, 4, 100, F32, cfg=(0, 0, 0, 0, 0, 0, -1)) == EINVAL


def test_early_launch_choice(L):
    """Programmatic dependent launch is the default on every path; 2 asks for
    plain stream order and 1 for the early launch, whatever the path."""
    for path in (0, 1, 2, 3):
        for op in (AR, RS, AG):
            st, ch, _, _ = plan_dev(L, op, 8, 1 << 20, F16, cfg=(path, 0, 0, 0, 0) if path else None)
            assert st == OK and ch["early_launch"] == 1, (path, op, ch)
            for el in (1, 2):
                st, ch, _, _ = plan_dev(L, op, 8, 1 << 20, F16, cfg=(path, 0, 0, 0, 0, 0, el))
                assert st == OK and ch["early_launch"] == el, (path, op, el, ch)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import ring_allreduce_reducescatter_gb300 as rr

    monkeypatch.setattr(rr, "_lib", None)
    monkeypatch.setattr(rr, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        rr.lib()


def test_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "ring_allreduce_reducescatter_gb300")
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"].*oracle)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    assert not pat.search(f.read()), fn


# --------------------------------------------------------------------------
# the launch planner, for a described GB300 (152 SMs, 228 KB / SM, 227 KB / CTA)
# --------------------------------------------------------------------------

GB300 = dict(sms=152, smem_per_sm=233472, optin=232448)


def plan_dev(L, op, R, count, dtype, wire=None, group=0, aligned=1, cfg=None, dev=GB300):
    import ring_allreduce_reducescatter_gb300 as rr

    chosen = rr.LaunchCfg()
    grid = ctypes.c_int(0)
    smem = ctypes.c_size_t(0)
    L.ring_plan_device.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(rr.LaunchCfg), ctypes.POINTER(rr.LaunchCfg),
                                   ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)]
    L.ring_plan_device.restype = ctypes.c_int
    st = L.ring_plan_device(op, R, count, dtype, dtype if wire is None else wire, group, aligned, dev["sms"],
                            dev["smem_per_sm"], dev["optin"],
                            ctypes.byref(rr.LaunchCfg(*cfg)) if cfg else None, ctypes.byref(chosen),
                            ctypes.byref(grid), ctypes.byref(smem))
    return st, chosen.as_dict(), grid.value, smem.value


def test_planner_invariants_every_rank_count(L):
    """Every plan keeps tiles on 16-byte multiples and within shared memory."""
    counts = [1, 7, 8, 100, 4096, 65537, 524_288, 1_048_576, 8_388_608, 50_000_017, 268_435_456]
    for R in range(1, 65):
        for op in (AR, RS, AG):
            for dtype, E in ((F32, 4), (F16, 2), (BF16, 2)):
                for N in counts:
                    for ctas in (0, 1, 2, 3, 4):
                        cfg = (0, 0, 0, ctas, 0) if ctas else None
                        st, ch, grid, smem = plan_dev(L, op, R, N, dtype, cfg=cfg)
                        assert st == OK, (R, op, dtype, N, ctas, st)
                        assert grid >= 1
                        if ch["path"] == 1:
                            slots = 1 if op == AG else R
                            tile = ch["tile_bytes"]
                            assert tile >= 16 and tile % 16 == 0 and tile % E == 0, (R, N, tile)
                            assert 2 <= ch["stages"] <= 16
                            assert smem == ch["stages"] * (tile * slots + 8)
                            assert smem <= min(GB300["optin"], GB300["smem_per_sm"] // ch["ctas_per_sm"] - 1024)
                            assert grid <= GB300["sms"] * ch["ctas_per_sm"]
                            assert (N * E) // 16 > 0
                            if op != AR:
                                assert (N // R * E) % 16 == 0
                        else:
                            assert 64 <= ch["threads"] <= 1024
                        if ch["path"] == 3:  # direct: at most sixteen 128-thread CTAs per SM, plus one
                            assert ch["threads"] == 128 and smem == 0
                            assert grid <= GB300["sms"] * 16 + 1, (R, op, dtype, N, grid)


def test_planner_paths(L):
    BULK, SIMPLE, DIRECT = 1, 2, 3
    # unaligned buffers or sub-16-byte messages take the simple path
    assert plan_dev(L, AR, 8, 1 << 20, F16, aligned=0)[1]["path"] == SIMPLE
    assert plan_dev(L, AR, 8, 7, F16)[1]["path"] == SIMPLE
    # the measured choice between the two aligned paths
    assert plan_dev(L, AR, 8, 1 << 28, F16)[1]["path"] == DIRECT
    assert plan_dev(L, AR, 32, 1 << 20, F16)[1]["path"] == DIRECT
    assert plan_dev(L, AR, 2, 1 << 28, F16)[1]["path"] == DIRECT
    assert plan_dev(L, RS, 2, 1 << 28, F16)[1]["path"] == DIRECT
    for R in (3, 4, 5, 6, 7, 9, 12, 24, 32):
        assert plan_dev(L, AR, R, 1 << 26, F32)[1]["path"] == DIRECT
    assert plan_dev(L, AR, 16, 1 << 22, F32)[1]["path"] == DIRECT     # 16 MiB per rank
    assert plan_dev(L, AR, 16, 1 << 24, F32)[1]["path"] == BULK       # 64 MiB per rank
    assert plan_dev(L, RS, 4, 1 << 22, F32)[1]["path"] == DIRECT
    assert plan_dev(L, AG, 16, 1 << 24, F32)[1]["path"] == DIRECT
    assert plan_dev(L, AG, 8, 1 << 24, F32)[1]["path"] == DIRECT
    assert plan_dev(L, AR, 8, 1 << 28, F16, cfg=(0, 0, 0, 0, 0, 96))[1]["path"] == BULK  # capped grid
    # ReduceScatter / AllGather with chunk boundaries off the 16-byte grid: the
    # direct path's shifted kernel; the tile pipeline needs them on the grid
    assert plan_dev(L, RS, 8, 8 * 1001, F16)[1]["path"] == DIRECT
    assert plan_dev(L, AG, 8, 8 * 1001 + 3, F32)[1]["path"] == DIRECT
    assert plan_dev(L, RS, 8, 8 * 1001, F16, aligned=0)[1]["path"] == SIMPLE
    assert plan_dev(L, RS, 8, 8 * 1024, F16, cfg=(BULK, 0, 0, 0, 0))[1]["path"] == BULK
    assert plan_dev(L, AG, 8, 8 * 1024, F32, cfg=(BULK, 0, 0, 0, 0))[1]["path"] == BULK
    # a forced bulk path the buffers do not allow is refused
    assert plan_dev(L, RS, 8, 8 * 1001, F16, cfg=(1, 0, 0, 0, 0))[0] == EUNSUP
    # a forced configuration that does not fit shared memory is refused
    assert plan_dev(L, AR, 64, 1 << 20, F32, cfg=(1, 4096, 8, 1, 0))[0] == EUNSUP
    # the two-level ring plans like the flat ring of all its ranks
    st, ch, _, _ = plan_dev(L, AR, 16, 1 << 24, F32, group=8)
    assert st == OK and ch["path"] == DIRECT


# --------------------------------------------------------------------------
# ranges and the host-buffer pipeline: argument checks
# --------------------------------------------------------------------------

def call_range(L, ins, outs, R, count, first, n, dtype, wire=None, group=0):
    import ring_allreduce_reducescatter_gb300 as rr

    rr.lib()
    return L.ring_allreduce_range(ptrs(ins), ptrs(outs), R, count, first, n, dtype,
                                  dtype if wire is None else wire, group, None, None)


def test_range_arguments(L):
    ins, outs = fake(4, 100, 4)
    assert call_range(L, ins, outs, 4, 100, 90, 11, F32) == EINVAL   # past the end
    assert call_range(L, ins, outs, 4, 100, 101, 0, F32) == EINVAL
    assert call_range(L, ins, outs, 4, 100, 100, 0, F32) == OK       # empty range at the end
    assert call_range(L, ins, outs, 4, 100, 0, 0, F32) == OK
    assert call_range(L, ins, outs, 0, 100, 0, 10, F32) == EINVAL
    assert call_range(L, ins, outs, 4, 100, 0, 10, F16, BF16) == EUNSUP
    assert call_range(L, ins, outs, 4, 100, 0, 10, F32, group=3) == EINVAL
    assert call_range(L, ins, [ins[1]] + outs[1:], 4, 100, 0, 10, F32) == EALIAS
    assert call_range(L, ins, list(ins), 4, 100, 50, 10, F32) not in (EINVAL, EALIAS, EUNSUP)


def call_host(L, hin, hout, R, count, dtype, ws, ws_bytes, wire=None, group=0):
    import ring_allreduce_reducescatter_gb300 as rr

    rr.lib()
    return L.ring_allreduce_host(ptrs(hin), ptrs(hout), R, count, dtype, dtype if wire is None else wire, group,
                                 ws, ws_bytes, None)


def test_host_pipeline_arguments(L):
    import ring_allreduce_reducescatter_gb300 as rr

    rr.lib()
    R, N = 4, 10_000
    hin, hout = fake(R, N, 4)
    ws = BASE + (1 << 40)
    need = L.ring_allreduce_host_workspace(R, 256, F32)
    assert need == 3 * R * 256 * 4
    assert L.ring_allreduce_host_workspace(R, 1, F16) == 3 * R * 256 * 2
    assert L.ring_allreduce_host_workspace(0, 256, F32) == 0
    assert L.ring_allreduce_host_workspace(R, 0, F32) == 0
    assert call_host(L, hin, hout, R, N, F32, None, need) == EINVAL          # no workspace
    assert call_host(L, hin, hout, R, N, F32, ws + 8, need) == EINVAL        # not 16-byte aligned
    assert call_host(L, hin, hout, R, N, F32, ws, need - 1) == EINVAL        # no room for 256 elements
    assert call_host(L, hin, hout, R, N, F32, hin[2] + 64, need) == EALIAS   # overlaps a host buffer
    assert call_host(L, hin, [hin[1]] + hout[1:], R, N, F32, ws, need) == EALIAS   # output 0 on input 1
    assert call_host(L, hin, hout, R, N, F16, ws, need, wire=BF16) == EUNSUP
    assert call_host(L, hin, hout, R, 0, F32, ws, need) == OK                # nothing to do
    assert call_host(L, hin, list(hin), R, N, F32, ws, need) not in (EINVAL, EALIAS, EUNSUP)  # in place
    # the copy schedule of ring_allreduce_host_ex: 0 or 1
    L.ring_allreduce_host_ex.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                                         ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    L.ring_allreduce_host_ex.restype = ctypes.c_int
    for mode, want in ((2, EINVAL), (-1, EINVAL)):
        assert L.ring_allreduce_host_ex(ptrs(hin), ptrs(hout), R, N, F32, F32, 0, ws, need, mode, None) == want


def test_algo_arguments(L):
    import ring_allreduce_reducescatter_gb300 as rr

    rr.lib()
    ins, outs = fake(8, 100, 4)
    call_algo = lambda algo, R=8, dt=F32, wire=F32, o=outs: L.ring_allreduce_algo(  # noqa: E731
        ptrs(ins[:R]), ptrs(o[:R]), R, 100, dt, wire, algo, None, None)
    assert call_algo(3) == EINVAL
    assert call_algo(-1) == EINVAL
    assert call_algo(1, R=0) == EINVAL
    assert call_algo(2, dt=F16, wire=BF16) == EUNSUP
    assert call_algo(1, o=[ins[1]] + outs[1:]) == EALIAS
    for algo in (0, 1, 2):  # valid: validation passes and the call then needs a device
        assert call_algo(algo) not in (EINVAL, EALIAS, EUNSUP)


def test_max_ctas_caps_the_grid(L):
    st, ch, grid, _ = plan_dev(L, AR, 8, 1 << 28, F16, cfg=(1, 0, 0, 0, 0))
    assert st == OK and grid == 456
    st, ch, grid, _ = plan_dev(L, AR, 8, 1 << 28, F16)  # the direct path: 16 CTAs of 128 per SM
    assert st == OK and ch["path"] == 3 and ch["threads"] == 128 and grid == 152 * 16
    st, ch, grid, smem = plan_dev(L, AR, 8, 1 << 28, F16, cfg=(0, 0, 0, 0, 0, 40))
    assert st == OK and grid == 40 and ch["max_ctas"] == 40
    # a capped grid gets one CTA per SM with larger tiles
    assert ch["ctas_per_sm"] == 1 and ch["tile_bytes"] == 8192 and ch["stages"] == 3 and smem <= GB300["optin"]
    st, ch, _, smem = plan_dev(L, AR, 16, 1 << 26, F32, cfg=(0, 0, 0, 0, 0, 64))
    assert st == OK and ch["tile_bytes"] == 4096 and smem <= GB300["optin"]
    st, ch, grid, _ = plan_dev(L, AR, 8, 1 << 10, F16, aligned=0, cfg=(0, 0, 0, 0, 0, 3))
    assert st == OK and grid == 3 and ch["path"] == 2
    assert plan_dev(L, AR, 8, 1 << 20, F16, cfg=(0, 0, 0, 0, 0, -1))[0] == EINVAL


def test_direct_path_plans(L):
    DIRECT = 3
    st, ch, grid, smem = plan_dev(L, AR, 8, 1 << 19, F16, cfg=(DIRECT, 0, 0, 0, 0))
    assert st == OK and ch["path"] == DIRECT and smem == 0
    assert ch["threads"] == 128 and grid == min((1 << 19) * 2 // 16 // 128, 152 * 16)
    # the same alignment needs as the bulk path, and at most 256 threads
    assert plan_dev(L, AR, 8, 1 << 19, F16, aligned=0, cfg=(DIRECT, 0, 0, 0, 0))[0] == EUNSUP
    assert plan_dev(L, RS, 8, 8 * 1001, F16, cfg=(DIRECT, 0, 0, 0, 0))[0] == OK  # the shifted kernel
    assert plan_dev(L, AR, 8, 1 << 19, F16, cfg=(DIRECT, 0, 0, 0, 512))[0] == EUNSUP
    assert plan_dev(L, AR, 8, 7, F16, cfg=(DIRECT, 0, 0, 0, 0))[0] == EUNSUP  # under 16 bytes
    st, _, grid, _ = plan_dev(L, AR, 8, 1 << 19, F16, cfg=(DIRECT, 0, 0, 0, 128, 10))
    assert st == OK and grid == 10


def test_direct_path_straddle_cta(L):
    """Chunk boundaries off the 16-byte grid get one extra CTA (within a cap,
    the cap's last CTA; a one-CTA cap folds them in the main loop)."""
    DIRECT = 3
    N = 6 * 87381  # base 87381 binary16 elements: boundaries fall inside vectors
    blocks = -(-(N * 2 // 16) // 128)
    st, ch, grid, _ = plan_dev(L, AR, 6, N, F16, cfg=(DIRECT, 0, 0, 0, 0))
    assert st == OK and grid == blocks + 1
    for cap in (1, 2, 7):
        st, ch, grid, _ = plan_dev(L, AR, 6, N, F16, cfg=(DIRECT, 0, 0, 0, 0, cap))
        assert st == OK and grid == cap
    # aligned boundaries, ReduceScatter, and the naive order need none
    st, ch, grid, _ = plan_dev(L, AR, 8, 1 << 19, F16, cfg=(DIRECT, 0, 0, 0, 0))
    assert grid == (1 << 19) * 2 // 16 // 128


def test_direct_grid_waves(L):
    """Looping direct grids: ReduceScatter and AllReduce over groups of at most
    three ranks take two whole waves of the resident CTAs (three 256-thread
    CTAs' worth of registers per SM: 6 CTAs of 128 a wave); other AllReduce
    and AllGather launches take sixteen 128-thread CTAs per SM, and so do the
    chunk-by-chunk rows of AllReduce over flat rings of up to four ranks from
    16 MiB per rank."""
    sms, n = GB300["sms"], 1 << 26  # 256 MiB of binary32 per rank
    assert plan_dev(L, RS, 4, n, F32)[2] == sms * 6 * 2
    assert plan_dev(L, RS, 16, n, F32)[2] == sms * 6 * 2
    assert plan_dev(L, AR, 3, 3 << 24, F16, wire=F32)[2] == sms * 2 * 2 * 2  # fp32 accumulators: two CTAs per SM
    # a flat ring of up to four ranks from 16 MiB: the chunk-by-chunk rows, sixteen CTAs per SM
    st, ch, grid, _ = plan_dev(L, AR, 3, 3 << 24, F16)
    assert st == OK and grid == sms * 16 and ch["vectors"] == 2 and ch["ctas_per_sm"] == 3
    # forcing four rows keeps the rows (two 256-thread CTAs' worth of registers);
    # one or three vectors, or a register budget, select the direct kernel
    DIRECT = 3
    st, ch, grid, _ = plan_dev(L, AR, 2, 2 << 23, F16, cfg=(DIRECT, 0, 0, 0, 0, 0, 0, 4))
    assert st == OK and ch["vectors"] == 4 and ch["ctas_per_sm"] == 2 and grid == sms * 16
    for cfg in ((DIRECT, 0, 0, 0, 0, 0, 0, 1), (DIRECT, 0, 0, 0, 0, 0, 0, 3), (DIRECT, 0, 0, 3, 0, 0, 0, 2)):
        st, ch, grid, _ = plan_dev(L, AR, 2, 2 << 23, F16, cfg=cfg)
        # the direct kernel: two whole waves of its resident CTAs (two ranks)
        assert st == OK and ch["vectors"] == (cfg[7] or 2), (cfg, ch)
        assert grid == sms * ch["ctas_per_sm"] * 2 * 2, (cfg, ch, grid)
    assert plan_dev(L, AR, 8, 1 << 26, F32, group=2)[2] == sms * 6 * 2
    assert plan_dev(L, AR, 4, 1 << 27, F16)[2] == sms * 16
    assert plan_dev(L, AR, 8, 1 << 28, F16)[2] == sms * 16
    assert plan_dev(L, AG, 4, n, F32)[2] == sms * 16
    # ReduceScatter from 64 MiB per rank takes two vectors a thread, so R = 8 is
    # not one batch of eight loads (which would keep two CTAs per SM): three
    # CTAs per SM, two waves
    assert plan_dev(L, RS, 8, n, F32)[2] == sms * 6 * 2
    # chunk boundaries off the 16-byte grid: the shifted ReduceScatter takes
    # twelve 128-thread CTAs per SM for up to four ranks and, for more, from 32
    # MiB per rank; sixteen otherwise
    assert plan_dev(L, RS, 8, (64 << 20) // 4 - 8, F32)[2] == sms * 12
    assert plan_dev(L, RS, 8, (16 << 20) // 2 - 8 + 3, F16)[2] == sms * 16
    assert plan_dev(L, RS, 4, (16 << 20) // 2 - 4 + 3, F16)[2] == sms * 12
    assert plan_dev(L, RS, 2, (64 << 20) // 2 + 2, F16)[2] == sms * 12
    st, _, grid, _ = plan_dev(L, RS, 4, (16 << 20) // 2 - 4 + 3, F16, cfg=(0, 0, 0, 0, 256))
    assert st == OK and grid == sms * 6                       # the same share of threads at 256 a CTA
    # ReduceScatter over two ranks from 32 MiB per rank, chunks on the grid:
    # the chunk-by-chunk kernel at four rows (two 256-thread CTAs' worth of
    # registers per SM), twelve CTAs per SM; below 32 MiB the direct kernel
    st, ch, grid, _ = plan_dev(L, RS, 2, 2 * (16 << 20), F16)
    assert st == OK and ch["vectors"] == 4 and ch["ctas_per_sm"] == 2 and grid == sms * 12
    st, ch, grid, _ = plan_dev(L, RS, 2, 2 * (8 << 20), F16)
    assert st == OK and ch["vectors"] == 4 and ch["ctas_per_sm"] == 2 and grid == sms * 12   # 32 MiB
    st, ch, grid, _ = plan_dev(L, RS, 2, 2 * (4 << 20), F16)
    assert st == OK and ch["vectors"] == 2 and ch["ctas_per_sm"] == 3 and grid == sms * 6   # one wave
    st, ch, _, _ = plan_dev(L, RS, 2, 2 * (16 << 20), F16, cfg=(3, 0, 0, 0, 0, 0, 0, 2))  # forced vectors: direct
    assert st == OK and ch["vectors"] == 2 and ch["ctas_per_sm"] == 3
    # AllGather over two ranks below 64 MiB per rank: two waves of two
    # 256-thread CTAs' worth of registers per SM
    assert plan_dev(L, AG, 2, 2 * (8 << 20), F16)[2] == sms * 4 * 2
    assert plan_dev(L, AG, 2, 2 * (256 << 10), F16)[2] == 2 * (256 << 10) * 2 // 16 // 128   # 1 MiB: one vector
    assert plan_dev(L, AG, 2, 2 * (64 << 20), F16)[2] == sms * 16
    assert plan_dev(L, AG, 3, 3 * (8 << 20), F16)[2] == sms * 16
    # a grid that fits under the cap is not changed (five ranks: no one-wave rule)
    assert plan_dev(L, RS, 5, 5 * (1 << 16), F32)[2] == 5 * (1 << 16) * 4 // 16 // 128  # one vector a thread


def test_one_wave_for_small_flat_rings(L):
    """Flat AllReduce under 16 MiB per rank and ReduceScatter under 32 MiB over
    up to four ranks: one wave of resident CTAs (128 threads; two 256-thread CTAs' worth of
    registers per SM up to 8 MiB, three above), one vector a thread when two
    would leave SMs idle, both L2 prefetches; not for AllGather, five or more
    ranks, two-level rings or 32 MiB and up."""
    sms = GB300["sms"]
    MiB = 1 << 20
    def plan(op, R, mib, dt=F16, E=2, **kw):
        st, ch, grid, _ = plan_dev(L, op, R, R * (mib * MiB // E // R // 8 * 8), dt, **kw)
        assert st == OK and ch["path"] == 3, (op, R, mib, ch)
        return ch["vectors"], ch["ctas_per_sm"], grid, ch["prefetch"] - 1
    assert plan(AR, 4, 4, F32, 4) == (2, 2, sms * 4, 3)      # workload 1
    assert plan(RS, 4, 4, F32, 4) == (2, 2, sms * 4, 3)
    assert plan(AR, 2, 8) == (2, 2, sms * 4, 3)
    assert plan(RS, 3, 16) == (2, 3, sms * 6, 3)
    v, occ, grid, pf = plan(AR, 4, 1)                         # 1 MiB: one vector, the grid under a wave
    assert (v, occ, pf) == (1, 2, 3) and grid <= sms * 4
    assert plan(AR, 4, 64)[2] == sms * 6 * 2 or plan(AR, 4, 64)[2] == sms * 16   # the usual rules from 32 MiB
    vecs = 4 * MiB // 16
    assert plan(AG, 4, 4)[0] == 2 and plan(AG, 4, 4)[2] == vecs // 256         # AllGather keeps its grid
    assert plan(AR, 8, 4)[2] == vecs // 128                                     # five or more ranks too
    assert plan(AR, 8, 4, group=4)[2] == vecs // 256                            # two-level rings too


def test_rank_buffers_layout():
    """rank_buffers: R views of one allocation, each 256-byte aligned relative
    to the first, staggered by the requested bytes, never overlapping."""
    import torch

    import ring_allreduce_reducescatter_gb300 as rr

    for dtype, e in ((torch.float32, 4), (torch.float16, 2), (torch.bfloat16, 2)):
        for counts in (7, 65537, [3, 0, 11, 256]):
            R = 4
            for stagger in (0, 256, 2 << 20):
                bufs = rr.rank_buffers(R, counts, dtype, "cpu", stagger_bytes=stagger)
                lens = [counts] * R if isinstance(counts, int) else counts
                assert [b.numel() for b in bufs] == lens
                base = bufs[0].data_ptr()
                ends = []
                for b, n in zip(bufs, lens):
                    if n == 0:
                        continue
                    off = b.data_ptr() - base
                    assert off % 256 == 0
                    assert all(off >= end + stagger for end in ends[-1:])
                    ends.append(off + -(-n * e // 256) * 256)
    with pytest.raises(ValueError):
        rr.rank_buffers(2, 8, torch.float32, "cpu", stagger_bytes=100)
    with pytest.raises(ValueError):
        rr.rank_buffers(3, [1, 2], torch.float32, "cpu")


def test_binding_checks_host_buffer_sizes(L):
    """The host-buffer entry points copy N elements per rank to and from raw
    host addresses, which the C ABI cannot bound, so the binding checks every
    list length and element count before it passes a pointer on."""
    import torch

    import ring_allreduce_reducescatter_gb300 as rr

    R, N = 4, 1000
    hin = [torch.zeros(N) for _ in range(R)]
    cases = [
        (hin, [torch.zeros(N) for _ in range(R - 1)], "host_outs: 3 buffers for 4 ranks"),
        (hin, [torch.zeros(N) for _ in range(R + 1)], "host_outs: 5 buffers for 4 ranks"),
        (hin, [torch.zeros(N) for _ in range(R - 1)] + [torch.zeros(N - 1)], "host_outs[3]: 999 elements"),
        (hin[:2] + [torch.zeros(N + 7)] + hin[3:], [torch.zeros(N) for _ in range(R)], "host_ins[2]: 1007"),
        (hin, [torch.zeros(N) for _ in range(R - 1)] + [torch.zeros(N, dtype=torch.float64)], "host_outs[3]: dtype"),
        (hin, [torch.zeros(N) for _ in range(R - 1)] + [torch.zeros(2 * N)[::2]], "host_outs[3]: every buffer"),
        ([], [], "host_ins: need at least one rank"),
    ]
    for ins, outs, msg in cases:
        with pytest.raises(ValueError, match=re.escape(msg)):
            rr.allreduce_host_static(ins, outs)
        with pytest.raises(ValueError, match=re.escape(msg)):
            rr.allreduce_host(ins, host_outs=outs, workspace=torch.empty(16, dtype=torch.uint8))


def test_forced_vectors_and_register_budget(L):
    """`vectors` and, on the direct path, `ctas_per_sm` select a kernel; only
    kernels the library builds are accepted, and the plan reports the choice."""
    D = 3  # RR_PATH_DIRECT
    N = 1 << 24
    built = {AR: {(1, 2), (1, 3), (2, 2), (2, 3), (3, 2), (4, 2)}, RS: {(1, 2), (1, 3), (2, 2), (2, 3), (3, 2), (4, 2)},
             AG: {(1, 2), (2, 2), (4, 2)}}
    for op, ok in built.items():
        for u in (1, 2, 3, 4):
            for occ in (2, 3):
                st, ch, grid, _ = plan_dev(L, op, 8, N, F32, cfg=(D, 0, 0, occ, 0, 0, 0, u))
                if (u, occ) in ok:
                    assert st == OK and ch["vectors"] == u and ch["ctas_per_sm"] == occ, (op, u, occ, ch)
                else:
                    assert st == EUNSUP, (op, u, occ, st)
    # binary32 accumulation of 16-bit storage: one or two vectors, two CTAs per SM
    for u, occ, want in ((1, 2, OK), (2, 2, OK), (2, 3, EUNSUP), (3, 2, EUNSUP)):
        assert plan_dev(L, AR, 8, N, F16, wire=F32, cfg=(D, 0, 0, occ, 0, 0, 0, u))[0] == want
    # shifted kernels (chunk boundaries off the 16-byte grid): rows per warp,
    # their register budget fixed by the row count
    Ns = 4 * (8 * 1000 + 1)
    for op, rows in ((RS, (1, 2, 3, 4)), (AG, (1, 2, 4))):
        for u in (1, 2, 3, 4):
            st, ch, _, _ = plan_dev(L, op, 4, Ns, F16, cfg=(D, 0, 0, 0, 0, 0, 0, u))
            if u in rows:
                assert st == OK and ch["vectors"] == u and ch["ctas_per_sm"] == (2 if u >= 3 else 3)
            else:
                assert st == EUNSUP
    assert plan_dev(L, RS, 4, Ns, F16, cfg=(D, 0, 0, 2, 0, 0, 0, 1))[0] == EUNSUP  # one row: three CTAs only
    assert plan_dev(L, RS, 4, Ns, F16, cfg=(0, 0, 0, 2, 0, 0, 0, 1))[0] == OK      # ignored on the automatic path
    # out-of-range values are argument errors
    assert plan_dev(L, AR, 8, N, F32, cfg=(0, 0, 0, 0, 0, 0, 0, 5))[0] == EINVAL
    assert plan_dev(L, AR, 8, N, F32, cfg=(0, 0, 0, 0, 0, 0, 0, -1))[0] == EINVAL
    assert plan_dev(L, AR, 8, N, F32, cfg=(0, 0, 0, 0, 0, 0, 0, 0, 2))[0] == EINVAL


def test_planner_vectors_for_few_ranks(L):
    """The measured choices of vectors (rows) a thread: ReduceScatter over three
    ranks two vectors at three CTAs per SM; AllGather one vector (the L2
    prefetch keeps its loads in flight), two over two ranks below 64 MiB per
    rank from 4 MiB, two over up to five ranks from 4 to 16 MiB; the shifted
    ReduceScatter 2 rows, but 4 for two ranks from 8 MiB per rank, 1 for four
    or more ranks below 8 MiB and 4 for eight or more from 128 MiB."""
    st, ch, _, _ = plan_dev(L, RS, 3, 3 * (1 << 22), F32)
    assert st == OK and ch["path"] == 3 and ch["vectors"] == 2 and ch["ctas_per_sm"] == 3
    # (R, N / R, vectors, register budget): binary32, so N / R = 2^18 is 4 MiB
    # per rank for R = 4; from 12 MiB per rank (two ranks: 64 MiB) the rows of
    # the chunk-by-chunk kernel (two rows at three CTAs per SM, four rows at
    # two for eight or more ranks from 64 MiB)
    for R, n, vectors, occ in ((2, 1 << 22, 2, 2), (2, 1 << 24, 2, 3), (2, 1 << 18, 1, 2), (3, 1 << 20, 2, 3),
                               (4, 1 << 19, 2, 2), (4, 1 << 18, 2, 2), (5, 1 << 19, 2, 2), (5, 1 << 22, 2, 3),
                               (8, 1 << 17, 1, 2), (4, 1 << 17, 1, 2), (4, 1 << 20, 2, 3), (8, 1 << 21, 4, 2),
                               (16, 1 << 18, 2, 3)):
        st, ch, _, _ = plan_dev(L, AG, R, R * n, F32)
        assert st == OK and ch["path"] == 3 and ch["vectors"] == vectors and ch["ctas_per_sm"] == occ, (R, n, ch)
    # (R, N / (8 R), rows): binary16, N = R (8 n + 3), so 8 n + 3 elements a chunk
    for R, n, rows in ((2, 100_000, 2), (2, 1_000_000, 4), (3, 100_000, 2), (3, 2_000_000, 2), (4, 100_000, 1),
                       (4, 1_000_000, 2), (5, 100_000, 1), (8, 100_000, 2), (8, 1_000_000, 2), (8, 10_000_000, 4),
                       (16, 100_000, 2), (16, 10_000, 1)):
        st, ch, _, _ = plan_dev(L, RS, R, R * (8 * n + 3), F16)
        assert st == OK and ch["path"] == 3 and ch["vectors"] == rows, (R, ch)
    # the shifted AllGather: two rows for up to four ranks; for more, one
    # vector a thread below 12 MiB per rank, else two rows (four for eight or
    # more ranks from 64 MiB)
    for R, n, vectors in ((2, 100_000, 2), (3, 100_000, 2), (4, 100_000, 2), (5, 100_000, 1), (8, 50_000, 1),
                          (8, 100_000, 2),
                          (5, 1_000_000, 2), (8, 1_000_000, 4), (16, 200_000, 2), (16, 2_000_000, 4)):
        st, ch, _, _ = plan_dev(L, AG, R, R * (8 * n + 3), F16)
        assert st == OK and ch["path"] == 3 and ch["vectors"] == vectors, (R, n, ch)


def test_beside_compute_caps_the_grid(L):
    """beside_compute: the grid takes RR_BESIDE_COMPUTE_SM_EIGHTHS eighths of
    the SMs, one tile pipeline each; an explicit max_ctas still wins."""
    with open(HEADER) as f:
        eighths = int(re.search(r"#define RR_BESIDE_COMPUTE_SM_EIGHTHS (\d+)", f.read()).group(1))
    want = GB300["sms"] * eighths // 8
    st, ch, grid, smem = plan_dev(L, AR, 8, 1 << 26, F16, cfg=(0, 0, 0, 0, 0, 0, 0, 0, 1))
    assert st == OK and grid == want and ch["path"] == 1 and ch["ctas_per_sm"] == 1 and ch["beside_compute"] == 1
    st, ch, grid, _ = plan_dev(L, AR, 8, 1 << 26, F16, cfg=(0, 0, 0, 0, 0, 40, 0, 0, 1))
    assert st == OK and grid == 40
    st, ch, grid, _ = plan_dev(L, AR, 8, 1 << 26, F16)
    assert st == OK and ch["beside_compute"] == 0 and grid == GB300["sms"] * 16


def test_planner_prefetch_policy(L):
    """L2 prefetch by size and ranks: before the launch wait below 64 MiB per
    rank or for up to four ranks a group; one iteration ahead for two ranks,
    AllGather, ReduceScatter over three ranks, and 8-64 MiB messages other
    than ReduceScatter over five or more ranks; never on the halving-doubling
    kernels; the shifted AllGather both, the shifted ReduceScatter the first
    item over three to five ranks below 32 MiB per rank, else none; the
    AllReduce rows the first item below 24 MiB, else none (prefetch reported
    as 1 + the bits)."""
    MiB = 1 << 20
    def pf(op, R, mib, dt=F16, E=2, **kw):
        st, ch, _, _ = plan_dev(L, op, R, R * (mib * MiB // E // R // 8 * 8), dt, **kw)
        assert st == OK and ch["path"] == 3, (op, R, mib, ch)
        return ch["prefetch"] - 1
    HEAD, AHEAD = 1, 2
    assert pf(AR, 8, 1) == HEAD
    assert pf(AR, 8, 16) == HEAD | AHEAD
    assert pf(AR, 8, 256) == 0
    assert pf(AR, 4, 256, F16, 2, wire=F32) == HEAD          # fp32 accumulators: the direct kernel
    assert pf(AR, 2, 256, F16, 2, wire=F32) == HEAD | AHEAD
    assert pf(AR, 4, 256) == 0                               # the chunk-by-chunk rows: the first item
    assert pf(AR, 2, 16) == HEAD                             # below 24 MiB only
    assert pf(RS, 8, 16) == HEAD
    assert pf(RS, 3, 256) == HEAD | AHEAD
    assert pf(AG, 8, 256) == HEAD | AHEAD  # the chunk-by-chunk rows from 16 MiB: both
    assert pf(AG, 8, 4) == HEAD | AHEAD
    assert pf(AG, 2, 128) == HEAD | AHEAD
    assert pf(AR, 4, 4, F32, 4) == HEAD | AHEAD  # a small flat ring of four: one wave, both
    assert pf(AR, 16, 64, group=8) == 0
    st, ch, _, _ = plan_dev(L, RS, 8, 8 * 1001, F16)  # shifted ReduceScatter: none
    assert st == OK and ch["prefetch"] == 1
    for R, n, bits in ((2, 100_000, 0), (3, 100_000, HEAD), (5, 100_000, HEAD), (4, 3_000_000, 0)):
        st, ch, _, _ = plan_dev(L, RS, R, R * (8 * n + 3), F16)
        assert st == OK and ch["prefetch"] == 1 + bits, (R, n, ch)
    st, ch, _, _ = plan_dev(L, AG, 8, 8 * 1001, F16)  # shifted AllGather: both
    assert st == OK and ch["prefetch"] == 1 + (HEAD | AHEAD)


def test_planner_matches_the_measured_path_table(L):
    """The planner's choice between the tile pipeline and the direct path is
    within 5 % of the faster one at every point of the committed sweep
    (profiles/path_choice_sweep_f16.md, written by bench.py --path-sweep
    --sweep-table on a GB300: AllReduce, ReduceScatter and AllGather over 2-32
    ranks at 1-256 MiB per rank, binary16)."""
    path = os.path.join(ROOT, "profiles", "path_choice_sweep_f16.md")
    rows = []
    with open(path) as f:
        for line in f:
            cells = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cells) == 9 and cells[0] in ("allreduce", "reduce_scatter", "allgather"):
                rows.append(cells)
    assert len(rows) >= 100
    ops = {"allreduce": AR, "reduce_scatter": RS, "allgather": AG}
    names = {1: "bulk", 3: "direct"}
    for op, R, count, _, off, bulk, direct, _, _ in rows:
        st, ch, _, _ = plan_dev(L, ops[op], int(R), int(count), F16)
        assert st == OK and ch["path"] in names, (op, R, count, ch)
        t = {"bulk": float(bulk) if bulk != "-" else None, "direct": float(direct)}
        best = min(v for v in t.values() if v is not None)
        mine = t[names[ch["path"]]]
        assert mine is not None and mine <= 1.05 * best, (op, R, count, names[ch["path"]], t)
