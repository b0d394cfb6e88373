"""GPU parity: libringred's CUDA kernels against the CPU oracle, bit for bit.

Every case runs through the C ABI (the Python binding only marshals) and is
compared element by element with the oracle's literal ring simulation, or, at
the full workload sizes, on sampled elements with the oracle's closed form
plus size-independent properties, and then on every element against the
oracle's closed form evaluated on all host cores.  The bar is bit-exact for
every format: both sides follow the same accumulation order and rounding.
"""
import collections
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
PAIRS = [(torch.float32, None), (torch.float16, None), (torch.bfloat16, None), (torch.float32, "bf16"),
         (torch.float32, "f16"), (torch.float16, "f32"), (torch.bfloat16, "f32")]


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import ring_allreduce_reducescatter_gb300 as mod

    torch.cuda.set_device(0)
    return mod


@pytest.fixture(autouse=True)
def device_status_stays_clear(request):
    """After every test: no kernel recorded a bounded-wait timeout or (in the
    debug build) an access outside its buffer."""
    yield
    if "rr" in request.fixturenames:
        assert request.getfixturevalue("rr").device_status() == 0, "a kernel set the device status word"


@pytest.fixture(scope="module")
def wl():
    from ring_allreduce_reducescatter_gb300 import workloads

    return workloads


def host(t):
    """Tensor -> numpy array in the oracle's element convention."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def assert_same(got, want, what):
    g, w = bits(got), bits(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{what}: {bad.size} of {g.size} elements differ, first at {int(bad[0])}: "
                             f"got {int(g[bad[0]]):#x} want {int(w[bad[0]]):#x}")


def gen(R, N, dtype, seed, dev="cuda", scale=1.0, lengths=None):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    xs = []
    for r in range(R):
        n = N if lengths is None else lengths[r]
        x = torch.randn(n, generator=g, device=dev, dtype=torch.float32) * scale
        # sprinkle exact ties and cancellations
        if n:
            k = torch.randint(0, n, (max(1, n // 8),), generator=g, device=dev)
            v = torch.tensor([1.0, -1.0, 2.0 ** -11, 2.0 ** -24, 2.0 ** -8, 0.0], device=dev)
            x[k] = v[torch.randint(0, v.numel(), (k.numel(),), generator=g, device=dev)]
        xs.append(x.to(dtype))
    return xs


def cfg_of(rr, path=0, tile=0, stages=0, ctas=0, threads=0):
    return rr.LaunchCfg(path, tile, stages, ctas, threads)


def direct_ok(N, R, E, op="ar"):
    """The direct path's condition: at least one 16-byte vector (chunk offsets
    off the 16-byte grid take its shifted ReduceScatter / AllGather kernel)."""
    return N * E >= 16


def run_ar(rr, xs, wire=None, group=0, cfg=None, inplace=False):
    if inplace:
        outs = [x.clone() for x in xs]
        rr.collective(rr.OP_ALLREDUCE, outs, outs, xs[0].numel(), wire, group, None, cfg)
        return outs
    outs = [torch.empty_like(x) for x in xs]
    rr.collective(rr.OP_ALLREDUCE, xs, outs, xs[0].numel(), wire, group, None, cfg)
    return outs


def check_ar(rr, xs, wire=None, group=0, cfg=None, inplace=False, what=""):
    outs = run_ar(rr, xs, wire, group, cfg, inplace)
    torch.cuda.synchronize()
    dt = NAME[xs[0].dtype]
    ref = oracle.allreduce([host(x) for x in xs], dt, wire, group)
    assert ref.status == oracle.OK
    for r in range(len(xs)):
        assert_same(host(outs[r]), ref.outs[r], f"{what} rank {r}")


def check_rs(rr, xs, wire=None, cfg=None, what=""):
    R, N = len(xs), xs[0].numel()
    outs = [torch.empty(rr.chunk_count(N, R, r), dtype=xs[0].dtype, device=xs[0].device) for r in range(R)]
    rr.collective(rr.OP_REDUCE_SCATTER, xs, outs, N, wire, 0, None, cfg)
    torch.cuda.synchronize()
    ref = oracle.reduce_scatter([host(x) for x in xs], NAME[xs[0].dtype], wire)
    assert ref.status == oracle.OK
    for r in range(R):
        assert_same(host(outs[r]), ref.outs[r], f"{what} rank {r}")


def check_ag(rr, chunks, N, cfg=None, what=""):
    R = len(chunks)
    outs = [torch.empty(N, dtype=chunks[0].dtype, device="cuda") for _ in range(R)]
    rr.collective(rr.OP_ALLGATHER, chunks, outs, N, None, 0, None, cfg)
    torch.cuda.synchronize()
    ref = oracle.allgather([host(c) for c in chunks], N, NAME[chunks[0].dtype])
    assert ref.status == oracle.OK
    for r in range(R):
        assert_same(host(outs[r]), ref.outs[r], f"{what} rank {r}")


def counts_for(R):
    c = {0, 1, 2, R - 1, R, R + 1, 2 * R + 3, 255, 4095, 4096, 4097, 65535, 65536, 65537, 100_003}
    return sorted(x for x in c if x >= 0)


# --------------------------------------------------------------------------
# edge grid: ranks x counts x formats x launch paths
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 7, 8, 16])
def test_allreduce_edge_grid(rr, dtype, wire, R):
    seed = 100 * R + 7
    for N in counts_for(R):
        xs = gen(R, N, dtype, seed + N)
        tag = f"AR {NAME[dtype]}/{wire} R={R} N={N}"
        check_ar(rr, xs, wire, what=tag + " auto")
        check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_SIMPLE), what=tag + " simple")
        if N * xs[0].element_size() >= 16:
            # tiny tiles: tiles straddle many chunks, vectors straddle chunk boundaries
            check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_BULK, tile=64, stages=3), what=tag + " bulk64")
            check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_BULK, tile=1024, stages=8, ctas=1,
                                               threads=128), what=tag + " bulk1k")
            check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag + " direct")
    xs = gen(R, 65537, dtype, seed)
    check_ar(rr, xs, wire, inplace=True, what=f"AR in place R={R}")
    check_ar(rr, xs, wire, inplace=True, cfg=cfg_of(rr, path=rr.PATH_DIRECT, threads=128),
             what=f"AR in place direct R={R}")


@pytest.mark.parametrize("dtype,wire", [(torch.float32, None), (torch.float16, None), (torch.float32, "bf16"),
                                        (torch.bfloat16, "f32")], ids=lambda v: str(v))
def test_maximum_rank_counts(rr, dtype, wire):
    """The largest rank counts (up to RR_MAX_RANKS = 64): flat and two-level
    AllReduce, ReduceScatter and AllGather on every path."""
    for R in (33, 64):
        for N in (1, R - 1, R, R + 1, 4097, 64 * 1031 + 5):
            xs = gen(R, N, dtype, 7 * R + N)
            tag = f"max R={R} {NAME[dtype]}/{wire} N={N}"
            check_ar(rr, xs, wire, what=tag)
            check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_SIMPLE), what=tag + " simple")
            if N * xs[0].element_size() >= 16:
                check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag + " direct")
                check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_BULK), what=tag + " bulk")
            if R == 64 and N > R:
                check_ar(rr, xs, wire, group=8, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag + " 8x8")
                check_ar(rr, xs, wire, group=16, what=tag + " 4x16")
    R = 64
    N = R * 2048
    xs = gen(R, N, dtype, 77)
    check_rs(rr, xs, wire, what="max RS")
    check_rs(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_BULK), what="max RS bulk")
    if wire is None:
        lens = [oracle.chunk_len(N + 13, R, c) for c in range(R)]
        chunks = gen(R, 0, dtype, 78, lengths=lens)
        check_ag(rr, chunks, N + 13, what="max AG")


@pytest.mark.parametrize("G,L", [(2, 8), (2, 2), (3, 4), (4, 1), (2, 4), (8, 2)])
@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_two_level_grid(rr, G, L, dtype, wire):
    R = G * L
    for N in (1, L - 1, L + 1, 4095, 65537, 100_003):
        if N < 1:
            continue
        xs = gen(R, N, dtype, 31 * R + N)
        tag = f"2lvl {G}x{L} {NAME[dtype]}/{wire} N={N}"
        check_ar(rr, xs, wire, group=L, what=tag)
        check_ar(rr, xs, wire, group=L, cfg=cfg_of(rr, path=rr.PATH_SIMPLE), what=tag + " simple")
        if N * xs[0].element_size() >= 16:
            check_ar(rr, xs, wire, group=L, cfg=cfg_of(rr, path=rr.PATH_BULK, tile=128), what=tag + " bulk128")
            check_ar(rr, xs, wire, group=L, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag + " direct")


@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
def test_reduce_scatter_grid(rr, dtype, wire, R):
    for N in counts_for(R) + [R * 1024, R * 4096 + 8 * R]:
        xs = gen(R, N, dtype, 17 * R + N)
        tag = f"RS {NAME[dtype]}/{wire} R={R} N={N}"
        check_rs(rr, xs, wire, what=tag)
        check_rs(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_SIMPLE), what=tag + " simple")
        if direct_ok(N, R, xs[0].element_size(), "rs"):
            check_rs(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag + " direct")


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16], ids=str)
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
def test_allgather_grid(rr, dtype, R):
    for N in counts_for(R) + [R * 1024, R * 4096 + 8 * R]:
        lens = [oracle.chunk_len(N, R, c) for c in range(R)]
        chunks = gen(R, 0, dtype, 23 * R + N, lengths=lens)
        tag = f"AG {NAME[dtype]} R={R} N={N}"
        check_ag(rr, chunks, N, what=tag)
        check_ag(rr, chunks, N, cfg=cfg_of(rr, path=rr.PATH_SIMPLE), what=tag + " simple")
        if direct_ok(N, R, chunks[-1].element_size(), "ag"):
            check_ag(rr, chunks, N, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag + " direct")


@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_shifted_reduce_scatter_and_allgather(rr, dtype, wire):
    """Chunk boundaries at every offset off the 16-byte grid: the direct path
    builds each vector from two aligned loads.  Chunk lengths from below one
    vector to several grid strides, the last vectors near the buffer ends."""
    E = torch.tensor([], dtype=dtype).element_size()
    V = 16 // E
    for R in (2, 3, 5, 8, 24):
        for base in [V * k + j for k in (0, 1, 37) for j in range(1, V)] + [V * 20011 + 1, V * 20011 + V - 1]:
            N = R * base + (R // 2)
            xs = gen(R, N, dtype, 13 * R + base)
            tag = f"shifted {NAME[dtype]}/{wire} R={R} base={base}"
            cfg = cfg_of(rr, path=rr.PATH_DIRECT) if direct_ok(N, R, E) else None  # under 16 bytes: simple
            check_rs(rr, xs, wire, cfg=cfg, what="RS " + tag)
            if wire is None:
                lens = [oracle.chunk_len(N, R, c) for c in range(R)]
                chunks = gen(R, 0, dtype, 17 * R + base, lengths=lens)
                check_ag(rr, chunks, N, cfg=cfg, what="AG " + tag)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16], ids=lambda v: str(v))
def test_shifted_allgather_rows_many_ranks(rr, dtype):
    """AllGather over five and eight ranks from 16 MiB per rank with chunk
    boundaries off the 16-byte grid: the shifted kernel in rows of 32 vectors,
    each row count the library builds.  Every output is the chunks joined, bit
    for bit."""
    E = torch.tensor([], dtype=dtype).element_size()
    V = 16 // E
    iv = torch.int16 if E == 2 else torch.int32
    for R in (5, 8):
        base = (16 << 20) // (E * R) // V * V + 1  # off the grid; R * base * E >= 16 MiB
        N = R * base + (R - 2)
        lens = [rr.chunk_count(N, R, c) for c in range(R)]
        chunks = gen(R, 0, dtype, 29 * R + E, lengths=lens)
        want = torch.cat(chunks).view(iv)
        for rows in (0, 1, 2, 4):  # 0: the planner's choice
            cfg = rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 0, 0, 0, rows) if rows else None
            outs = [torch.full((N,), float("nan"), dtype=dtype, device="cuda") for _ in range(R)]
            rr.collective(rr.OP_ALLGATHER, chunks, outs, N, None, 0, None, cfg)
            torch.cuda.synchronize()
            for r in range(R):
                assert torch.equal(outs[r].view(iv), want), f"AG rows {NAME[dtype]} R={R} rows={rows} rank {r}"
            del outs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=lambda v: str(v))
def test_allgather_rows_aligned_chunks(rr, dtype):
    """AllGather from 16 MiB per rank (two ranks: 64 MiB) with chunk boundaries
    on the 16-byte grid: the planner takes the chunk-by-chunk rows, which then
    shift by nothing; a ragged last chunk.  Every output is the chunks joined,
    bit for bit."""
    E = torch.tensor([], dtype=dtype).element_size()
    V = 16 // E
    iv = torch.int16 if E == 2 else torch.int32
    for R, mib in ((2, 64), (3, 16), (8, 16)):
        base = -(-(mib << 20) // (E * R * V)) * V  # a multiple of V; R * base * E >= mib MiB
        N = R * base + (R - 1)
        lens = [rr.chunk_count(N, R, c) for c in range(R)]
        chunks = gen(R, 0, dtype, 31 * R + E, lengths=lens)
        outs = [torch.full((N,), float("nan"), dtype=dtype, device="cuda") for _ in range(R)]
        plan = rr.plan(rr.OP_ALLGATHER, chunks, outs, N)
        assert plan["path"] == rr.PATH_DIRECT and plan["vectors"] == 2 and plan["ctas_per_sm"] == 3, (R, plan)
        rr.collective(rr.OP_ALLGATHER, chunks, outs, N)
        torch.cuda.synchronize()
        want = torch.cat(chunks).view(iv)
        for r in range(R):
            assert torch.equal(outs[r].view(iv), want), f"AG rows aligned {NAME[dtype]} R={R} rank {r}"
        del outs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("algo", ["hd", "naive"])
def test_allgather_equals_every_schedule(rr, algo):
    """On one GPU the AllGather is a copy: ring_allgather's outputs equal the
    oracle's tree (recursive doubling) and gather-broadcast schedules bit for bit."""
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        for R in (3, 5, 8, 12):
            N = R * 4099 + 5
            lens = [oracle.chunk_len(N, R, c) for c in range(R)]
            chunks = gen(R, 0, dtype, 71 * R, lengths=lens)
            outs = rr.allgather(chunks, N)
            torch.cuda.synchronize()
            ref = oracle.allgather_algo([host(c) for c in chunks], N, NAME[dtype], algo)
            assert ref.status == oracle.OK
            for r in range(R):
                assert_same(host(outs[r]), ref.outs[r], f"AG vs {algo} {NAME[dtype]} R={R} rank {r}")


def test_aligned_paths_are_chosen_when_aligned(rr):
    xs = gen(8, 1 << 20, torch.float16, 5)
    outs = [torch.empty_like(x) for x in xs]
    assert rr.plan(rr.OP_ALLREDUCE, xs, outs, 1 << 20)["path"] in (rr.PATH_BULK, rr.PATH_DIRECT)
    # chunk boundaries off the 16-byte grid: ReduceScatter takes the direct
    # path's shifted kernel; the tile pipeline refuses
    N = 8 * 1001
    xs = gen(8, N, torch.float16, 5)
    rs = [torch.empty(N // 8, dtype=torch.float16, device="cuda") for _ in range(8)]
    assert rr.plan(rr.OP_REDUCE_SCATTER, xs, rs, N)["path"] == rr.PATH_DIRECT
    check_rs(rr, xs, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what="shifted RS")
    with pytest.raises(rr.RingError) as e:
        rr.collective(rr.OP_REDUCE_SCATTER, xs, rs, N, cfg=cfg_of(rr, path=rr.PATH_BULK))
    assert e.value.status == rr.ERR_UNSUPPORTED


def test_misaligned_buffers(rr):
    # element-aligned but not 16-byte aligned views: the simple path, same bits
    for dtype, wire in PAIRS:
        R, N = 5, 70_001
        bufs = gen(R, N + 3, dtype, 77)
        xs = [b[1 + (r % 3): 1 + (r % 3) + N] for r, b in enumerate(bufs)]
        check_ar(rr, xs, wire, what=f"misaligned {NAME[dtype]}/{wire}")


def test_outputs_do_not_write_outside(rr):
    # guard bands around every output stay untouched (both paths, all ops)
    R, N = 8, 100_003
    for dtype in (torch.float32, torch.float16):
        xs = gen(R, N, dtype, 9)
        pad = 64
        for path in (rr.PATH_AUTO, rr.PATH_SIMPLE):
            big = [torch.full((N + 2 * pad,), 7.0, dtype=dtype, device="cuda") for _ in range(R)]
            outs = [b[pad:pad + N] for b in big]
            rr.collective(rr.OP_ALLREDUCE, xs, outs, N, cfg=cfg_of(rr, path=path))
            torch.cuda.synchronize()
            for b in big:
                assert torch.all(b[:pad] == 7.0) and torch.all(b[pad + N:] == 7.0)
        M = 8 * 4096
        xs = gen(R, M, dtype, 10)
        big = [torch.full((M // 8 + 2 * pad,), 7.0, dtype=dtype, device="cuda") for _ in range(R)]
        outs = [b[pad:pad + M // 8] for b in big]
        rr.collective(rr.OP_REDUCE_SCATTER, xs, outs, M)
        torch.cuda.synchronize()
        for b in big:
            assert torch.all(b[:pad] == 7.0) and torch.all(b[pad + M // 8:] == 7.0)


def test_alias_rejected_on_device_buffers(rr):
    xs = gen(4, 1024, torch.float32, 1)
    big = torch.empty(4096 + 16, device="cuda")
    outs = [big[0:1024], big[512:1536], big[2048:3072], big[3072:4096]]
    with pytest.raises(rr.RingError) as e:
        rr.allreduce(xs, outs=outs)
    assert e.value.status == rr.ERR_ALIAS


def test_bounded_wait_gives_up_and_context_survives(rr):
    import time

    t = time.time()
    st = rr.selftest_bounded_wait(50_000_000)  # 50 ms
    dt = time.time() - t
    assert st == rr.ERR_TIMEOUT
    assert dt >= 0.04
    assert rr.device_status() == 0  # the self test cleared its bit
    xs = gen(4, 4099, torch.float32, 3)
    check_ar(rr, xs, what="after bounded-wait self test")


def test_streams_and_ordering(rr):
    # the call enqueues on the given stream: back-to-back dependent calls on a side stream
    s = torch.cuda.Stream()
    xs = gen(4, 1 << 16, torch.float32, 4)
    with torch.cuda.stream(s):
        a = rr.allreduce(xs, stream=s)
        b = rr.allreduce(a, stream=s)
    s.synchronize()
    ref_a = oracle.allreduce([host(x) for x in xs], "f32")
    ref_b = oracle.allreduce(ref_a.outs, "f32")
    for r in range(4):
        assert_same(host(b[r]), ref_b.outs[r], f"chained rank {r}")


# --------------------------------------------------------------------------
# back-to-back dependent kernels: with programmatic dependent launch a kernel
# may be scheduled while the one before it runs, and must still see its writes
# --------------------------------------------------------------------------

CHAIN_PATHS = {"bulk": 1, "direct": 3, "simple": 2}


def chain_device(rr, xs, cfg, rounds, stream=None):
    """RS -> AG -> in-place AR -> (a torch kernel) -> in-place AR -> RS -> AG ...,
    every step reading what the step before wrote, enqueued with no sync."""
    R, N = len(xs), xs[0].numel()
    lens = [rr.chunk_count(N, R, c) for c in range(R)]
    parts = [torch.empty(n, dtype=xs[0].dtype, device="cuda") for n in lens]
    full = [torch.empty(N, dtype=xs[0].dtype, device="cuda") for _ in range(R)]
    rr.collective(rr.OP_REDUCE_SCATTER, xs, parts, N, None, 0, stream, cfg)
    for _ in range(rounds):
        rr.collective(rr.OP_ALLGATHER, parts, full, N, None, 0, stream, cfg)
        rr.collective(rr.OP_ALLREDUCE, full, full, N, None, 0, stream, cfg)
        full[1].neg_()
        rr.collective(rr.OP_ALLREDUCE, full, full, N, None, 0, stream, cfg)
        rr.collective(rr.OP_REDUCE_SCATTER, full, parts, N, None, 0, stream, cfg)
    rr.collective(rr.OP_ALLGATHER, parts, full, N, None, 0, stream, cfg)
    return full


def chain_oracle(xs, rounds):
    dt = NAME[xs[0].dtype]
    R, N = len(xs), xs[0].numel()
    parts = oracle.reduce_scatter([host(x) for x in xs], dt).outs
    for _ in range(rounds):
        full = oracle.allgather(parts, N, dt).outs
        full = oracle.allreduce(full, dt).outs
        full[1] = -full[1] if dt == "f32" else full[1] ^ np.uint16(0x8000)
        full = oracle.allreduce(full, dt).outs
        parts = oracle.reduce_scatter(full, dt).outs
    return oracle.allgather(parts, N, dt).outs


@pytest.mark.parametrize("early", [1, 2], ids=["early", "ordered"])
@pytest.mark.parametrize("path", list(CHAIN_PATHS))
@pytest.mark.parametrize("N", [16 * 4 * 97, 4 * 65540])
def test_dependent_launch_chain(rr, path, early, N):
    R = 4
    xs = gen(R, N, torch.float32, 21, scale=0.25)
    cfg = rr.LaunchCfg(CHAIN_PATHS[path], 0, 0, 0, 0, 0, early)
    got = chain_device(rr, xs, cfg, rounds=3)
    torch.cuda.synchronize()
    want = chain_oracle(xs, rounds=3)
    for r in range(R):
        assert_same(host(got[r]), want[r], f"{path} early={early} N={N} rank {r}")


@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_direct_occupancy_variants(rr, dtype, wire):
    """Messages large enough that the direct path's threads loop (the
    85-register variant with one and two vectors a thread) and grouped rings
    (the 128-register variant), with ragged chunk boundaries."""
    V = 16 // torch.tensor([], dtype=dtype).element_size()
    for R, group, N in ((3, 0, 3 * (1 << 19) + 5), (5, 0, 5 * 300_001), (9, 0, 9 * 200_003),
                        (8, 4, 8 * 150_001), (16, 0, 16 * 160_001)):
        xs = gen(R, N, dtype, 61 * R + group)
        plan = rr.plan(rr.OP_ALLREDUCE, xs, [torch.empty_like(x) for x in xs], N, wire, group)
        assert plan["path"] == rr.PATH_DIRECT or R == 16, plan
        check_ar(rr, xs, wire, group=group, cfg=cfg_of(rr, path=rr.PATH_DIRECT),
                 what=f"occupancy {NAME[dtype]}/{wire} R={R} group={group} N={N} V={V}")
    for R, N in ((4, 4 * (1 << 19)), (8, 8 * 300_000), (12, 12 * 160_000)):  # two vectors a thread, then one
        xs = gen(R, N, dtype, 67 + R)
        check_rs(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=f"occupancy RS {NAME[dtype]}/{wire} R={R}")


@pytest.mark.parametrize("dtype,wire", [(torch.float32, None), (torch.float16, None), (torch.float32, "bf16"),
                                        (torch.bfloat16, "f32")], ids=lambda v: str(v))
def test_reduce_scatter_two_vectors_large(rr, dtype, wire):
    """ReduceScatter of 64 MiB or more per rank over five and nine ranks: two
    vectors a thread in batches of four ranks (the last batch partial), chunk
    boundaries on the 16-byte grid, a ragged last chunk.  Every output element
    is written; sampled elements (every chunk boundary, both ends, random ones)
    equal the oracle's closed form."""
    E = torch.tensor([], dtype=dtype).element_size()
    V = 16 // E
    for R in (5, 9):
        base = -(-(64 << 20) // (E * R * V)) * V  # a multiple of V elements; R * base * E >= 64 MiB
        N = R * base + (R - 2)  # floor(N / R) = base: the last chunk takes R - 2 more
        xs = gen(R, N, dtype, 71 * R + E)
        parts = [torch.full((rr.chunk_count(N, R, c),), float("nan"), dtype=dtype, device="cuda") for c in range(R)]
        assert rr.plan(rr.OP_REDUCE_SCATTER, xs, parts, N, wire)["path"] == rr.PATH_DIRECT
        rr.collective(rr.OP_REDUCE_SCATTER, xs, parts, N, wire)
        torch.cuda.synchronize()
        what = f"RS two vectors {NAME[dtype]}/{wire} R={R} N={N}"
        for c in range(R):
            assert not torch.isnan(parts[c]).any(), f"{what}: chunk {c} has unwritten elements"
        idx = sample_indices(N, R)
        vals = [host(x[torch.from_numpy(idx).cuda()]) for x in xs]
        want = oracle.fold_gathered(vals, idx.astype(np.uint64), N, NAME[dtype], wire, 0)
        owner = np.minimum(idx // base, R - 1)
        for c in range(R):
            sel = np.flatnonzero(owner == c)
            loc = torch.from_numpy(idx[sel] - c * base).cuda()
            assert_same(host(parts[c][loc]), want[sel], f"{what} chunk {c}")
        del xs, parts
        torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_vectors_over_chunk_boundaries(rr, dtype, wire):
    """Chunk boundaries inside 16-byte vectors: the direct path's extra CTA
    folds those vectors in two ring orders at once (and chunks shorter than a
    vector element by element); every cap of the grid, in place and not."""
    V = 16 // torch.tensor([], dtype=dtype).element_size()
    for R in (3, 5, 6, 7, 9, 12, 24):
        for base in (V * 2500 + 1, V * 2501 + V // 2, V * 999 + V - 1, 3):
            N = R * base + (R - 1)
            xs = gen(R, N, dtype, 53 * R + base)
            tag = f"straddle {NAME[dtype]}/{wire} R={R} base={base}"
            check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag)
            if dtype == torch.float16 and wire is None:
                for cap in (1, 2, 7):
                    check_ar(rr, xs, wire, cfg=rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 0, cap),
                             what=f"{tag} cap={cap}")
                check_ar(rr, xs, wire, cfg=cfg_of(rr, path=rr.PATH_DIRECT), inplace=True, what=tag + " in place")
                check_ar(rr, xs, wire, group=R if R % 3 else 3, cfg=cfg_of(rr, path=rr.PATH_DIRECT),
                         what=tag + " grouped")


@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_staggered_rank_buffers(rr, dtype, wire):
    """Rank vectors laid out by rank_buffers (views of one allocation, odd
    lengths padded to 256 bytes) reduce like separate tensors."""
    R, N = 8, 65537
    src = gen(R, N, dtype, 23)
    ins = rr.rank_buffers(R, N, dtype, "cuda")
    outs = rr.rank_buffers(R, N, dtype, "cuda", stagger_bytes=4096)
    for a, b in zip(ins, src):
        a.copy_(b)
    rr.collective(rr.OP_ALLREDUCE, ins, outs, N, wire, 0, None, None)
    torch.cuda.synchronize()
    ref = oracle.allreduce([host(x) for x in src], NAME[dtype], wire)
    for r in range(R):
        assert_same(host(outs[r]), ref.outs[r], f"staggered rank {r}")


def test_dependent_launch_chain_in_a_graph(rr):
    """The same chain captured in a CUDA graph (programmatic edges) and replayed."""
    R, N = 8, 16 * 8 * 33
    xs = gen(R, N, torch.float16, 22, scale=0.05)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain_device(rr, xs, None, rounds=1, stream=s)  # warm-up outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            got = chain_device(rr, xs, None, rounds=2, stream=s)
    for _ in range(3):
        for r in range(R):
            got[r].fill_(7.0)
        g.replay()
    torch.cuda.synchronize()
    want = chain_oracle(xs, rounds=2)
    for r in range(R):
        assert_same(host(got[r]), want[r], f"graph replay rank {r}")


# --------------------------------------------------------------------------
# the workloads, at full size, in the launch configuration the benchmark uses
# --------------------------------------------------------------------------

def sample_indices(N, L, k=1 << 19, seed=0):
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, N, size=k)]
    base = N // L
    for c in range(1, L):
        b = c * base
        idx.append(np.arange(max(0, b - 24), min(N, b + 24)))
    idx.append(np.arange(0, min(N, 64)))
    idx.append(np.arange(max(0, N - 64), N))
    return np.unique(np.concatenate(idx)).astype(np.int64)


def check_sampled(rr, xs, outs, wire=None, group=0, what=""):
    R, N = len(xs), xs[0].numel()
    L = group or R
    idx = sample_indices(N, L)
    ti = torch.from_numpy(idx).cuda()
    vals = [host(x[ti]) for x in xs]
    want = oracle.fold_gathered(vals, idx.astype(np.uint64), N, NAME[xs[0].dtype], wire, group)
    for r in range(R):
        assert_same(host(outs[r][ti]), want, f"{what} sampled rank {r}")
        if r:
            assert torch.equal(outs[r].view(torch.int16 if outs[r].element_size() == 2 else torch.int32),
                               outs[0].view(torch.int16 if outs[0].element_size() == 2 else torch.int32)), \
                f"{what}: output {r} differs from output 0"


def full_check_workers():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def check_full(rr, xs, outs, wire=None, group=0, algo="ring", what="", piece=1 << 21):
    """Every element of the AllReduce against the oracle's closed form.

    Output 0 is compared element by element with the closed form over the
    whole index range [0, N).  The range is split into disjoint pieces that the
    host's cores evaluate at once: the closed form is element-wise (each
    element's fold depends only on its own chunk), so the split cannot change
    a bit, and ctypes releases the interpreter lock during the oracle call.
    Inputs and output come back from the device one piece at a time, so host
    memory stays bounded.  Every other output in outs must equal output 0 bit
    for bit (compared on the device); a ReduceScatter passes its chunks joined
    as the one output."""
    R, N = len(xs), xs[0].numel()
    dt = NAME[xs[0].dtype]
    workers = full_check_workers()

    def one(a, vals, got):
        idx = np.arange(a, a + got.size, dtype=np.uint64)
        if algo == "ring":
            want = oracle.fold_gathered(vals, idx, N, dt, wire, group)
        else:
            want = oracle.fold_gathered_algo(vals, idx, N, dt, wire, algo)
        g, w = bits(got), bits(want)
        if np.array_equal(g, w):
            return None
        bad = np.flatnonzero(g != w)
        k = int(bad[0])
        return f"{bad.size} of {g.size} elements of [{a}, {a + g.size}) differ, first at {a + k}: " \
               f"got {int(g[k]):#x} want {int(w[k]):#x}"

    failures = []
    with ThreadPoolExecutor(max_workers=workers) as ex:
        pending = collections.deque()
        for a in range(0, N, piece):
            b = min(N, a + piece)
            pending.append(ex.submit(one, a, [host(x[a:b]) for x in xs], host(outs[0][a:b])))
            while len(pending) > workers + 2:
                err = pending.popleft().result()
                if err:
                    failures.append(err)
        while pending:
            err = pending.popleft().result()
            if err:
                failures.append(err)
    assert not failures, f"{what} rank 0: " + "; ".join(failures[:4])
    iv = torch.int16 if outs[0].element_size() == 2 else torch.int32
    for r in range(1, len(outs)):
        assert torch.equal(outs[r].view(iv), outs[0].view(iv)), f"{what}: output {r} differs from output 0"


def big_inputs(R, N, dtype, seed, piece=1 << 28):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    xs = []
    for _ in range(R):
        x = torch.empty(N, dtype=dtype, device="cuda")
        for a in range(0, N, piece):
            b = min(N, a + piece)
            x[a:b].copy_(torch.randn(b - a, generator=g, device="cuda") * 0.01)
        xs.append(x)
    return xs


@pytest.mark.parametrize("R,N", [(2, (1 << 32) + (1 << 20) + 5), (3, (1 << 32) + 7)])
def test_counts_beyond_32_bits(rr, R, N):
    """Rank vectors of more than 2^32 elements (8 GiB of binary16 each): every
    element index and byte offset needs 64 bits.  Each path, sampled against the
    closed form (chunk boundaries, both ends, random elements)."""
    xs = big_inputs(R, N, torch.float16, 81 + R)
    outs = [torch.empty_like(x) for x in xs]
    for path in (rr.PATH_AUTO, rr.PATH_DIRECT, rr.PATH_BULK, rr.PATH_SIMPLE):
        for o in outs:
            o.fill_(float("nan"))
        rr.collective(rr.OP_ALLREDUCE, xs, outs, N, None, 0, None, cfg_of(rr, path=path))
        torch.cuda.synchronize()
        check_sampled(rr, xs, outs, what=f"N=2^32+{N - (1 << 32)} R={R} path={path}")
    del xs, outs
    torch.cuda.empty_cache()


def test_reduce_scatter_beyond_32_bits(rr):
    """ReduceScatter of two 2^32 + 16 element vectors: output chunks start past
    the 8 GiB mark of the inputs."""
    R, N = 2, (1 << 32) + 16
    xs = big_inputs(R, N, torch.float16, 91)
    base = N // R
    outs = [torch.empty(base, dtype=torch.float16, device="cuda") for _ in range(R)]
    idx = np.unique(np.concatenate([np.arange(0, 64), np.arange(base - 64, base),
                                    np.random.default_rng(5).integers(0, base, 1 << 16)])).astype(np.int64)
    for path in (rr.PATH_AUTO, rr.PATH_DIRECT, rr.PATH_BULK):
        rr.collective(rr.OP_REDUCE_SCATTER, xs, outs, N, None, 0, None, cfg_of(rr, path=path))
        torch.cuda.synchronize()
        for c in range(R):
            gi = idx + c * base  # global indices of chunk c's sampled elements
            tg = torch.from_numpy(gi).cuda()
            vals = [host(x[tg]) for x in xs]
            want = oracle.fold_gathered(vals, gi.astype(np.uint64), N, "f16", None, 0)
            assert_same(host(outs[c][torch.from_numpy(idx).cuda()]), want, f"RS 2^32+ path={path} chunk {c}")
    del xs, outs
    torch.cuda.empty_cache()


def test_workload1_full(rr, wl):
    w = wl.config1()
    xs = wl.inputs(w, "cuda")
    check_ar(rr, xs, what="workload 1 AR")
    check_rs(rr, xs, what="workload 1 RS")
    lens = [rr.chunk_count(w.count, w.R, c) for c in range(w.R)]
    chunks = wl.inputs(wl.config1("allgather"), "cuda", lengths=lens)
    check_ag(rr, chunks, w.count, what="workload 1 AG")


@pytest.mark.parametrize("mib", [1, 16])
def test_workload2_full_oracle(rr, wl, mib):
    xs = wl.inputs(wl.config2(mib), "cuda")
    check_ar(rr, xs, what=f"workload 2 {mib} MiB")


@pytest.mark.parametrize("dtype,wire", [(torch.float16, None), (torch.bfloat16, None), (torch.float32, "f16")],
                         ids=lambda v: str(v))
def test_allreduce_rows_few_ranks(rr, dtype, wire):
    """AllReduce over two to four ranks from 16 MiB per rank with chunk
    boundaries on the 16-byte grid and a ragged last chunk: the chunk-by-chunk
    rows (forced two and four rows, and the planner's choice).  Every element
    of every output equals the oracle's closed form."""
    E = torch.tensor([], dtype=dtype).element_size()
    V = 16 // E
    for R in (2, 3, 4):
        base = -(-(16 << 20) // (E * R * V)) * V + 37 * V  # a multiple of V; R * base * E > 16 MiB
        N = R * base + (R - 1) * V + (V - 1)               # the last chunk: R - 1 more vectors and a ragged end
        xs = gen(R, N, dtype, 89 * R + E)
        for rows in (0, 2, 4):
            cfg = rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 0, 0, 0, rows) if rows else None
            outs = [torch.full((N,), float("nan"), dtype=dtype, device="cuda") for _ in range(R)]
            rr.collective(rr.OP_ALLREDUCE, xs, outs, N, wire, 0, None, cfg)
            torch.cuda.synchronize()
            check_full(rr, xs, outs, wire=wire, what=f"AR rows {NAME[dtype]}/{wire} R={R} rows={rows}")
            del outs
        # in place: each vector is read and written by one lane only
        outs = run_ar(rr, xs, wire, inplace=True)
        torch.cuda.synchronize()
        check_full(rr, xs, outs, wire=wire, what=f"AR rows in place {NAME[dtype]}/{wire} R={R}")
        del outs
        del xs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype,wire", [(torch.float16, None), (torch.float32, "bf16")], ids=lambda v: str(v))
def test_reduce_scatter_two_ranks_chunk_by_chunk(rr, dtype, wire):
    """ReduceScatter over two ranks from 32 MiB per rank (here 64 MiB) with chunk
    boundaries on the 16-byte grid: the planner takes the chunk-by-chunk kernel,
    which then shifts by nothing; the last chunk is ragged.  Every output
    element equals the oracle's closed form."""
    E = torch.tensor([], dtype=dtype).element_size()
    base = (32 << 20) // E  # a multiple of the vector: 64 MiB per rank over two chunks
    N = 2 * base + 3
    xs = gen(2, N, dtype, 83 + E)
    parts = [torch.full((rr.chunk_count(N, 2, c),), float("nan"), dtype=dtype, device="cuda") for c in range(2)]
    plan = rr.plan(rr.OP_REDUCE_SCATTER, xs, parts, N, wire)
    assert plan["path"] == rr.PATH_DIRECT and plan["vectors"] == 4 and plan["ctas_per_sm"] == 2, plan
    rr.collective(rr.OP_REDUCE_SCATTER, xs, parts, N, wire)
    torch.cuda.synchronize()
    what = f"RS chunk by chunk {NAME[dtype]}/{wire} N={N}"
    for c in range(2):
        assert not torch.isnan(parts[c]).any(), f"{what}: chunk {c} has unwritten elements"
    check_full(rr, xs, [torch.cat(parts)], wire=wire, what=what)
    del parts, xs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mib", [128, 512])
def test_workload2_full_size(rr, wl, mib):
    """The benchmark's workload in its launch configuration (staggered rank
    buffers), every element of every output."""
    w = wl.config2(mib)
    xs = rr.rank_buffers(w.R, w.count, w.dtype, "cuda")
    for r in range(w.R):
        wl.rank_values(w.wid, r, w.count, w.dtype, w.dist, "cuda", out=xs[r])
    outs = rr.rank_buffers(w.R, w.count, w.dtype, "cuda")
    rr.allreduce(xs, outs=outs)
    torch.cuda.synchronize()
    check_sampled(rr, xs, outs, what=f"workload 2 {mib} MiB")  # quick pre-check
    check_full(rr, xs, outs, what=f"workload 2 {mib} MiB")
    del outs, xs
    torch.cuda.empty_cache()


def test_workload3_full_size(rr, wl):
    w = wl.config3()
    xs = wl.inputs(w, "cuda")
    outs = rr.allreduce(xs, wire="bf16")
    torch.cuda.synchronize()
    check_sampled(rr, xs, outs, wire="bf16", what="workload 3")
    check_full(rr, xs, outs, wire="bf16", what="workload 3")
    del outs, xs
    torch.cuda.empty_cache()


def test_workload3_shape_full_oracle(rr):
    # the same formats and an uneven prime-like count, small enough for the literal oracle
    N = 5_000_011
    g = torch.Generator(device="cuda")
    g.manual_seed(3000)
    xs = [torch.randn(N, generator=g, device="cuda") for _ in range(8)]
    check_ar(rr, xs, "bf16", what="workload 3 shape")


def test_workload4_full_oracle(rr, wl):
    w = wl.config4()
    xs = wl.inputs(w, "cuda")
    check_ar(rr, xs, group=w.group_size, what="workload 4")


@pytest.mark.parametrize("bucket", [0, 48])
def test_workload5_bucket_full_size(rr, wl, bucket):
    w = wl.config5(bucket)
    xs = wl.inputs(w, "cuda", bucket=bucket)
    outs = rr.allreduce(xs)
    torch.cuda.synchronize()
    check_sampled(rr, xs, outs, what=f"workload 5 bucket {bucket}")
    check_full(rr, xs, outs, what=f"workload 5 bucket {bucket}")
    del outs, xs
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------
# ranges (chunked AllReduce) and the host-buffer pipeline
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,wire,R,L", [(torch.float16, None, 8, 0), (torch.float32, "bf16", 8, 0),
                                            (torch.float32, None, 16, 8), (torch.bfloat16, None, 3, 0),
                                            (torch.float32, "f16", 5, 0)])
def test_ranges_concatenate_to_the_allreduce(rr, dtype, wire, R, L):
    N = 200_003
    xs = gen(R, N, dtype, 41 + R)
    Lc = L or R
    base = N // Lc
    rng = np.random.default_rng(R)
    # split points: chunk boundaries and their neighbours, 16-byte multiples, odd places
    cuts = {0, N, 1, N - 1, 4096, 65536, 12_345}
    for c in range(1, Lc):
        cuts |= {c * base - 1, c * base, c * base + 3}
    cuts |= set(int(v) for v in rng.integers(0, N, 12))
    cuts = sorted(v for v in cuts if 0 <= v <= N)
    outs = [torch.full_like(x, 0) for x in xs]
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b > a:
            rr.allreduce_range([x[a:b] for x in xs], [o[a:b] for o in outs], N, a, wire, L)
    torch.cuda.synchronize()
    ref = oracle.allreduce([host(x) for x in xs], NAME[dtype], wire, L)
    for r in range(R):
        assert_same(host(outs[r]), ref.outs[r], f"ranges {NAME[dtype]}/{wire} R={R} L={L} rank {r}")
    # in place, a range at a time
    ys = [x.clone() for x in xs]
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b > a:
            rr.allreduce_range([y[a:b] for y in ys], [y[a:b] for y in ys], N, a, wire, L)
    torch.cuda.synchronize()
    for r in range(R):
        assert_same(host(ys[r]), ref.outs[r], f"ranges in place rank {r}")


@pytest.mark.parametrize("dtype,wire,R,L,N,piece", [
    (torch.float16, None, 8, 0, 1_000_003, 4096),      # 245 pieces, ragged last piece
    (torch.float32, "bf16", 8, 0, 300_001, 65536),
    (torch.float32, None, 16, 8, 100_000, 1000),       # piece rounds up to 1024
    (torch.bfloat16, None, 4, 0, 4_097, 1 << 20),      # one piece
    (torch.float32, None, 1, 0, 12_345, 256),
])
def test_host_pipeline_parity(rr, dtype, wire, R, L, N, piece):
    g = torch.Generator()
    g.manual_seed(N + R)
    for pinned in (True, False):
        hin = [torch.randn(N, generator=g).to(dtype) for _ in range(R)]
        if pinned:
            hin = [t.pin_memory() for t in hin]
        ws = torch.empty(rr.host_workspace_bytes(R, piece, dtype), dtype=torch.uint8, device="cuda")
        hout = rr.allreduce_host(hin, workspace=ws, wire=wire, group_size=L)
        torch.cuda.current_stream().synchronize()
        ref = oracle.allreduce([host(t) for t in hin], NAME[dtype], wire, L)
        for r in range(R):
            assert_same(host(hout[r]), ref.outs[r], f"host pipeline pinned={pinned} rank {r}")
        # a second call on the same workspace, in place on the host buffers
        hin2 = [t * 0.5 for t in hin]
        ref2 = oracle.allreduce([host(t) for t in hin2], NAME[dtype], wire, L)
        if pinned:
            hin2 = [t.pin_memory() for t in hin2]
        rr.allreduce_host(hin2, host_outs=hin2, workspace=ws, wire=wire, group_size=L)
        torch.cuda.current_stream().synchronize()
        for r in range(R):
            assert_same(host(hin2[r]), ref2.outs[r], f"host pipeline second call rank {r}")
        # the one-direction-at-a-time copy schedule, twice on the same workspace
        for call in range(2):
            hout3 = rr.allreduce_host(hin, workspace=ws, wire=wire, group_size=L, copy_mode=rr.HOST_COPIES_ONE_WAY)
            torch.cuda.current_stream().synchronize()
            for r in range(R):
                assert_same(host(hout3[r]), ref.outs[r], f"host pipeline one-way call {call} pinned={pinned} rank {r}")


def test_host_pipeline_orders_after_prior_stream_work(rr):
    # the copies must wait for work already enqueued on the stream (here: a
    # device-to-host copy that fills the host inputs)
    R, N = 4, 1 << 20
    dev_src = gen(R, N, torch.float32, 5)
    hin = [torch.empty(N, dtype=torch.float32).pin_memory() for _ in range(R)]
    s = torch.cuda.current_stream()
    torch.cuda._sleep(20_000_000)  # keep the stream busy so the copies below are still queued
    for r in range(R):
        hin[r].copy_(dev_src[r], non_blocking=True)
    hout = rr.allreduce_host(hin, piece_count=65536)
    s.synchronize()
    ref = oracle.allreduce([host(x) for x in dev_src], "f32")
    for r in range(R):
        assert_same(host(hout[r]), ref.outs[r], f"ordered host pipeline rank {r}")


# --------------------------------------------------------------------------
# the other AllReduce algorithms: halving-doubling and naive
# --------------------------------------------------------------------------

def check_algo(rr, xs, wire, algo, cfg=None, what=""):
    outs = rr.allreduce_algo(xs, wire=wire, algo=algo, cfg=cfg)
    torch.cuda.synchronize()
    ref = oracle.allreduce_algo([host(x) for x in xs], NAME[xs[0].dtype], wire, algo)
    assert ref.status == oracle.OK
    for r in range(len(xs)):
        assert_same(host(outs[r]), ref.outs[r], f"{what} rank {r}")


@pytest.mark.parametrize("algo", ["hd", "naive"])
@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_algorithm_grid(rr, algo, dtype, wire):
    for R in (1, 2, 3, 4, 5, 7, 8, 12, 16, 17, 24, 33, 48, 64):
        for N in (1, R + 1, 4097, 65_537):
            xs = gen(R, N, dtype, 7 * R + N)
            tag = f"{algo} {NAME[dtype]}/{wire} R={R} N={N}"
            check_algo(rr, xs, wire, algo, what=tag)
            check_algo(rr, xs, wire, algo, cfg=cfg_of(rr, path=rr.PATH_SIMPLE), what=tag + " simple")
            if N * xs[0].element_size() >= 16 and R <= 16:
                check_algo(rr, xs, wire, algo, cfg=cfg_of(rr, path=rr.PATH_BULK, tile=256), what=tag + " bulk256")
            if N * xs[0].element_size() >= 16:
                check_algo(rr, xs, wire, algo, cfg=cfg_of(rr, path=rr.PATH_DIRECT), what=tag + " direct")


@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_algorithm_occupancy_variants(rr, dtype, wire):
    """Messages large enough that the direct path's threads loop, so that
    halving-doubling below seven ranks runs its three-CTA kernels (with and
    without extra ranks), and the naive order its looping ring kernel."""
    for R, N in ((3, 3 * 400_003), (4, 4 * 300_007), (5, 5 * 250_001), (6, 6 * 200_003), (12, 12 * 100_003)):
        xs = gen(R, N, dtype, 91 * R)
        for algo in ("hd", "naive"):
            check_algo(rr, xs, wire, algo, cfg=cfg_of(rr, path=rr.PATH_DIRECT),
                       what=f"{algo} {NAME[dtype]}/{wire} R={R} N={N} direct")


@pytest.mark.parametrize("algo", ["hd", "naive"])
def test_algorithm_full_size(rr, wl, algo):
    xs = wl.inputs(wl.config2(512), "cuda")
    outs = rr.allreduce_algo(xs, algo=algo)
    torch.cuda.synchronize()
    N = xs[0].numel()
    idx = sample_indices(N, 8)
    ti = torch.from_numpy(idx).cuda()
    want = oracle.fold_gathered_algo([host(x[ti]) for x in xs], idx.astype(np.uint64), N, "f16", None, algo)
    for r in range(8):  # quick pre-check on sampled elements
        assert_same(host(outs[r][ti]), want, f"{algo} 512 MiB sampled rank {r}")
    check_full(rr, xs, outs, algo=algo, what=f"{algo} 512 MiB")
    del outs, xs
    torch.cuda.empty_cache()


def test_capped_grids(rr):
    # a persistent grid of a few CTAs walks many tiles each; same bits
    for dtype, wire in PAIRS[:4]:
        xs = gen(8, 300_007, dtype, 99)
        for cap in (1, 7, 100):
            check_ar(rr, xs, wire, cfg=cfg_of(rr) if cap == 0 else rr.LaunchCfg(0, 0, 0, 0, 0, cap),
                     what=f"max_ctas={cap} {NAME[dtype]}/{wire}")
            check_ar(rr, xs, wire, cfg=rr.LaunchCfg(rr.PATH_SIMPLE, 0, 0, 0, 0, cap),
                     what=f"simple max_ctas={cap} {NAME[dtype]}/{wire}")
            check_ar(rr, xs, wire, cfg=rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 128, cap),
                     what=f"direct max_ctas={cap} {NAME[dtype]}/{wire}")
    # few ranks: the direct path takes several vectors per thread
    for R in (2, 3, 4):
        xs = gen(R, 300_007, torch.float16, 98)
        for cap in (1, 7, 100):
            check_ar(rr, xs, cfg=rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 256, cap), what=f"direct R={R} cap={cap}")
            check_rs(rr, xs[:R], cfg=rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 64, cap), what=f"direct RS R={R} cap={cap}") \
                if (300_007 // R * 2) % 16 == 0 else None


# --------------------------------------------------------------------------
# every direct-path kernel variant, forced through the launch configuration
# --------------------------------------------------------------------------

def direct_variants(op, wide, shifted):
    """(vectors, register budget) of every direct-path kernel the library
    builds for this collective (0 = the budget the planner gives it)."""
    if shifted:
        rows = (1, 2, 4) if op == "ag" else ((1, 2) if wide else (1, 2, 3, 4))
        return [(u, 0) for u in rows]
    if op == "ag":
        return [(1, 2), (2, 2), (4, 2)]
    if wide:
        return [(1, 2), (2, 2)]
    return [(1, 2), (1, 3), (2, 2), (2, 3), (3, 2), (4, 2)]


@pytest.mark.parametrize("dtype,wire", PAIRS, ids=lambda v: str(v))
def test_every_direct_variant(rr, dtype, wire):
    """Each direct-path kernel (1-4 vectors a thread, both register budgets;
    the shifted kernels at 1-4 rows a warp) on chunk boundaries on and off the
    16-byte grid with a ragged last chunk, on the planner's grid and on a grid
    of five CTAs whose threads loop many times; bit for bit against the oracle."""
    E = torch.tensor([], dtype=dtype).element_size()
    V = 16 // E
    wide = dtype != torch.float32 and wire == "f32"
    for R in (2, 3, 4, 5, 9):
        for off_grid in (False, True):
            base = V * 4001 + (1 if off_grid else 0)
            N = R * base + (R - 1)
            xs = gen(R, N, dtype, 1009 * R + base)
            hx = [host(x) for x in xs]
            ref_ar = oracle.allreduce(hx, NAME[dtype], wire)
            ref_rs = oracle.reduce_scatter(hx, NAME[dtype], wire)
            lens = [oracle.chunk_len(N, R, c) for c in range(R)]
            chunks = gen(R, 0, dtype, 2003 * R + base, lengths=lens)
            ref_ag = oracle.allgather([host(c) for c in chunks], N, NAME[dtype]) if wire is None else None
            for cap in (0, 5):
                for u, occ in direct_variants("ar", wide, False):
                    cfg = rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, occ, 0, cap, 0, u)
                    outs = run_ar(rr, xs, wire, cfg=cfg)
                    torch.cuda.synchronize()
                    for r in range(R):
                        assert_same(host(outs[r]), ref_ar.outs[r], f"AR U={u} occ={occ} cap={cap} R={R} "
                                                                   f"off_grid={off_grid} rank {r}")
                for u, occ in direct_variants("rs", wide, off_grid):
                    cfg = rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, occ, 0, cap, 0, u)
                    parts = [torch.full((lens[c],), float("nan"), dtype=dtype, device="cuda") for c in range(R)]
                    rr.collective(rr.OP_REDUCE_SCATTER, xs, parts, N, wire, 0, None, cfg)
                    torch.cuda.synchronize()
                    for c in range(R):
                        assert_same(host(parts[c]), ref_rs.outs[c], f"RS U={u} occ={occ} cap={cap} R={R} "
                                                                    f"off_grid={off_grid} chunk {c}")
                for pf in (2, 3, 4):  # L2 prefetch before the wait, one iteration ahead, both
                    cfg = rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 0, cap, 0, 0, 0, pf)
                    outs = run_ar(rr, xs, wire, cfg=cfg)
                    torch.cuda.synchronize()
                    for r in range(R):
                        assert_same(host(outs[r]), ref_ar.outs[r], f"AR prefetch={pf} cap={cap} R={R} rank {r}")
                    parts = [torch.full((lens[c],), float("nan"), dtype=dtype, device="cuda") for c in range(R)]
                    rr.collective(rr.OP_REDUCE_SCATTER, xs, parts, N, wire, 0, None, cfg)
                    torch.cuda.synchronize()
                    for c in range(R):
                        assert_same(host(parts[c]), ref_rs.outs[c], f"RS prefetch={pf} cap={cap} R={R} chunk {c}")
                if ref_ag is None:
                    continue
                for u, occ in direct_variants("ag", False, off_grid):
                    cfg = rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, occ, 0, cap, 0, u)
                    outs = [torch.full((N,), float("nan"), dtype=dtype, device="cuda") for _ in range(R)]
                    rr.collective(rr.OP_ALLGATHER, chunks, outs, N, None, 0, None, cfg)
                    torch.cuda.synchronize()
                    for r in range(R):
                        assert_same(host(outs[r]), ref_ag.outs[r], f"AG U={u} occ={occ} cap={cap} R={R} "
                                                                   f"off_grid={off_grid} rank {r}")
                for pf in (2, 3, 4):
                    outs = [torch.full((N,), float("nan"), dtype=dtype, device="cuda") for _ in range(R)]
                    rr.collective(rr.OP_ALLGATHER, chunks, outs, N, None, 0, None,
                                  rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 0, cap, 0, 0, 0, pf))
                    torch.cuda.synchronize()
                    for r in range(R):
                        assert_same(host(outs[r]), ref_ag.outs[r], f"AG prefetch={pf} cap={cap} R={R} rank {r}")
    assert rr.device_status() == 0


def test_launch_config_rejects_kernels_not_built(rr):
    """A forced direct path asking for a kernel the library does not build is
    RR_ERR_UNSUPPORTED, before anything is launched."""
    xs = gen(4, 4 * 8192, torch.float32, 3)
    outs = [torch.empty_like(x) for x in xs]
    for u, occ in ((3, 3), (4, 3)):
        with pytest.raises(rr.RingError) as e:
            rr.collective(rr.OP_ALLREDUCE, xs, outs, xs[0].numel(), None, 0, None,
                          rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, occ, 0, 0, 0, u))
        assert e.value.status == rr.ERR_UNSUPPORTED
    with pytest.raises(rr.RingError) as e:  # AllGather: no three-vector kernel
        rr.collective(rr.OP_ALLGATHER, [x[:8192] for x in xs], outs, xs[0].numel(), None, 0, None,
                      rr.LaunchCfg(rr.PATH_DIRECT, 0, 0, 0, 0, 0, 0, 3))
    assert e.value.status == rr.ERR_UNSUPPORTED
