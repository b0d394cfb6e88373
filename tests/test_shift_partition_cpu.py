"""The shifted kernel's work partition, modelled on the CPU.

rr_shift_kernel (csrc/rr_kernels.cuh) splits each chunk's output vectors into
work items of US rows and runs most items with no bounds check at all; the
rest (a ReduceScatter or AllReduce chunk's last item, an AllGather chunk's
first item and last three) go through the checked code, one row to a warp, and the warps take
the checked rows first and the inner items after, in turn.  These tests
restate that index arithmetic in Python and check, over many chunk lengths,
rank counts and row counts, that every output vector wholly inside a chunk is
written exactly once and that every vector of an unchecked item has its
source blocks inside the buffers (so the unchecked loads and stores stay in
bounds).  Chunk partition: block c of floor(N / R) elements starts at c *
floor(N / R), the last takes the rest (page hwcomputing.csdn.net
6a0dc11a10ee7a33f273f7fd.html, section "Ring 通信为什么常见")."""

import random

import pytest


def first_inner_item(warp, n_warps, n_edge):
    """The kernel's w0: units are dealt in turn, the n_edge checked rows first."""
    if warp < n_edge:
        return warp + (n_edge - warp + n_warps - 1) // n_warps * n_warps - n_edge
    return warp - n_edge


def walk(w0, inc, L):
    """Chunk and item of inner item w0 (chunks 0..L-2 hold inc each)."""
    if w0 < (L - 1) * inc:
        return w0 // inc, w0 - (w0 // inc) * inc
    return L - 1, w0 - (L - 1) * inc


def step(c, item, n_warps, inc, L):
    item += n_warps
    while c < L - 1 and item >= inc:
        item -= inc
        c += 1
    return c, item


def reduce_scatter_partition(N, L, V, US, n_warps):
    base = N // L
    len_last = N - (L - 1) * base
    per_item = 31 * US
    ipc = (base // V + per_item - 1) // per_item
    ipl = (len_last // V + per_item - 1) // per_item
    inc, inl = max(ipc - 1, 0), max(ipl - 1, 0)
    n_inner = (L - 1) * inc + inl
    n_edge = L * US
    written = {}

    def put(c, u):
        written.setdefault((c, u), 0)
        written[(c, u)] += 1

    for e in range(n_edge):  # checked rows: chunk e // US's last item, row e % US
        ce, k = e // US, e % US
        ln = base if ce < L - 1 else len_last
        nv, n_c = ln // V, (ipc if ce < L - 1 else ipl)
        if n_c == 0:
            continue
        for lane in range(31):
            u = (n_c - 1) * per_item + 31 * k + lane
            if u < nv:
                put(ce, u)
    for warp in range(n_warps):  # inner items
        w = first_inner_item(warp, n_warps, n_edge)
        if w >= n_inner:
            continue
        c, item = walk(w, inc, L)
        while w < n_inner:
            ln = base if c < L - 1 else len_last
            nv, g0 = ln // V, c * base
            a0 = g0 - g0 % V  # element of output vector 0's aligned block
            for k in range(US):
                for lane in range(32):
                    u = item * per_item + 31 * k + lane
                    assert u <= nv - 1 and a0 + (u + 1) * V <= N, (N, L, V, US, c, item, u)  # unchecked load
                    if lane < 31:
                        assert u < nv - 1, (N, L, V, US, c, item, u)  # unchecked store, no tail
                        put(c, u)
            c, item = step(c, item, n_warps, inc, L)
            w += n_warps
    for c in range(L):
        nv = (base if c < L - 1 else len_last) // V
        for u in range(nv):
            assert written.get((c, u)) == 1, (N, L, V, US, c, u, written.get((c, u)))
    assert all(u < (base if c < L - 1 else len_last) // V for c, u in written)


def allgather_partition(N, L, V, US, n_warps):
    base = N // L
    len_last = N - (L - 1) * base
    nvec = N // V
    rpc, rpl = (base // V + 64) // 32, (len_last // V + 64) // 32
    ipc, ipl = (rpc + US - 1) // US, (rpl + US - 1) // US
    inc, inl = max(ipc - 4, 0), max(ipl - 4, 0)
    epc, epl = (ipc - inc) * US, (ipl - inl) * US
    n_edge, n_inner = (L - 1) * epc + epl, (L - 1) * inc + inl

    def chunk(c):
        cb = c * base
        ln = base if c < L - 1 else len_last
        vf = (cb + V - 1) // V
        return ln, vf, min((cb + ln) // V, nvec)

    written = {}
    for e in range(n_edge):  # checked rows: a chunk's first item, then its last three
        ce = e // epc if e < (L - 1) * epc else L - 1
        u = e - ce * epc
        j, in_c = u // US, (inc if ce < L - 1 else inl)
        it = j if (j == 0 or in_c == 0) else j + in_c
        ln, vf, ve = chunk(ce)
        for lane in range(32):
            v = (vf // 32 + it * US + u % US) * 32 + lane
            if vf <= v < ve:
                written[v] = written.get(v, 0) + 1
    for warp in range(n_warps):  # inner items
        w = first_inner_item(warp, n_warps, n_edge)
        if w >= n_inner:
            continue
        c, item = walk(w, inc, L)
        while w < n_inner:
            ln, vf, ve = chunk(c)
            for r in range(US):
                for lane in range(32):
                    v = (vf // 32 + (1 + item) * US + r) * 32 + lane
                    assert vf <= v < ve, (N, L, V, US, c, item, v)  # wholly in the chunk
                    assert (v - vf + 2) * V <= ln, (N, L, V, US, c, item, v)  # both source blocks inside
                    written[v] = written.get(v, 0) + 1
            c, item = step(c, item, n_warps, inc, L)
            w += n_warps
    for c in range(L):
        _, vf, ve = chunk(c)
        for v in range(vf, ve):
            assert written.get(v) == 1, (N, L, V, US, c, v, written.get(v))
    assert all(any(chunk(c)[1] <= v < chunk(c)[2] for c in range(L)) for v in written)


def allreduce_partition(N, L, V, US, n_warps):
    """The AllReduce rows (chunks on the grid): rows of 32 whole vectors."""
    base = N // L
    len_last = N - (L - 1) * base
    per_item = 32 * US
    nvc, nvl = base // V, len_last // V
    ipc, ipl = (nvc + per_item - 1) // per_item, (nvl + per_item - 1) // per_item
    inc, inl = max(ipc - 1, 0), max(ipl - 1, 0)
    n_inner, n_edge = (L - 1) * inc + inl, L * US
    written = {}
    for e in range(n_edge):
        ce, k = e // US, e % US
        nv, n_c = (nvc, ipc) if ce < L - 1 else (nvl, ipl)
        if n_c == 0:
            continue
        for lane in range(32):
            u = (n_c - 1) * per_item + 32 * k + lane
            if u < nv:
                written[(ce, u)] = written.get((ce, u), 0) + 1
    for warp in range(n_warps):
        w = first_inner_item(warp, n_warps, n_edge)
        if w >= n_inner:
            continue
        c, item = walk(w, inc, L)
        while w < n_inner:
            nv = nvc if c < L - 1 else nvl
            for k in range(US):
                for lane in range(32):
                    u = item * per_item + 32 * k + lane
                    assert u < nv, (N, L, V, US, c, item, u)  # a whole vector of the chunk: no check needed
                    written[(c, u)] = written.get((c, u), 0) + 1
            c, item = step(c, item, n_warps, inc, L)
            w += n_warps
    for c in range(L):
        for u in range(nvc if c < L - 1 else nvl):
            assert written.get((c, u)) == 1, (N, L, V, US, c, u, written.get((c, u)))
    assert all(u < (nvc if c < L - 1 else nvl) for c, u in written)


def lengths(seed):
    """Chunk lengths from under one vector to several items' worth of rows."""
    rng = random.Random(seed)
    fixed = [1, 2, 7, 8, 9, 31, 255, 256, 257, 1023, 2047, 4095, 4097, 12_345]
    return fixed + [rng.randrange(1, 20_000) for _ in range(3)]


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 8])
def test_reduce_scatter_inner_items_stay_in_bounds(L):
    for V in (4, 8):
        for US in (1, 2, 3, 4):
            for n in lengths(10 * L + US):
                for n_warps in (1, 7, 97):
                    reduce_scatter_partition(n * L + L // 2, L, V, US, n_warps)


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 8])
def test_allgather_inner_items_stay_in_bounds(L):
    for V in (4, 8):
        for US in (1, 2, 4):
            for n in lengths(20 * L + US):
                for n_warps in (1, 7, 97):
                    allgather_partition(n * L + L // 2, L, V, US, n_warps)


@pytest.mark.parametrize("L", [1, 2, 3, 4])
def test_allreduce_rows_inner_items_stay_in_bounds(L):
    for V in (4, 8):
        for US in (2, 4):
            for n in lengths(30 * L + US):
                n = n // V * V or V  # chunks on the 16-byte grid
                for n_warps in (1, 7, 97):
                    allreduce_partition(n * L + V // 2, L, V, US, n_warps)
