"""Pins of the oracle's ring simulation against what the pages and arithmetic fix.

Each pin is independent of the oracle's own code: hand-derived values from the
pages (tests/golden), exact integer sums, numpy / torch arithmetic, the
traffic formula printed on the pages, invariants (all outputs identical,
AllReduce = AllGather after ReduceScatter) and the closed form of the fold.
The last test plants mistakes in a copy of the oracle and checks that these
pins catch every one of them.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
PAIRS = [("f32", "f32"), ("f16", "f16"), ("bf16", "bf16"), ("f32", "bf16"), ("f32", "f16"), ("f16", "f32"),
         ("bf16", "f32")]
EB = {"f32": 4, "f16": 2, "bf16": 2}


def golden_lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def hexarr(tokens, dtype):
    if dtype == "f32":
        return np.array([int(t, 16) for t in tokens], dtype=np.uint32).view(np.float32)
    return np.array([int(t, 16) for t in tokens], dtype=np.uint16)


def bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def rand_inputs(rng, R, N, dtype, scale=1.0, special=False):
    xs = []
    for _ in range(R):
        v = (rng.standard_normal(N) * scale).astype(np.float32)
        if special and N:
            # sprinkle values whose sums tie or cancel
            k = rng.integers(0, N, size=max(1, N // 4))
            v[k] = rng.choice(np.array([1.0, -1.0, 2.0 ** -11, 2.0 ** -24, 2.0 ** -8, 0.0, -0.0],
                                       dtype=np.float32), size=k.size)
        if dtype == "f32":
            xs.append(v)
        elif dtype == "f16":
            xs.append(v.astype(np.float16).view(np.uint16))
        else:
            xs.append(torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    return xs


def to_f64(a, dtype):
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def int_inputs(rng, R, N, dtype):
    xs = []
    for _ in range(R):
        v = rng.integers(-8, 9, size=N).astype(np.float32)
        if dtype == "f32":
            xs.append(v)
        elif dtype == "f16":
            xs.append(v.astype(np.float16).view(np.uint16))
        else:
            xs.append(torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    return xs


# --------------------------------------------------------------------------
# pins from the pages (golden fixtures)
# --------------------------------------------------------------------------

def pin_schedule_r4():
    rows = golden_lines("ring_schedule_r4.txt")
    want = [(r[0], int(r[1]), int(r[2]), int(r[3]), int(r[4])) for r in rows]
    x = [np.zeros(8, np.float32) for _ in range(4)]
    res = oracle.allreduce(x, "f32", trace_cap=256)
    assert res.status == oracle.OK
    name = {oracle.PHASE_RS: "RS", oracle.PHASE_AG: "AG"}
    got = [(name[p], s, a, b, c) for (p, s, a, b, c, _) in res.trace]
    assert sorted(got) == sorted(want)


def pin_fold_order_r3():
    for row in golden_lines("fold_order_r3.txt"):
        dtype, wire = row[0], row[1]
        groups = " ".join(row[2:]).split("|")[1:]
        xs = [hexarr(g.split(), dtype) for g in groups[:3]]
        want = hexarr(groups[3].split(), dtype)
        res = oracle.allreduce(xs, dtype, wire)
        assert res.status == oracle.OK
        for r in range(3):
            assert bits(res.outs[r]).tolist() == bits(want).tolist(), (dtype, wire, r)


def pin_partition_r4_n10():
    rows = golden_lines("partition_r4_n10.txt")
    xs = [hexarr(r[2:], "f16") for r in rows if r[0] == "in"]
    want = hexarr([r for r in rows if r[0] == "out"][0][1:], "f16")
    res = oracle.allreduce(xs, "f16")
    assert res.status == oracle.OK
    for r in range(4):
        assert res.outs[r].tolist() == want.tolist()
    rs = oracle.reduce_scatter(xs, "f16")
    assert rs.status == oracle.OK
    for row in rows:
        if row[0] == "rs":
            assert rs.outs[int(row[1])].tolist() == hexarr(row[2:], "f16").tolist()


def pin_two_level():
    for row in golden_lines("two_level.txt"):
        R, L, N = int(row[1]), int(row[2]), int(row[3])
        groups = " ".join(row[4:]).split("|")[1:]
        xs = [hexarr(g.split(), "f16") for g in groups[:R]]
        want = hexarr(groups[R].split(), "f16")
        assert all(x.size == N for x in xs)
        res = oracle.allreduce(xs, "f16", group_size=L)
        assert res.status == oracle.OK
        for r in range(R):
            assert res.outs[r].tolist() == want.tolist(), (row[0], r)


def test_golden_schedule_r4():
    pin_schedule_r4()


def test_golden_fold_order_r3():
    pin_fold_order_r3()


def test_golden_partition_r4_n10():
    pin_partition_r4_n10()


def test_golden_two_level():
    pin_two_level()


# --------------------------------------------------------------------------
# schedule and traffic
# --------------------------------------------------------------------------

def pin_ring_neighbours():
    for R in range(1, 10):
        x = [np.zeros(3 * R + 1, np.float32) for _ in range(R)]
        res = oracle.allreduce(x, "f32", trace_cap=4096)
        assert res.status == oracle.OK
        for phase in (oracle.PHASE_RS, oracle.PHASE_AG):
            msgs = [m for m in res.trace if m[0] == phase]
            assert len(msgs) == R * (R - 1)  # R-1 steps, one send per rank per step
            assert {m[1] for m in msgs} == set(range(R - 1))
            for (_, step, src, dst, chunk, _) in msgs:
                assert dst == (src + 1) % R  # only the next neighbour on the ring
            for step in range(R - 1):
                assert sorted(m[2] for m in msgs if m[1] == step) == list(range(R))


def pin_traffic():
    # per rank 2(N-1)*S/N for AllReduce (page hwcomputing.csdn.net/6a0dc11a..., "Ring 通信为什么常见"),
    # (n-1)*S/n for AllGather (page ai6s.net/6a102b54..., "分布式推理中的通信"); the same
    # (R-1)*S/R holds for the reduce-scatter half.
    rng = np.random.default_rng(1)
    for R in (1, 2, 3, 4, 8):
        for dtype, wire in PAIRS:
            N = 6 * R
            xs = rand_inputs(rng, R, N, dtype)
            S = N * EB[wire]
            ar = oracle.allreduce(xs, dtype, wire)
            assert ar.sent_bytes == [2 * (R - 1) * S // R] * R
            rs = oracle.reduce_scatter(xs, dtype, wire)
            assert rs.sent_bytes == [(R - 1) * S // R] * R
            ag = oracle.allgather([x[: N // R] for x in xs], N, dtype)
            assert ag.sent_bytes == [(R - 1) * N * EB[dtype] // R] * R


def test_ring_neighbours_and_steps():
    pin_ring_neighbours()


def test_traffic_formula():
    pin_traffic()


# --------------------------------------------------------------------------
# arithmetic pins
# --------------------------------------------------------------------------

def pin_small_integers():
    # integers in [-8, 8]: every partial sum is an integer below 2^8 in magnitude,
    # exact in all three formats, so every output is the exact sum
    rng = np.random.default_rng(2)
    for R in (1, 2, 3, 5, 8, 16):
        for dtype, wire in PAIRS:
            for N in (0, 1, R - 1, R, R + 1, 37):
                xs = int_inputs(rng, R, N, dtype)
                exact = sum(to_f64(x, dtype) for x in xs) if R else 0
                res = oracle.allreduce(xs, dtype, wire)
                assert res.status == oracle.OK
                for r in range(R):
                    np.testing.assert_array_equal(to_f64(res.outs[r], dtype), exact)
                for L in [d for d in (1, 2, 4) if R % d == 0 and d < R]:
                    res = oracle.allreduce(xs, dtype, wire, group_size=L)
                    for r in range(R):
                        np.testing.assert_array_equal(to_f64(res.outs[r], dtype), exact)


def pin_literal_equals_closed_form():
    rng = np.random.default_rng(3)
    for R in range(1, 10):
        for N in list(range(0, 41)):
            for dtype, wire in PAIRS:
                xs = rand_inputs(rng, R, N, dtype, scale=1.0, special=True)
                res = oracle.allreduce(xs, dtype, wire)
                assert res.status == oracle.OK
                if N == 0:
                    continue
                cf = oracle.fold_gathered(xs, np.arange(N), N, dtype, wire)
                for r in range(R):
                    assert bits(res.outs[r]).tolist() == bits(cf).tolist(), (R, N, dtype, wire, r)


def pin_two_level_closed_form():
    rng = np.random.default_rng(4)
    for G in (1, 2, 3, 4):
        for L in (1, 2, 3, 4, 8):
            R = G * L
            for N in (1, 2, L - 1 if L > 1 else 3, L + 1, 3 * L + 2, 40):
                for dtype, wire in PAIRS:
                    xs = rand_inputs(rng, R, N, dtype, special=True)
                    res = oracle.allreduce(xs, dtype, wire, group_size=L)
                    assert res.status == oracle.OK
                    cf = oracle.fold_gathered(xs, np.arange(N), N, dtype, wire, group_size=L)
                    for r in range(R):
                        assert bits(res.outs[r]).tolist() == bits(cf).tolist(), (G, L, N, dtype, wire)


def test_small_integers_exact():
    pin_small_integers()


def test_literal_simulation_equals_closed_form():
    pin_literal_equals_closed_form()


def test_two_level_equals_closed_form():
    pin_two_level_closed_form()


def test_outputs_identical():
    rng = np.random.default_rng(5)
    for dtype, wire in PAIRS:
        for R, L in ((8, 0), (16, 8), (12, 4)):
            xs = rand_inputs(rng, R, 1001, dtype, special=True)
            res = oracle.allreduce(xs, dtype, wire, group_size=L)
            for r in range(1, R):
                assert bits(res.outs[r]).tolist() == bits(res.outs[0]).tolist()


def test_r1_is_identity_or_cast_round_trip():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(257).astype(np.float32)
    assert bits(oracle.allreduce([x], "f32").outs[0]).tolist() == bits(x).tolist()
    h = x.astype(np.float16).view(np.uint16)
    assert oracle.allreduce([h], "f16").outs[0].tolist() == h.tolist()
    via_bf16 = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert bits(oracle.allreduce([x], "f32", "bf16").outs[0]).tolist() == bits(via_bf16).tolist()
    via_f16 = x.astype(np.float16).astype(np.float32)
    assert bits(oracle.allreduce([x], "f32", "f16").outs[0]).tolist() == bits(via_f16).tolist()
    assert bits(oracle.reduce_scatter([x], "f32").outs[0]).tolist() == bits(x).tolist()
    assert bits(oracle.allgather([x], x.size, "f32").outs[0]).tolist() == bits(x).tolist()


def pin_r2_single_add():
    # two ranks: one hop, i.e. one correctly rounded addition in the wire format
    rng = np.random.default_rng(7)
    a32, b32 = rng.standard_normal((2, 4099)).astype(np.float32)
    res = oracle.allreduce([a32, b32], "f32")
    assert bits(res.outs[0]).tolist() == bits(a32 + b32).tolist()
    a16, b16 = (a32 * 1e-3).astype(np.float16), (b32 * 1e-3).astype(np.float16)
    res = oracle.allreduce([a16.view(np.uint16), b16.view(np.uint16)], "f16")
    assert res.outs[1].tolist() == (a16 + b16).view(np.uint16).tolist()
    ta, tb = torch.from_numpy(a32).to(torch.bfloat16), torch.from_numpy(b32).to(torch.bfloat16)
    want = (ta + tb).view(torch.int16).numpy().view(np.uint16)
    res = oracle.allreduce([ta.view(torch.int16).numpy().view(np.uint16),
                            tb.view(torch.int16).numpy().view(np.uint16)], "bf16")
    assert res.outs[0].tolist() == want.tolist()
    # binary32 storage on a bfloat16 wire: cast both, add once, widen
    res = oracle.allreduce([a32, b32], "f32", "bf16")
    assert bits(res.outs[0]).tolist() == bits((ta + tb).to(torch.float32).numpy()).tolist()


def test_r2_is_one_rounded_add():
    pin_r2_single_add()


@pytest.mark.parametrize("dtype,wire,R,L,dist", [
    ("f16", "f32", 8, 0, "grad"),
    ("bf16", "f32", 8, 0, "grad2"),
    ("f32", "f32", 4, 0, "uniform"),
    ("f16", "f16", 8, 0, "grad"),
    ("f32", "bf16", 8, 0, "normal"),
    ("f32", "f32", 16, 8, "uniform"),
    ("bf16", "bf16", 8, 0, "grad2"),
])
def test_error_bound_against_fp64(dtype, wire, R, L, dist):
    """|out - exact| <= tol * sum_r |x_r|: the recursive-summation bound.

    tol = 1e-6 for binary32 ((R-1) * 2^-24 < 1e-6 for R <= 16), R * 2^-10 for a
    binary16 wire and R * 2^-7 for a bfloat16 wire (ingress rounding plus R-1
    hops, 2x margin).  Binary16 subnormals add at most (R-1) half-spacings 2^-25.
    """
    rng = np.random.default_rng(8)
    N = 20011
    if dist == "uniform":
        xs32 = [rng.uniform(-1, 1, N).astype(np.float32) for _ in range(R)]
    elif dist == "normal":
        xs32 = [rng.standard_normal(N).astype(np.float32) for _ in range(R)]
    else:
        sig = 1e-3 if dist == "grad" else 1e-2
        xs32 = [(rng.standard_normal(N) * sig).astype(np.float32) for _ in range(R)]
    if dtype == "f16":
        xs = [x.astype(np.float16).view(np.uint16) for x in xs32]
    elif dtype == "bf16":
        xs = [torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for x in xs32]
    else:
        xs = xs32
    x64 = [to_f64(x, dtype) for x in xs]
    exact = np.sum(x64, axis=0)
    mag = np.sum(np.abs(x64), axis=0)
    tol = {"f32": 1e-6, "f16": R * 2.0 ** -10, "bf16": R * 2.0 ** -7}[wire]
    if wire == "f32" and dtype != "f32":
        # binary32 accumulation: (R-1) binary32 roundings, then one rounding to storage
        tol = (R - 1) * 2.0 ** -24 + {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}[dtype]
    floor = (R - 1) * 2.0 ** -25 if wire == "f16" else (2.0 ** -25 if dtype == "f16" else 0.0)
    out = to_f64(oracle.allreduce(xs, dtype, wire, group_size=L).outs[0], dtype)
    err = np.abs(out - exact)
    assert np.all(err <= tol * mag + floor), float(np.max(err / (mag + 1e-300)))


# --------------------------------------------------------------------------
# composition and placement
# --------------------------------------------------------------------------

def pin_composition():
    # the pages: HCCL's AllReduce is ReduceScatter followed by AllGather
    rng = np.random.default_rng(9)
    for R in (1, 2, 3, 4, 7, 8):
        for N in (0, 1, R + 3, 10 * R, 101):
            for dtype, wire in PAIRS:
                xs = rand_inputs(rng, R, N, dtype, special=True)
                ar = oracle.allreduce(xs, dtype, wire)
                rs = oracle.reduce_scatter(xs, dtype, wire)
                ag = oracle.allgather(rs.outs, N, dtype)
                assert ar.status == rs.status == ag.status == oracle.OK
                for r in range(R):
                    assert bits(ag.outs[r]).tolist() == bits(ar.outs[r]).tolist()


def pin_allgather_concat():
    rng = np.random.default_rng(10)
    for R in (1, 2, 3, 5, 8):
        for N in (0, 1, R - 1, R, 2 * R + 1, 64):
            for dtype in ("f32", "f16", "bf16"):
                base = N // R
                lens = [base] * (R - 1) + [N - (R - 1) * base]
                chunks = rand_inputs(rng, 1, N, dtype)[0]
                ins = np.split(chunks, np.cumsum(lens)[:-1]) if R > 1 else [chunks]
                ins = [np.ascontiguousarray(c) for c in ins]
                res = oracle.allgather(ins, N, dtype)
                for r in range(R):
                    assert bits(res.outs[r]).tolist() == bits(chunks).tolist()


def test_allreduce_is_allgather_after_reducescatter():
    pin_composition()


def test_allgather_is_concatenation():
    pin_allgather_concat()


def test_two_level_g2_is_sum_of_group_rings():
    # G = 2: each group runs the flat ring of L ranks, then one hop adds the two
    # group results; computed here with the flat oracle and the wire add
    rng = np.random.default_rng(11)
    for dtype, wire in PAIRS:
        L, N = 8, 1003
        xs = rand_inputs(rng, 2 * L, N, dtype, special=True)
        two = oracle.allreduce(xs, dtype, wire, group_size=L).outs[0]
        if dtype != wire:
            continue  # the flat group results are already widened; covered by the closed form
        g0 = oracle.allreduce(xs[:L], dtype, wire).outs[0]
        g1 = oracle.allreduce(xs[L:], dtype, wire).outs[0]
        if dtype == "f32":
            want = g0 + g1
        else:
            want = oracle.wire_add(g0, g1, wire)
        assert bits(two).tolist() == bits(want).tolist()


def test_partition_properties():
    for R in range(1, 20):
        for N in list(range(0, 50)) + [50_000_017, 2 ** 31 + 5]:
            lens = [oracle.chunk_len(N, R, c) for c in range(R)]
            offs = [oracle.chunk_off(N, R, c) for c in range(R)]
            assert sum(lens) == N
            assert all(l == N // R for l in lens[:-1])
            assert all(offs[c] + lens[c] == (offs[c + 1] if c + 1 < R else N) for c in range(R))


# --------------------------------------------------------------------------
# fault handling of the simulated transport (host side only)
# --------------------------------------------------------------------------

def test_faults_are_detected():
    x = [np.ones(16, np.float32) for _ in range(4)]
    assert oracle.allreduce(x, "f32").status == oracle.OK
    r = oracle.allreduce(x, "f32", fault=(oracle.FAULT_DROP, 2, oracle.PHASE_RS, 1))
    assert r.status == oracle.ETIMEOUT
    r = oracle.allreduce(x, "f32", fault=(oracle.FAULT_DUP, 1, oracle.PHASE_AG, 0))
    assert r.status == oracle.EPROTO
    r = oracle.allreduce(x, "f32", fault=(oracle.FAULT_SILENT, 3, oracle.PHASE_RS, 2), poll_limit=3)
    assert r.status == oracle.ETIMEOUT
    r = oracle.reduce_scatter(x, "f32", fault=(oracle.FAULT_DROP, 0, oracle.PHASE_RS, 0))
    assert r.status == oracle.ETIMEOUT
    r = oracle.allgather([np.ones(4, np.float32)] * 4, 16, "f32",
                         fault=(oracle.FAULT_SILENT, 1, oracle.PHASE_AG, 0))
    assert r.status == oracle.ETIMEOUT
    x16 = [np.ones(16, np.float32) for _ in range(16)]
    r = oracle.allreduce(x16, "f32", group_size=8, fault=(oracle.FAULT_DROP, 0, oracle.PHASE_XCHG, 0))
    assert r.status == oracle.ETIMEOUT


def test_bad_arguments():
    x = [np.ones(4, np.float32)] * 3
    assert oracle.allreduce(x, "f32", group_size=2).status == oracle.EINVAL
    h = [x[0].astype(np.float16).view(np.uint16)] * 3
    assert oracle.allreduce(h, "f16", "bf16").status == oracle.EUNSUPPORTED
    assert oracle.allreduce(h, "bf16", "f16").status == oracle.EUNSUPPORTED
    assert oracle.allreduce(h, "f16", "f32").status == oracle.OK


# --------------------------------------------------------------------------
# planted mistakes: every one must be caught by a pin above
# --------------------------------------------------------------------------

MUTATIONS = {
    # the reduce-scatter walks the ring the wrong way
    "rs_direction": ("int cs = mod(l - t, L);", "int cs = mod(l + t, L);"),
    # the received chunk index is off by one
    "rs_recv_chunk": ("int cr = mod(l - t - 1, L);", "int cr = mod(l - t, L);"),
    # the closed form folds in the reverse direction
    "closed_form_direction": ("int r = g * L + (c + step) % L;", "int r = g * L + (c + L - step) % L;"),
    # the remainder goes to the first chunk instead of the last
    "partition_remainder": ("  if (c < R - 1) return base;\n  return count - (size_t)(R - 1) * base;",
                            "  if (c > 0) return base;\n  return count - (size_t)(R - 1) * base;"),
    # ties round away from zero instead of to even
    "rounding_ties": ("if (rem > half || (rem == half && (M & 1ull))) M += 1;",
                      "if (rem >= half) M += 1;"),
    # the wire rounding after a hop is dropped (sum kept in binary32)
    "no_hop_rounding": ("  return value_to_bits(wire, s);                             /* identity for binary32 */",
                        "  if (wire != ORC_F32) { uint32_t u; memcpy(&u, &s, 4); return (u + 0x8000u) >> 16; }\n"
                        "  return value_to_bits(wire, s);"),
    # the ingress cast truncates instead of rounding
    "ingress_truncates": ("  return value_to_bits(wire, bits_to_value(dtype, v));\n}\n\n/* Wire encoding -> storage",
                          "  return f32_bits(bits_to_value(dtype, v)) >> 16;\n}\n\n/* Wire encoding -> storage"),
    # the AllGather forwards the wrong chunk
    "ag_chunk": ("int cs = mod(l + shift - t, L);", "int cs = mod(l + shift + t, L);"),
    # the closed form folds the group sums starting at the last group
    "group_order": [("    for (int g = 0; g < G; g++) {\n      uint32_t acc = ingress(",
                     "    for (int g = G - 1; g >= 0; g--) {\n      uint32_t acc = ingress("),
                    ("      total = (g == 0) ? acc : orc_wire_add(wire, total, acc);",
                     "      total = (g == G - 1) ? acc : orc_wire_add(wire, total, acc);")],
    # the literal simulation chains the exchange from the last group down
    "exchange_chain": [("      sim_send(s, ORC_PHASE_XCHG, k, k * L + own, (k + 1) * L + own, c,",
                        "      sim_send(s, ORC_PHASE_XCHG, k, (G - 1 - k) * L + own, (G - 2 - k) * L + own, c,"),
                       ("      recv_add(s, (k + 1) * L + own, k * L + own, c,",
                        "      recv_add(s, (G - 2 - k) * L + own, (G - 1 - k) * L + own, c,"),
                       ("      sim_send(s, ORC_PHASE_XBCAST, g, (G - 1) * L + own, g * L + own, c,",
                        "      sim_send(s, ORC_PHASE_XBCAST, g, own, (g + 1) * L + own, c,"),
                       ("      recv_copy(s, g * L + own, (G - 1) * L + own, c,",
                        "      recv_copy(s, (g + 1) * L + own, own, c,")],
    # the traffic counter counts storage bytes instead of wire bytes
    "byte_count": ("  uint64_t bytes = (uint64_t)len * s->ew;", "  uint64_t bytes = (uint64_t)len * 4;"),
}

QUICK_PINS = [pin_schedule_r4, pin_fold_order_r3, pin_partition_r4_n10, pin_two_level,
              pin_ring_neighbours, pin_traffic, pin_small_integers, pin_r2_single_add,
              pin_composition, pin_allgather_concat, pin_literal_equals_closed_form,
              pin_two_level_closed_form]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    edits = MUTATIONS[name]
    if isinstance(edits, tuple):
        edits = [edits]
    src = oracle.source()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    lib = oracle.load(oracle.build_variant(src, str(tmp_path / "libvariant.so")))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for pin in QUICK_PINS:
        try:
            pin()
        except (AssertionError, RuntimeError):  # a failed check or an oracle error status
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_binary32_accumulation_is_more_accurate(dtype):
    """Ablation of the per-hop rounding: on gradient-like data, accumulating in
    binary32 and rounding once leaves a smaller error than rounding every hop,
    and never a larger one than half a unit of the storage format per element
    beyond the binary32 part."""
    rng = np.random.default_rng(21)
    R, N = 8, 50_000
    x32 = [(rng.standard_normal(N) * 1e-3).astype(np.float32) for _ in range(R)]
    if dtype == "f16":
        xs = [x.astype(np.float16).view(np.uint16) for x in x32]
    else:
        xs = [torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for x in x32]
    exact = np.sum([to_f64(x, dtype) for x in xs], axis=0)
    hop = to_f64(oracle.allreduce(xs, dtype).outs[0], dtype)
    acc = to_f64(oracle.allreduce(xs, dtype, "f32").outs[0], dtype)
    e_hop, e_acc = np.abs(hop - exact), np.abs(acc - exact)
    assert e_acc.mean() < 0.5 * e_hop.mean()
    # one final rounding of a value within (R-1) binary32 roundings of the exact sum
    ulp_half = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}[dtype]
    assert np.all(e_acc <= ulp_half * np.abs(exact) * 1.0001 + (R - 1) * 2.0 ** -24 * np.sum(
        [np.abs(to_f64(x, dtype)) for x in xs], axis=0) + 2.0 ** -25)
