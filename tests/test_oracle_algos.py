"""Pins of the oracle's halving-doubling and naive AllReduce.

Same kinds of pins as the ring's: hand-derived values (tests/golden/algorithms.txt),
exact small-integer sums, the literal simulation against the closed form,
all outputs identical, message schedule and traffic, and planted mistakes.
"""
import os

import numpy as np
import pytest

import oracle
from test_oracle_ring import PAIRS, bits, golden_lines, hexarr, int_inputs, rand_inputs, to_f64

ALGOS = ("ring", "hd", "naive")
RS_ = [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 17, 31, 32, 33, 64]


def pin_golden_algorithms():
    for row in golden_lines("algorithms.txt"):
        algo, R = row[0], int(row[1])
        want = hexarr(" ".join(row[2:]).split("|")[1].split(), "f16")
        xs = [np.full(R, 0x3C00, np.uint16)] + [np.full(R, 0x1000, np.uint16) for _ in range(R - 1)]
        res = oracle.allreduce_algo(xs, "f16", algo=algo)
        assert res.status == oracle.OK
        for r in range(R):
            assert res.outs[r].tolist() == want.tolist(), (algo, R, r)


def pin_algo_closed_form():
    rng = np.random.default_rng(31)
    for algo in ("hd", "naive"):
        for R in RS_:
            for N in (1, 2, R - 1, R, R + 1, 3 * R + 5, 97):
                if N < 1:
                    continue
                for dtype, wire in PAIRS:
                    xs = rand_inputs(rng, R, N, dtype, special=True)
                    res = oracle.allreduce_algo(xs, dtype, wire, algo)
                    assert res.status == oracle.OK
                    cf = oracle.fold_gathered_algo(xs, np.arange(N), N, dtype, wire, algo)
                    for r in range(R):
                        assert bits(res.outs[r]).tolist() == bits(cf).tolist(), (algo, R, N, dtype, wire, r)


def pin_algo_integers():
    rng = np.random.default_rng(32)
    for algo in ("hd", "naive"):
        for R in (1, 2, 3, 5, 8, 12, 16):
            for dtype, wire in PAIRS:
                for N in (1, R, 2 * R + 1, 33):
                    xs = int_inputs(rng, R, N, dtype)
                    exact = sum(to_f64(x, dtype) for x in xs)
                    res = oracle.allreduce_algo(xs, dtype, wire, algo)
                    for r in range(R):
                        np.testing.assert_array_equal(to_f64(res.outs[r], dtype), exact)


def pin_algo_traffic_and_schedule():
    for R in RS_:
        N = 4 * R * 3
        xs = [np.zeros(N, np.float32) for _ in range(R)]
        S = 4 * N
        nv = oracle.allreduce_algo(xs, "f32", algo="naive", trace_cap=1 << 14)
        assert nv.sent_bytes == [(R - 1) * S] + [S] * (R - 1)  # the collector's link carries everything
        assert len(nv.trace) == 2 * (R - 1)
        hd = oracle.allreduce_algo(xs, "f32", algo="hd", trace_cap=1 << 14)
        P = 1
        while P * 2 <= R:
            P *= 2
        E, steps = R - P, P.bit_length() - 1
        rs = [m for m in hd.trace if m[0] == oracle.PHASE_RS]
        ag = [m for m in hd.trace if m[0] == oracle.PHASE_AG]
        assert len(rs) == len(ag) == P * steps  # logarithmic number of steps
        assert len([m for m in hd.trace if m[0] == oracle.PHASE_PRE]) == E
        assert len([m for m in hd.trace if m[0] == oracle.PHASE_POST]) == E
        vrank = {(2 * v + 1 if v < E else v + E): v for v in range(P)}
        for (_, t, src, dst, _, _) in rs:  # partners at distance P/2, P/4, ..., 1
            assert vrank[src] ^ vrank[dst] == P >> (t + 1)
        for (_, t, src, dst, _, _) in ag:  # and back: 1, 2, ..., P/2
            assert vrank[src] ^ vrank[dst] == 1 << t
        if E == 0 and N % R == 0:
            assert hd.sent_bytes == [2 * (R - 1) * S // R] * R  # the same volume as the ring


def ag_inputs(rng, R, N, dtype):
    """Chunk c of a random N-element vector, for c < R."""
    full = rand_inputs(rng, 1, N, dtype)[0]
    return full, [full[oracle.chunk_off(N, R, c):oracle.chunk_off(N, R, c) + oracle.chunk_len(N, R, c)].copy()
                  for c in range(R)]


def pin_allgather_schedules():
    """Every AllGather schedule delivers, to every rank, the chunks in place:
    out[r][off(c) + j] = in[c][j] (the definition, built here with numpy)."""
    rng = np.random.default_rng(35)
    for dtype in ("f32", "f16", "bf16"):
        for R in (1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 17):
            for N in (0, 1, R - 1, R, 4 * R + 3, 1001):
                full, chunks = ag_inputs(rng, R, N, dtype)
                for algo in ("ring", "hd", "naive"):
                    res = oracle.allgather_algo(chunks, N, dtype, algo)
                    assert res.status == oracle.OK, (dtype, R, N, algo, res.status)
                    for r in range(R):
                        assert bits(res.outs[r]).tolist() == bits(full).tolist(), (dtype, R, N, algo, r)


def pin_allgather_traffic_and_schedule():
    for R in RS_:
        N = 4 * R * 3
        full, chunks = ag_inputs(np.random.default_rng(R), R, N, "f32")
        S = 4 * N
        nv = oracle.allgather_algo(chunks, N, "f32", "naive", trace_cap=1 << 14)
        assert nv.sent_bytes == [(R - 1) * S] + [S // R] * (R - 1)  # chunks in, whole vectors out
        tr = oracle.allgather_algo(chunks, N, "f32", "hd", trace_cap=1 << 14)
        P = 1
        while P * 2 <= R:
            P *= 2
        E, steps = R - P, P.bit_length() - 1
        ag = [m for m in tr.trace if m[0] == oracle.PHASE_AG]
        assert len(ag) == P * steps  # log2(P) steps of P messages
        assert len([m for m in tr.trace if m[0] == oracle.PHASE_PRE]) == E
        assert len([m for m in tr.trace if m[0] == oracle.PHASE_POST]) == E
        vrank = {(2 * v + 1 if v < E else v + E): v for v in range(P)}
        for (_, t, src, dst, _, nbytes) in ag:  # partners 1, 2, 4, ... apart, each step doubling the data
            assert vrank[src] ^ vrank[dst] == 1 << t
            if E == 0:
                assert nbytes == (1 << t) * S // R
        if E == 0:
            assert tr.sent_bytes == [(R - 1) * S // R] * R  # the same volume as the ring AllGather


def test_allgather_schedules_deliver_the_definition():
    pin_allgather_schedules()


def test_allgather_traffic_and_schedule():
    pin_allgather_traffic_and_schedule()


def test_allgather_schedule_faults():
    full, chunks = ag_inputs(np.random.default_rng(36), 6, 600, "f32")
    r = oracle.allgather_algo(chunks, 600, "f32", "hd", fault=(oracle.FAULT_DROP, 1, oracle.PHASE_AG, 1))
    assert r.status == oracle.ETIMEOUT
    r = oracle.allgather_algo(chunks, 600, "f32", "naive", fault=(oracle.FAULT_DUP, 2, oracle.PHASE_RS, 1))
    assert r.status == oracle.EPROTO
    assert oracle.allgather_algo(chunks, 600, "f32", "hd").status == oracle.OK


def test_golden_algorithms():
    pin_golden_algorithms()


def test_algorithms_literal_equals_closed_form():
    pin_algo_closed_form()


def test_algorithms_small_integers_exact():
    pin_algo_integers()


def test_algorithms_traffic_and_schedule():
    pin_algo_traffic_and_schedule()


def test_algorithms_agree_for_two_ranks_and_outputs_identical():
    rng = np.random.default_rng(33)
    for dtype, wire in PAIRS:
        xs = rand_inputs(rng, 2, 501, dtype, special=True)
        outs = [oracle.allreduce_algo(xs, dtype, wire, a).outs for a in ALGOS]
        for o in outs[1:]:
            assert bits(o[0]).tolist() == bits(outs[0][0]).tolist()
        xs = rand_inputs(rng, 13, 301, dtype, special=True)
        for a in ALGOS:
            o = oracle.allreduce_algo(xs, dtype, wire, a).outs
            for r in range(1, 13):
                assert bits(o[r]).tolist() == bits(o[0]).tolist()


@pytest.mark.parametrize("algo", ["hd", "naive"])
def test_algorithms_error_bound(algo):
    rng = np.random.default_rng(34)
    R, N = 8, 20011
    xs = [(rng.standard_normal(N) * 1e-3).astype(np.float16).view(np.uint16) for _ in range(R)]
    x64 = [to_f64(x, "f16") for x in xs]
    exact, mag = np.sum(x64, axis=0), np.sum(np.abs(x64), axis=0)
    out = to_f64(oracle.allreduce_algo(xs, "f16", algo=algo).outs[0], "f16")
    assert np.all(np.abs(out - exact) <= R * 2.0 ** -10 * mag + (R - 1) * 2.0 ** -25)


def test_algorithm_faults_and_arguments():
    x = [np.ones(64, np.float32) for _ in range(6)]
    r = oracle.allreduce_algo(x, "f32", algo="hd", fault=(oracle.FAULT_DROP, 0, oracle.PHASE_PRE, 0))
    assert r.status == oracle.ETIMEOUT
    r = oracle.allreduce_algo(x, "f32", algo="naive", fault=(oracle.FAULT_DUP, 3, oracle.PHASE_RS, 2))
    assert r.status == oracle.EPROTO
    r = oracle.allreduce_algo(x, "f32", algo="hd", fault=(oracle.FAULT_SILENT, 5, oracle.PHASE_AG, 0))
    assert r.status == oracle.ETIMEOUT


MUTATIONS = {
    # halving starts with the nearest partner instead of the farthest
    "hd_partner_order": ("    const int d = P >> (t + 1);\n    int keep_lo[64], keep_hi[64];",
                         "    const int d = 1 << t;\n    int keep_lo[64], keep_hi[64];"),
    # the closed form pairs neighbours first
    "hd_closed_form_pairs": ("      for (int d = P / 2; d >= 1; d /= 2)\n        for (int v = 0; v < d; v++) leaf[v] = orc_wire_add(wire, leaf[v], leaf[v + d]);",
                             "      for (int d = 1; d < P; d *= 2)\n        for (int v = 0; v + d < P; v += 2 * d) leaf[v] = orc_wire_add(wire, leaf[v], leaf[v + d]);"),
    # the extra rank folds into the wrong neighbour
    "hd_fold_partner": ("static int hd_rank(int v, int E) { return v < E ? 2 * v + 1 : v + E; }",
                        "static int hd_rank(int v, int E) { return v < E ? 2 * v : v + E; }"),
    # the collector adds in reverse rank order
    "naive_order": ("      y = x[0];\n      for (int r = 1; r < R; r++) y = orc_wire_add(wire, y, x[r]);",
                    "      y = x[R - 1];\n      for (int r = R - 2; r >= 0; r--) y = orc_wire_add(wire, y, x[r]);"),
    # the tree AllGather starts with the farthest partner
    "tree_ag_partner_order": ("    const int d = 1 << t;\n    for (int v = 0; v < P; v++) {\n      const int c0 = tree_first_chunk",
                              "    const int d = P >> (t + 1);\n    for (int v = 0; v < P; v++) {\n      const int c0 = tree_first_chunk"),
    # the extra rank's chunk lands one chunk off
    "tree_ag_extra_chunk": ("static int tree_first_chunk(int v, int E) { return v < E ? 2 * v : v + E; }",
                            "static int tree_first_chunk(int v, int E) { return v < E ? 2 * v + 1 : v + E; }"),
    # the broadcast skips the last rank
    "naive_ag_broadcast": ("  for (int k = 1; k < R && s->status == ORC_OK; k++) { /* and sends the whole vector out */",
                           "  for (int k = 1; k < R - 1 && s->status == ORC_OK; k++) { /* and sends the whole vector out */"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_in_algorithms_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = oracle.source()
    assert src.count(old) == 1, name
    lib = oracle.load(oracle.build_variant(src.replace(old, new), str(tmp_path / "libvariant.so")))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for pin in (pin_golden_algorithms, pin_algo_closed_form, pin_algo_integers, pin_algo_traffic_and_schedule,
                pin_allgather_schedules, pin_allgather_traffic_and_schedule):
        try:
            pin()
        except (AssertionError, RuntimeError, KeyError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"
