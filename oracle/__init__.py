"""CPU oracle of the ring AllReduce / ReduceScatter / AllGather (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never imports it and shares no code with it: the C sources in
this directory are a separate, single-threaded, literal simulation of the ring
(see ``ring_oracle.h`` for the sources it follows and the readings it takes).

Element conventions: ``"f32"`` arrays are ``numpy.float32``; ``"f16"`` and
``"bf16"`` arrays hold the 16-bit encodings as ``numpy.uint16``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ring_oracle.c")
_HDR = os.path.join(_HERE, "ring_oracle.h")
_LIB_PATH = os.path.join(_HERE, "libringoracle.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
NP_STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}

OK, EINVAL, EUNSUPPORTED, ENOMEM, EPROTO, ETIMEOUT = 0, 1, 2, 3, 4, 5
PHASE_RS, PHASE_XCHG, PHASE_XBCAST, PHASE_AG, PHASE_PRE, PHASE_POST = 0, 1, 2, 3, 4, 5
ALGO_RING, ALGO_HALVING_DOUBLING, ALGO_NAIVE = 0, 1, 2
ALGOS = {"ring": ALGO_RING, "hd": ALGO_HALVING_DOUBLING, "halving_doubling": ALGO_HALVING_DOUBLING,
         "naive": ALGO_NAIVE}
FAULT_NONE, FAULT_DROP, FAULT_DUP, FAULT_SILENT = 0, 1, 2, 3

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def _digest() -> str:
    """Digest of the oracle's sources, the gcc command line and the machine type."""
    h = hashlib.sha256()
    for f in (_SRC, _HDR):
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    h.update(" ".join(CFLAGS).encode() + platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile the oracle into ``libringoracle.so`` (gcc, plain C11).  A library
    is reused only when the digest recorded beside it (``.libringoracle.digest``)
    matches its sources, flags and machine type."""
    digest = _digest()
    stamp = os.path.join(_HERE, ".libringoracle.digest")
    if not force and os.path.exists(_LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    with open(stamp + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(stamp + f".tmp{os.getpid()}", stamp)
    return _LIB_PATH


class Msg(ctypes.Structure):
    _fields_ = [("phase", ctypes.c_int32), ("step", ctypes.c_int32), ("src", ctypes.c_int32),
                ("dst", ctypes.c_int32), ("chunk", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("bytes", ctypes.c_uint64)]


class Fault(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("rank", ctypes.c_int32), ("phase", ctypes.c_int32),
                ("step", ctypes.c_int32)]


class Opts(ctypes.Structure):
    _fields_ = [("sent_bytes", ctypes.POINTER(ctypes.c_uint64)), ("trace", ctypes.POINTER(Msg)),
                ("trace_cap", ctypes.c_size_t), ("trace_len", ctypes.c_size_t), ("fault", Fault),
                ("poll_limit", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load(path: str):
    """Load an oracle shared library from ``path`` and declare its C signatures."""
    L = ctypes.CDLL(path)
    vpp = ctypes.POINTER(ctypes.c_void_p)
    L.orc_allreduce.argtypes = [vpp, vpp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.POINTER(Opts)]
    L.orc_reduce_scatter.argtypes = [vpp, vpp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int,
                                     ctypes.c_int, ctypes.POINTER(Opts)]
    L.orc_allgather.argtypes = [vpp, vpp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int,
                                ctypes.POINTER(Opts)]
    L.orc_fold_gathered.argtypes = [vpp, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                    ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_void_p]
    for f in ("orc_allreduce", "orc_reduce_scatter", "orc_allgather", "orc_fold_gathered"):
        getattr(L, f).restype = ctypes.c_int
    L.orc_allreduce_algo.argtypes = [vpp, vpp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.POINTER(Opts)]
    L.orc_allreduce_algo.restype = ctypes.c_int
    L.orc_allgather_algo.argtypes = [vpp, vpp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(Opts)]
    L.orc_allgather_algo.restype = ctypes.c_int
    L.orc_fold_gathered_algo.argtypes = [vpp, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_size_t,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    L.orc_fold_gathered_algo.restype = ctypes.c_int
    L.orc_chunk_len.argtypes = [ctypes.c_size_t, ctypes.c_int, ctypes.c_int]
    L.orc_chunk_len.restype = ctypes.c_size_t
    L.orc_chunk_off.argtypes = [ctypes.c_size_t, ctypes.c_int, ctypes.c_int]
    L.orc_chunk_off.restype = ctypes.c_size_t
    L.orc_wire_add.argtypes = [ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32]
    L.orc_wire_add.restype = ctypes.c_uint32
    L.orc_f32_to_wire_batch.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_size_t]
    L.orc_f32_to_wire_batch.restype = None
    L.orc_wire_add_batch.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_size_t]
    L.orc_wire_add_batch.restype = None
    return L


def lib():
    """The oracle library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load(_LIB_PATH)
    return _lib


def build_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the tests that plant
    a mistake in the oracle and check that a pin catches it)."""
    d = os.path.dirname(out_path)
    c_path = os.path.join(d, "ring_oracle_variant.c")
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *CFLAGS, "-I", _HERE, "-o", out_path, c_path, "-lm"], check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def chunk_len(count: int, R: int, c: int) -> int:
    return int(lib().orc_chunk_len(count, R, c))


def chunk_off(count: int, R: int, c: int) -> int:
    return int(lib().orc_chunk_off(count, R, c))


def _ptrs(arrays):
    arr = (ctypes.c_void_p * len(arrays))()
    for k, a in enumerate(arrays):
        arr[k] = None if a is None or a.size == 0 else a.ctypes.data
    return arr


def _check(arrays, dtype):
    for a in arrays:
        if a is None:
            continue
        assert a.dtype == NP_STORAGE[dtype] and a.flags["C_CONTIGUOUS"], (a.dtype, dtype)


class Result:
    """Outputs of one simulated collective plus its transport record."""

    def __init__(self, status, outs, sent_bytes, trace):
        self.status = status
        self.outs = outs
        self.sent_bytes = sent_bytes
        self.trace = trace


def _opts(R, trace_cap, fault, poll_limit):
    o = Opts()
    sent = (ctypes.c_uint64 * R)()
    o.sent_bytes = ctypes.cast(sent, ctypes.POINTER(ctypes.c_uint64))
    tr = (Msg * max(trace_cap, 1))()
    o.trace = ctypes.cast(tr, ctypes.POINTER(Msg)) if trace_cap else None
    o.trace_cap = trace_cap
    if fault is not None:
        o.fault = Fault(*fault)
    o.poll_limit = poll_limit
    return o, sent, tr


def _finish(st, outs, o, sent, tr, R):
    trace = [(m.phase, m.step, m.src, m.dst, m.chunk, m.bytes)
             for m in tr[:min(o.trace_len, o.trace_cap)]] if o.trace_cap else None
    return Result(st, outs, [int(x) for x in sent[:R]], trace)


def allreduce(ins, dtype="f32", wire=None, group_size=0, trace_cap=0, fault=None, poll_limit=0,
              outs=None):
    """Literal ring AllReduce over len(ins) simulated ranks."""
    wire = wire or dtype
    R = len(ins)
    N = ins[0].size if R else 0
    _check(ins, dtype)
    if outs is None:
        outs = [np.empty(N, dtype=NP_STORAGE[dtype]) for _ in range(R)]
    o, sent, tr = _opts(R, trace_cap, fault, poll_limit)
    st = lib().orc_allreduce(_ptrs(ins), _ptrs(outs), R, N, DTYPES[dtype], DTYPES[wire],
                             group_size, ctypes.byref(o))
    return _finish(st, outs, o, sent, tr, R)


def reduce_scatter(ins, dtype="f32", wire=None, trace_cap=0, fault=None, poll_limit=0):
    """Literal ring ReduceScatter; outs[r] is chunk r."""
    wire = wire or dtype
    R = len(ins)
    N = ins[0].size if R else 0
    _check(ins, dtype)
    outs = [np.empty(chunk_len(N, R, r), dtype=NP_STORAGE[dtype]) for r in range(R)]
    o, sent, tr = _opts(R, trace_cap, fault, poll_limit)
    st = lib().orc_reduce_scatter(_ptrs(ins), _ptrs(outs), R, N, DTYPES[dtype], DTYPES[wire],
                                  ctypes.byref(o))
    return _finish(st, outs, o, sent, tr, R)


def allgather(ins, count, dtype="f32", trace_cap=0, fault=None, poll_limit=0):
    """Literal ring AllGather; ins[c] holds chunk c of a ``count``-element vector."""
    R = len(ins)
    _check(ins, dtype)
    outs = [np.empty(count, dtype=NP_STORAGE[dtype]) for _ in range(R)]
    o, sent, tr = _opts(R, trace_cap, fault, poll_limit)
    st = lib().orc_allgather(_ptrs(ins), _ptrs(outs), R, count, DTYPES[dtype], ctypes.byref(o))
    return _finish(st, outs, o, sent, tr, R)


def allgather_algo(ins, count, dtype="f32", algo="ring", trace_cap=0, fault=None, poll_limit=0):
    """Literal AllGather by schedule ("ring", "hd" = the tree / recursive doubling, "naive" =
    gather to rank 0 then broadcast); ins[c] holds chunk c of a ``count``-element vector."""
    R = len(ins)
    _check(ins, dtype)
    outs = [np.empty(count, dtype=NP_STORAGE[dtype]) for _ in range(R)]
    o, sent, tr = _opts(R, trace_cap, fault, poll_limit)
    st = lib().orc_allgather_algo(_ptrs(ins), _ptrs(outs), R, count, DTYPES[dtype], ALGOS[algo], ctypes.byref(o))
    return _finish(st, outs, o, sent, tr, R)


def allreduce_algo(ins, dtype="f32", wire=None, algo="ring", trace_cap=0, fault=None, poll_limit=0):
    """Literal AllReduce by algorithm ("ring", "hd" = halving-doubling, "naive")."""
    wire = wire or dtype
    R = len(ins)
    N = ins[0].size if R else 0
    _check(ins, dtype)
    outs = [np.empty(N, dtype=NP_STORAGE[dtype]) for _ in range(R)]
    o, sent, tr = _opts(R, trace_cap, fault, poll_limit)
    st = lib().orc_allreduce_algo(_ptrs(ins), _ptrs(outs), R, N, DTYPES[dtype], DTYPES[wire], ALGOS[algo],
                                  ctypes.byref(o))
    return _finish(st, outs, o, sent, tr, R)


def fold_gathered_algo(vals, idx, count, dtype="f32", wire=None, algo="ring"):
    """Closed form of allreduce_algo at global indices ``idx``."""
    wire = wire or dtype
    R = len(vals)
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    vals = [np.ascontiguousarray(v) for v in vals]
    _check(vals, dtype)
    out = np.empty(idx.size, dtype=NP_STORAGE[dtype])
    st = lib().orc_fold_gathered_algo(_ptrs(vals), idx.ctypes.data if idx.size else None, idx.size, R, count,
                                      DTYPES[dtype], DTYPES[wire], ALGOS[algo],
                                      out.ctypes.data if out.size else None)
    if st != OK:
        raise RuntimeError(f"orc_fold_gathered_algo failed with status {st}")
    return out


def fold_gathered(vals, idx, count, dtype="f32", wire=None, group_size=0):
    """Closed-form AllReduce result at global indices ``idx``; vals[r][k] is rank r's input there."""
    wire = wire or dtype
    R = len(vals)
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    vals = [np.ascontiguousarray(v) for v in vals]
    _check(vals, dtype)
    out = np.empty(idx.size, dtype=NP_STORAGE[dtype])
    st = lib().orc_fold_gathered(_ptrs(vals), idx.ctypes.data if idx.size else None, idx.size, R,
                                 count, DTYPES[dtype], DTYPES[wire], group_size,
                                 out.ctypes.data if out.size else None)
    if st != OK:
        raise RuntimeError(f"orc_fold_gathered failed with status {st}")
    return out


def f32_to_wire(x, wire):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.size, dtype=np.uint16)
    lib().orc_f32_to_wire_batch(DTYPES[wire], x.ctypes.data, out.ctypes.data, x.size)
    return out


def wire_add(a, b, wire):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(a.size, dtype=np.uint16)
    lib().orc_wire_add_batch(DTYPES[wire], a.ctypes.data, b.ctypes.data, out.ctypes.data, a.size)
    return out
