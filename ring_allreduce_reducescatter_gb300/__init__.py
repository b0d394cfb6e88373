"""libringred: ring AllReduce / ReduceScatter / AllGather over R virtual ranks on one GPU.

This module is a thin ctypes binding of the C ABI in ``include/ringred.h``.  It
only marshals arguments (tensor lists to device-pointer arrays, the current
CUDA stream); every step of the collective runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  There is no fallback:
if ``libringred.so`` has not been built, importing the library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "RingError", "lib", "allreduce", "reduce_scatter", "allgather", "collective", "plan",
    "allreduce_range", "allreduce_host", "allreduce_host_static", "host_workspace_bytes", "allreduce_algo",
    "chunk_count", "chunk_offset", "device_status", "selftest_bounded_wait", "LaunchCfg", "rank_buffers",
    "debug_checks", "debug_set_margin", "HOST_COPIES_OVERLAP", "HOST_COPIES_ONE_WAY",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_ALIAS", "ERR_CUDA", "ERR_TIMEOUT",
    "OP_ALLREDUCE", "OP_REDUCE_SCATTER", "OP_ALLGATHER", "PATH_AUTO", "PATH_BULK", "PATH_SIMPLE", "PATH_DIRECT",
]

_DIR = os.path.dirname(os.path.abspath(__file__))
# RINGRED_LIBRARY names another build of the library to load instead (the
# debug build with device-side bounds checks, libringred_debug.so)
LIB_PATH = os.environ.get("RINGRED_LIBRARY") or os.path.join(_DIR, "libringred.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIAS, ERR_CUDA, ERR_TIMEOUT = range(6)
OP_ALLREDUCE, OP_REDUCE_SCATTER, OP_ALLGATHER = 0, 1, 2
PATH_AUTO, PATH_BULK, PATH_SIMPLE, PATH_DIRECT = 0, 1, 2, 3
FP32, FP16, BF16 = 0, 1, 2

_TORCH_CODE = {torch.float32: FP32, torch.float16: FP16, torch.bfloat16: BF16}
_NAME_CODE = {"f32": FP32, "fp32": FP32, "float32": FP32, "f16": FP16, "fp16": FP16,
              "float16": FP16, "bf16": BF16, "bfloat16": BF16}


RANK_STAGGER_BYTES = 2 << 20


def rank_buffers(R: int, count, dtype: torch.dtype, device=None, stagger_bytes: int = RANK_STAGGER_BYTES):
    """R rank vectors as views of one device allocation (plain torch memory;
    the library itself allocates nothing).  ``count`` is one length for every
    rank or a list of R lengths.  Each vector starts 256-byte aligned and
    ``stagger_bytes`` past the end of the one before.  Vectors whose start
    addresses agree modulo a large power of two (separate allocations of one
    power-of-two size, or rows of an unpadded [R, N] tensor) send all their
    concurrent accesses to the same memory channels: the R = 8, 512 MiB
    AllReduce ran about 2 % slower on them than on vectors staggered by
    1-17 MiB."""
    counts = [int(count)] * R if isinstance(count, int) else [int(c) for c in count]
    if len(counts) != R or min(counts, default=0) < 0:
        raise ValueError("need R non-negative lengths")
    e = torch.tensor([], dtype=dtype).element_size()
    if stagger_bytes < 0 or stagger_bytes % 256:
        raise ValueError("stagger_bytes must be a non-negative multiple of 256")
    offs, off = [], 0
    for c in counts:
        offs.append(off)
        off += (-(-c * e // 256) * 256 + stagger_bytes) // e
    slab = torch.empty(max(off, 1), dtype=dtype, device=device)
    return [slab[o:o + c] for o, c in zip(offs, counts)]


class RingError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.cuda_error = 0
        msg = f"{what}: {status_string(status)} (status {status})"
        if status == ERR_CUDA:
            self.cuda_error = int(lib().ring_last_cuda_error())
            msg += f": CUDA error {self.cuda_error}, {lib().ring_last_cuda_error_string().decode()}"
        super().__init__(msg)


class LaunchCfg(ctypes.Structure):
    """rr_launch_cfg: zero fields mean automatic."""

    _fields_ = [("path", ctypes.c_int), ("tile_bytes", ctypes.c_int), ("stages", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("threads", ctypes.c_int), ("max_ctas", ctypes.c_int),
                ("early_launch", ctypes.c_int), ("vectors", ctypes.c_int), ("beside_compute", ctypes.c_int),
                ("prefetch", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libringred.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vpp = ctypes.POINTER(ctypes.c_void_p)
        sz, i, vp = ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
        L.ring_collective.argtypes = [i, vpp, vpp, i, sz, i, i, i, ctypes.POINTER(LaunchCfg), vp]
        L.ring_plan.argtypes = [i, vpp, vpp, i, sz, i, i, i, ctypes.POINTER(LaunchCfg),
                                ctypes.POINTER(LaunchCfg)]
        L.ring_allreduce.argtypes = [vpp, vpp, i, sz, i, vp]
        L.ring_allreduce_ex.argtypes = [vpp, vpp, i, sz, i, i, i, vp]
        L.ring_reduce_scatter.argtypes = [vpp, vpp, i, sz, i, vp]
        L.ring_reduce_scatter_ex.argtypes = [vpp, vpp, i, sz, i, i, vp]
        L.ring_allgather.argtypes = [vpp, vpp, i, sz, i, vp]
        for f in ("ring_collective", "ring_plan", "ring_allreduce", "ring_allreduce_ex",
                  "ring_reduce_scatter", "ring_reduce_scatter_ex", "ring_allgather",
                  "ring_device_status", "ring_selftest_bounded_wait"):
            getattr(L, f).restype = i
        L.ring_allreduce_algo.argtypes = [vpp, vpp, i, sz, i, i, i, ctypes.POINTER(LaunchCfg), vp]
        L.ring_allreduce_algo.restype = i
        L.ring_allreduce_range.argtypes = [vpp, vpp, i, sz, sz, sz, i, i, i, ctypes.POINTER(LaunchCfg), vp]
        L.ring_allreduce_range.restype = i
        L.ring_allreduce_host.argtypes = [vpp, vpp, i, sz, i, i, i, vp, sz, vp]
        L.ring_allreduce_host.restype = i
        L.ring_allreduce_host_ex.argtypes = [vpp, vpp, i, sz, i, i, i, vp, sz, i, vp]
        L.ring_allreduce_host_ex.restype = i
        L.ring_allreduce_host_static.argtypes = [vpp, vpp, i, sz, i, i, i, sz, vp]
        L.ring_allreduce_host_static.restype = i
        L.ring_allreduce_host_workspace.argtypes = [i, sz, i]
        L.ring_allreduce_host_workspace.restype = sz
        L.ring_chunk_count.argtypes = [sz, i, i]
        L.ring_chunk_count.restype = sz
        L.ring_chunk_offset.argtypes = [sz, i, i]
        L.ring_chunk_offset.restype = sz
        L.ring_status_string.argtypes = [i]
        L.ring_status_string.restype = ctypes.c_char_p
        L.ring_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.ring_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, vp]
        L.ring_abi_version.argtypes = []
        L.ring_abi_version.restype = i
        L.ring_last_cuda_error.argtypes = []
        L.ring_last_cuda_error.restype = i
        L.ring_last_cuda_error_string.argtypes = []
        L.ring_last_cuda_error_string.restype = ctypes.c_char_p
        L.ring_debug_checks.argtypes = []
        L.ring_debug_checks.restype = i
        L.ring_debug_set_margin.argtypes = [sz]
        L.ring_debug_set_margin.restype = i
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ring_status_string(status).decode()


def chunk_count(count: int, R: int, c: int) -> int:
    return int(lib().ring_chunk_count(count, R, c))


def chunk_offset(count: int, R: int, c: int) -> int:
    return int(lib().ring_chunk_offset(count, R, c))


def _code(t) -> int:
    if isinstance(t, torch.dtype):
        return _TORCH_CODE[t]
    if isinstance(t, str):
        return _NAME_CODE[t.lower()]
    return int(t)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _ptr_array(tensors: Sequence[Optional[torch.Tensor]]):
    arr = (ctypes.c_void_p * len(tensors))()
    for k, t in enumerate(tensors):
        arr[k] = None if t is None or t.numel() == 0 else t.data_ptr()
    return arr


def _check_tensors(ts, dtype, name):
    for t in ts:
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
            raise ValueError(f"{name}: every buffer must be a CUDA tensor")
        if t.dtype != dtype:
            raise ValueError(f"{name}: mixed dtypes ({t.dtype} vs {dtype})")
        if not t.is_contiguous():
            raise ValueError(f"{name}: buffers must be contiguous")


def collective(op: int, ins, outs, count: int, wire=None, group_size: int = 0, stream=None,
               cfg: Optional[LaunchCfg] = None) -> None:
    """ring_collective on tensor lists (outputs preallocated by the caller)."""
    dtype = next(t.dtype for t in list(ins) + list(outs) if t is not None)
    _check_tensors(ins, dtype, "ins")
    _check_tensors(outs, dtype, "outs")
    if len(ins) != len(outs):
        raise ValueError("ins and outs must have one buffer per rank")
    dt = _code(dtype)
    wt = dt if wire is None else _code(wire)
    st = lib().ring_collective(op, _ptr_array(ins), _ptr_array(outs), len(ins), count, dt, wt,
                               group_size, ctypes.byref(cfg) if cfg is not None else None,
                               _stream_handle(stream))
    if st != OK:
        raise RingError(st, "ring_collective")


def plan(op: int, ins, outs, count: int, wire=None, group_size: int = 0,
         cfg: Optional[LaunchCfg] = None) -> dict:
    """The launch configuration ring_collective would pick (ring_plan)."""
    dtype = next(t.dtype for t in list(ins) + list(outs) if t is not None)
    dt = _code(dtype)
    wt = dt if wire is None else _code(wire)
    chosen = LaunchCfg()
    st = lib().ring_plan(op, _ptr_array(ins), _ptr_array(outs), len(ins), count, dt, wt, group_size,
                         ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(chosen))
    if st != OK:
        raise RingError(st, "ring_plan")
    return chosen.as_dict()


def allreduce(ins: Sequence[torch.Tensor], outs: Optional[Sequence[torch.Tensor]] = None, wire=None,
              group_size: int = 0, stream=None, cfg: Optional[LaunchCfg] = None):
    """Ring AllReduce; ``outs`` defaults to new tensors (pass ``ins`` for in place)."""
    ins = list(ins)
    if outs is None:
        outs = [torch.empty_like(t) for t in ins]
    collective(OP_ALLREDUCE, ins, list(outs), ins[0].numel(), wire, group_size, stream, cfg)
    return outs


def reduce_scatter(ins: Sequence[torch.Tensor], outs: Optional[Sequence[torch.Tensor]] = None,
                   wire=None, stream=None, cfg: Optional[LaunchCfg] = None):
    """Ring ReduceScatter: outs[r] receives chunk r (chunk_count(N, R, r) elements)."""
    ins = list(ins)
    R, N = len(ins), ins[0].numel()
    if outs is None:
        outs = [torch.empty(chunk_count(N, R, r), dtype=ins[0].dtype, device=ins[0].device)
                for r in range(R)]
    collective(OP_REDUCE_SCATTER, ins, list(outs), N, wire, 0, stream, cfg)
    return outs


def allgather(ins: Sequence[torch.Tensor], count: Optional[int] = None,
              outs: Optional[Sequence[torch.Tensor]] = None, stream=None,
              cfg: Optional[LaunchCfg] = None):
    """Ring AllGather: ins[c] is chunk c of a ``count``-element vector."""
    ins = list(ins)
    if count is None:
        count = sum(t.numel() for t in ins)
    ref = next(t for t in ins if t is not None)
    if outs is None:
        outs = [torch.empty(count, dtype=ref.dtype, device=ref.device) for _ in ins]
    collective(OP_ALLGATHER, ins, list(outs), count, None, 0, stream, cfg)
    return outs


ALGO_RING, ALGO_HALVING_DOUBLING, ALGO_NAIVE = 0, 1, 2
_ALGO_CODE = {"ring": ALGO_RING, "hd": ALGO_HALVING_DOUBLING, "halving_doubling": ALGO_HALVING_DOUBLING,
              "naive": ALGO_NAIVE}


def allreduce_algo(ins, outs=None, wire=None, algo="ring", stream=None, cfg: Optional[LaunchCfg] = None):
    """ring_allreduce_algo: the AllReduce summed in the order of another algorithm
    ("ring", "hd" = halving-doubling, "naive" = Reduce + Broadcast)."""
    ins = list(ins)
    if outs is None:
        outs = [torch.empty_like(t) for t in ins]
    outs = list(outs)
    dtype = ins[0].dtype
    _check_tensors(ins, dtype, "ins")
    _check_tensors(outs, dtype, "outs")
    dt = _code(dtype)
    wt = dt if wire is None else _code(wire)
    code = _ALGO_CODE[algo] if isinstance(algo, str) else int(algo)
    st = lib().ring_allreduce_algo(_ptr_array(ins), _ptr_array(outs), len(ins), ins[0].numel(), dt, wt, code,
                                   ctypes.byref(cfg) if cfg is not None else None, _stream_handle(stream))
    if st != OK:
        raise RingError(st, "ring_allreduce_algo")
    return outs


def allreduce_range(ins, outs, count: int, first: int, wire=None, group_size: int = 0, stream=None,
                    cfg: Optional[LaunchCfg] = None) -> None:
    """ring_allreduce_range: ins[r] / outs[r] hold elements [first, first + n) of
    rank r's count-element vector; outs receive those elements of the AllReduce."""
    ins, outs = list(ins), list(outs)
    dtype = ins[0].dtype
    _check_tensors(ins, dtype, "ins")
    _check_tensors(outs, dtype, "outs")
    dt = _code(dtype)
    wt = dt if wire is None else _code(wire)
    st = lib().ring_allreduce_range(_ptr_array(ins), _ptr_array(outs), len(ins), count, first, ins[0].numel(), dt,
                                    wt, group_size, ctypes.byref(cfg) if cfg is not None else None,
                                    _stream_handle(stream))
    if st != OK:
        raise RingError(st, "ring_allreduce_range")


def host_workspace_bytes(R: int, piece_count: int, dtype) -> int:
    return int(lib().ring_allreduce_host_workspace(R, piece_count, _code(dtype)))


def _check_host_buffers(host_ins, host_outs):
    """The host-buffer entry points copy count * element-size bytes per rank
    to and from the given addresses, and the C ABI cannot see how large a host
    buffer is, so every size is checked here: one input and one output per
    rank, all contiguous CPU tensors of one dtype holding exactly N elements.
    Returns (R, N)."""
    if not host_ins:
        raise ValueError("host_ins: need at least one rank")
    R, N, dtype = len(host_ins), host_ins[0].numel(), host_ins[0].dtype
    if len(host_outs) != R:
        raise ValueError(f"host_outs: {len(host_outs)} buffers for {R} ranks")
    for name, ts in (("host_ins", host_ins), ("host_outs", host_outs)):
        for r, t in enumerate(ts):
            if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or not t.is_contiguous():
                raise ValueError(f"{name}[{r}]: every buffer must be a contiguous CPU tensor")
            if t.dtype != dtype:
                raise ValueError(f"{name}[{r}]: dtype {t.dtype}, expected {dtype}")
            if t.numel() != N:
                raise ValueError(f"{name}[{r}]: {t.numel()} elements, expected {N}")
    return R, N


HOST_COPIES_OVERLAP, HOST_COPIES_ONE_WAY = 0, 1


def allreduce_host(host_ins, host_outs=None, workspace: Optional[torch.Tensor] = None, wire=None,
                   group_size: int = 0, stream=None, piece_count: int = 1 << 24, copy_mode: Optional[int] = None):
    """ring_allreduce_host: CPU tensors in and out (page-locked for overlap),
    pipelined through a device workspace (allocated here if not given).
    copy_mode (HOST_COPIES_OVERLAP / HOST_COPIES_ONE_WAY) calls
    ring_allreduce_host_ex with that copy schedule."""
    host_ins = list(host_ins)
    if host_outs is None:
        host_outs = [torch.empty_like(t, pin_memory=t.is_pinned()) for t in host_ins]
    host_outs = list(host_outs)
    R, N = _check_host_buffers(host_ins, host_outs)
    dtype = host_ins[0].dtype
    if workspace is None:
        nbytes = host_workspace_bytes(R, min(piece_count, max(N, 1)), dtype)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=torch.cuda.current_device())
    dt = _code(dtype)
    wt = dt if wire is None else _code(wire)
    hin = (ctypes.c_void_p * R)(*[t.data_ptr() for t in host_ins])
    hout = (ctypes.c_void_p * R)(*[t.data_ptr() for t in host_outs])
    if copy_mode is None:
        st = lib().ring_allreduce_host(hin, hout, R, N, dt, wt, group_size, workspace.data_ptr(), workspace.numel(),
                                       _stream_handle(stream))
    else:
        st = lib().ring_allreduce_host_ex(hin, hout, R, N, dt, wt, group_size, workspace.data_ptr(),
                                          workspace.numel(), int(copy_mode), _stream_handle(stream))
    if st != OK:
        raise RingError(st, "ring_allreduce_host" if copy_mode is None else "ring_allreduce_host_ex")
    return host_outs


def allreduce_host_static(host_ins, host_outs, wire=None, group_size: int = 0, piece_count: int = 0,
                          stream=None) -> None:
    """ring_allreduce_host_static: like allreduce_host, but the pieces go through
    staging memory built into the library, so nothing is allocated (host_outs
    must be given; it may be host_ins for in place)."""
    host_ins, host_outs = list(host_ins), list(host_outs)
    R, N = _check_host_buffers(host_ins, host_outs)
    dtype = host_ins[0].dtype
    dt = _code(dtype)
    wt = dt if wire is None else _code(wire)
    hin = (ctypes.c_void_p * R)(*[t.data_ptr() for t in host_ins])
    hout = (ctypes.c_void_p * R)(*[t.data_ptr() for t in host_outs])
    st = lib().ring_allreduce_host_static(hin, hout, R, N, dt, wt, group_size, piece_count,
                                          _stream_handle(stream))
    if st != OK:
        raise RingError(st, "ring_allreduce_host_static")


def debug_checks() -> bool:
    """True when the loaded library is the debug build (device-side bounds checks)."""
    return bool(lib().ring_debug_checks())


def debug_set_margin(nbytes: int) -> None:
    """Debug build: the checks treat every buffer as nbytes shorter (0 restores)."""
    st = lib().ring_debug_set_margin(nbytes)
    if st != OK:
        raise RingError(st, "ring_debug_set_margin")


def device_status() -> int:
    """Read and clear the current device's sticky status word (synchronizes the device)."""
    v = ctypes.c_uint(0)
    st = lib().ring_device_status(ctypes.byref(v))
    if st != OK:
        raise RingError(st, "ring_device_status")
    return int(v.value)


def selftest_bounded_wait(limit_ns: int, stream=None) -> int:
    """Run the bounded-wait self test; returns its status (ERR_TIMEOUT is the expected one)."""
    return int(lib().ring_selftest_bounded_wait(limit_ns, _stream_handle(stream)))
