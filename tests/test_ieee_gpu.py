"""The GPU's rounding against the oracle's, over whole input spaces.

Through the C ABI, with the library's own kernels:
  * an AllReduce of one rank on a 16-bit wire (binary32 storage) is the
    ingress rounding followed by the exact widening back, so it runs the
    library's binary32 -> binary16 / bfloat16 conversion (CUDA's
    round-to-nearest-even intrinsics) on its input; all 2^32 binary32
    encodings go through it, on the direct path (16-byte vectors, paired
    conversions) and on the one-element path;
  * an AllReduce of two ranks with 16-bit storage and wire is one hop,
    a + b rounded once, for every element; all 2^32 pairs of 16-bit encodings
    go through it.
Each result is compared with the oracle's own bit-level conversion and hop
(pinned in turn to the compiler's casts and an exact binary64 sum by
tests/test_oracle_ieee.py).  NaN payloads are not compared: a NaN must stay
a NaN.  The host side runs the oracle on all cores, slice by slice.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

SLICE = 1 << 28  # elements per GPU call (1 GiB of binary32)
PIECE = 1 << 23  # elements per host task


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import ring_allreduce_reducescatter_gb300 as mod

    torch.cuda.set_device(0)
    return mod


def workers():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def is_nan16(u, ebits):
    mbits = 15 - ebits
    return ((u >> mbits) & ((1 << ebits) - 1) == (1 << ebits) - 1) & ((u & ((1 << mbits) - 1)) != 0)


def same16(got, want, ebits):
    """Bitwise equal, except that any NaN equals any NaN."""
    nan_g, nan_w = is_nan16(got, ebits), is_nan16(want, ebits)
    return ((got == want) & ~nan_g & ~nan_w) | (nan_g & nan_w)


def narrow_bits(out_f32, wire):
    """The 16-bit encoding of each (exactly widened) binary32 result."""
    if wire == "bf16":
        return (out_f32.view(np.uint32) >> 16).astype(np.uint16)
    return out_f32.astype(np.float16).view(np.uint16)  # exact: the values are binary16 values


def signed(t, bits):
    """Non-negative integers below 2^bits as the signed integers of the same bits."""
    return t - ((t >> (bits - 1)) & 1) * (1 << bits)


def run_slices(ex, slices, check):
    """For each slice, `slices` yields pieces (args of check) once the GPU work
    of the slice is done; the host checks one slice while the GPU runs the
    next, so at most two slices are held.  Returns the failure messages."""
    bad, pending = [], []
    for pieces in slices:
        futs = [ex.submit(check, *args) for args in pieces]
        for f in pending:
            r = f.result()
            if r:
                bad.append(r)
        pending = futs
    for f in pending:
        r = f.result()
        if r:
            bad.append(r)
    return bad


@pytest.mark.parametrize("wire", ["f16", "bf16"])
@pytest.mark.parametrize("path", ["direct", "simple"])
def test_ingress_rounding_every_binary32(rr, wire, path):
    cfg = rr.LaunchCfg(rr.PATH_DIRECT if path == "direct" else rr.PATH_SIMPLE)
    ebits = 8 if wire == "bf16" else 5
    x = torch.empty(SLICE, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)

    def check(lo, enc, got):
        want = oracle.f32_to_wire(enc.view(np.float32), wire)
        mine = narrow_bits(got, wire)
        ok = same16(mine, want, ebits)
        if not ok.all():
            k = int(np.flatnonzero(~ok)[0])
            return f"input {lo + k:#010x}: GPU {int(mine[k]):#06x}, oracle {int(want[k]):#06x}"
        return None

    def slices():
        for s0 in range(0, 1 << 32, SLICE):
            enc = signed(torch.arange(s0, s0 + SLICE, dtype=torch.int64, device="cuda"), 32).to(torch.int32)
            x.view(torch.int32).copy_(enc)
            rr.collective(rr.OP_ALLREDUCE, [x], [y], SLICE, wire, 0, None, cfg)
            got = y.cpu().numpy()
            enc_h = np.arange(SLICE, dtype=np.uint32) + np.uint32(s0)
            yield [(s0 + a, enc_h[a:a + PIECE], got[a:a + PIECE]) for a in range(0, SLICE, PIECE)]

    with ThreadPoolExecutor(workers()) as ex:
        bad = run_slices(ex, slices(), check)
    assert not bad, f"{wire} {path}: {len(bad)} pieces differ; " + "; ".join(bad[:4])
    assert rr.device_status() == 0


@pytest.mark.parametrize("wire", ["f16", "bf16"])
def test_hop_every_pair(rr, wire):
    dtype = torch.float16 if wire == "f16" else torch.bfloat16
    ebits = 8 if wire == "bf16" else 5
    a = torch.empty(SLICE, dtype=dtype, device="cuda")
    b = torch.empty_like(a)
    out = [torch.empty_like(a), torch.empty_like(a)]

    def check(lo, ah, bh, got):
        want = oracle.wire_add(ah, bh, wire)
        ok = same16(got, want, ebits)
        if not ok.all():
            k = int(np.flatnonzero(~ok)[0])
            return f"pair {lo + k:#010x}: GPU {int(got[k]):#06x}, oracle {int(want[k]):#06x}"
        return None

    def slices():
        for s0 in range(0, 1 << 32, SLICE):  # pair k = (k >> 16, k & 0xffff)
            k = torch.arange(s0, s0 + SLICE, dtype=torch.int64, device="cuda")
            a.view(torch.int16).copy_(signed(k >> 16, 16).to(torch.int16))
            b.view(torch.int16).copy_(signed(k & 0xFFFF, 16).to(torch.int16))
            del k
            rr.collective(rr.OP_ALLREDUCE, [a, b], out, SLICE, None, 0, None, None)
            assert torch.equal(out[0].view(torch.int16), out[1].view(torch.int16)), "the two outputs differ"
            got = out[0].view(torch.int16).cpu().numpy().view(np.uint16)
            idx = np.arange(SLICE, dtype=np.uint32)
            ah = ((idx >> 16) + np.uint32(s0 >> 16)).astype(np.uint16)
            bh = (idx & 0xFFFF).astype(np.uint16)
            del idx
            yield [(s0 + p, ah[p:p + PIECE], bh[p:p + PIECE], got[p:p + PIECE]) for p in range(0, SLICE, PIECE)]

    with ThreadPoolExecutor(workers()) as ex:
        bad = run_slices(ex, slices(), check)
    assert not bad, f"{wire} hop: {len(bad)} pieces differ; " + "; ".join(bad[:4])
    assert rr.device_status() == 0
