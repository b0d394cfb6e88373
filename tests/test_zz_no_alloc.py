"""ring_allreduce_host_static against ring_allreduce_host, through the C ABI.

Some callers cannot give the library device memory for a workspace: code
loaded as a plugin into a program whose own allocator owns all of the GPU's
memory and hands out no raw buffers, or a latency-critical path that must not
risk an allocation failing or blocking while it runs.  ring_allreduce_host_static
serves them: it stages the pieces through a fixed block of device memory built
into the library instead of a caller workspace.  Its results must be those of
the workspace entry point, bit for bit, call after call (the block keeps the
previous call's contents).

This file is named so that pytest collects it last.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import ring_allreduce_reducescatter_gb300 as mod

    torch.cuda.set_device(0)
    return mod


def same_bits(a, b):
    view = torch.int16 if a.element_size() == 2 else torch.int32
    return torch.equal(a.view(view), b.view(view))


def host_inputs(R, N, dtype, seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return [(torch.randn(N, generator=g) * 1e-3).to(dtype).pin_memory() for _ in range(R)]


@pytest.mark.parametrize("dtype,wire,R,L,N,piece", [
    (torch.float16, None, 8, 0, 3_000_017, 0),          # the largest piece that fits
    (torch.float32, "bf16", 16, 8, 1_000_003, 4096),    # bf16 wire, two-level ring, many pieces
])
def test_static_staging_matches_workspace_entry_point(rr, dtype, wire, R, L, N, piece):
    ws = torch.empty(rr.host_workspace_bytes(R, 1 << 16, dtype), dtype=torch.uint8, device="cuda")
    for call in range(2):  # two calls in a row: the second finds the first call's data in the staging block
        hin = host_inputs(R, N, dtype, seed=1000 * call + R)
        want = [torch.empty_like(t).pin_memory() for t in hin]
        got = [torch.full_like(t, 7).pin_memory() for t in hin]
        rr.allreduce_host(hin, host_outs=want, workspace=ws, wire=wire, group_size=L)
        rr.allreduce_host_static(hin, got, wire=wire, group_size=L, piece_count=piece)
        torch.cuda.current_stream().synchronize()
        for r in range(R):
            assert same_bits(got[r], want[r]), f"call {call}, rank {r}"


def static_scratch_bytes():
    """RR_STATIC_SCRATCH_BYTES as the public header defines it."""
    import os
    import re

    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ringred.h")
    with open(header) as f:
        m = re.search(r"#define\s+RR_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", f.read())
    assert m, "RR_STATIC_SCRATCH_BYTES not found in ringred.h"
    return int(m.group(1)) << int(m.group(2))


def largest_static_piece(rr, R, dtype):
    """The largest piece_count whose three slots fit the staging array, found
    through the ABI's own workspace rule (ring_allreduce_host_workspace) by
    bisection, so the test follows the header's documented limit and not a
    copy of the library's internal constants."""
    limit = static_scratch_bytes()
    lo, hi = 0, limit  # workspace(lo) fits (or lo = 0), workspace(hi) does not
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if rr.host_workspace_bytes(R, mid, dtype) <= limit:
            lo = mid
        else:
            hi = mid
    return lo


@pytest.mark.parametrize("R,dtype", [(64, torch.float32), (8, torch.float16)])
def test_static_staging_rejects_pieces_beyond_its_size(rr, R, dtype):
    largest = largest_static_piece(rr, R, dtype)
    assert largest > 0
    N = 2 * largest + 1000  # three pieces at the largest size, the last one ragged
    hin = host_inputs(R, N, dtype, seed=5 + R)
    got = [torch.full_like(t, 7).pin_memory() for t in hin]
    with pytest.raises(rr.RingError) as e:
        rr.allreduce_host_static(hin, got, piece_count=largest + 1)
    assert e.value.status == rr.ERR_INVALID_ARG
    assert all(torch.equal(t, torch.full_like(t, 7)) for t in got)  # rejected before anything was written
    ws = torch.empty(rr.host_workspace_bytes(R, 1 << 16, dtype), dtype=torch.uint8, device="cuda")
    want = [torch.empty_like(t).pin_memory() for t in hin]
    rr.allreduce_host(hin, host_outs=want, workspace=ws)
    rr.allreduce_host_static(hin, got, piece_count=largest)  # the largest piece fits
    torch.cuda.current_stream().synchronize()
    for r in range(R):
        assert same_bits(got[r], want[r]), f"largest piece, rank {r}"


def test_static_staging_in_place(rr):
    """host_outs may be host_ins: the result replaces the inputs."""
    R, N, dtype = 8, 1_500_007, torch.bfloat16
    ws = torch.empty(rr.host_workspace_bytes(R, 1 << 16, dtype), dtype=torch.uint8, device="cuda")
    for call in range(2):
        hin = host_inputs(R, N, dtype, seed=77 + call)
        want = [torch.empty_like(t).pin_memory() for t in hin]
        rr.allreduce_host([t.clone() for t in hin], host_outs=want, workspace=ws)
        rr.allreduce_host_static(hin, hin, piece_count=65536 if call else 0)
        torch.cuda.current_stream().synchronize()
        for r in range(R):
            assert same_bits(hin[r], want[r]), f"in place, call {call}, rank {r}"
