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


def test_static_staging_rejects_pieces_beyond_its_size(rr):
    R = 64
    hin = host_inputs(R, 1024, torch.float32, seed=5)
    out = [torch.empty_like(t) for t in hin]
    largest = (32 << 20) // (3 * R * 4) // 256 * 256
    with pytest.raises(rr.RingError) as e:
        rr.allreduce_host_static(hin, out, piece_count=largest + 1)
    assert e.value.status == rr.ERR_INVALID_ARG
    rr.allreduce_host_static(hin, out, piece_count=largest)  # the largest piece fits
    torch.cuda.current_stream().synchronize()
