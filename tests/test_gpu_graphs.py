"""CUDA graphs and concurrent streams.

No entry point allocates device memory or synchronises, so a compression
and a decompression can be captured once in a CUDA graph and replayed on new
data in the same buffers; and calls with their own workspaces can run on
different streams at the same time. Both must give the blobs a plain call
gives (which the parity tests tie to the oracle).
"""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import entropy_coding_gb300 as zc  # noqa: E402
from entropy_coding_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda:0")


def _buffers(n_elems: int, dtype, code: int, flags: int = 0):
    nbytes = n_elems * torch.empty(0, dtype=dtype).element_size()
    return dict(
        src=torch.empty(nbytes, dtype=torch.uint8, device=DEV),
        blob=torch.zeros(zc.blob_size(nbytes, code, flags=flags), dtype=torch.uint8, device=DEV),
        ws=torch.empty(zc.workspace_size(nbytes, code, flags=flags), dtype=torch.uint8, device=DEV),
        nb=torch.zeros(1, dtype=torch.int64, device=DEV),
        st=torch.zeros(1, dtype=torch.int32, device=DEV),
        out=torch.empty(nbytes, dtype=torch.uint8, device=DEV),
    )


@pytest.mark.parametrize("flags", [0, zc.SHARED_TABLES])
def test_compress_and_decompress_replay_in_a_cuda_graph(flags):
    n = 1 << 20
    b = _buffers(n, torch.bfloat16, wl.BF16, flags)
    g = torch.Generator(device=DEV).manual_seed(11)
    first = (torch.randn(n, generator=g, device=DEV) * 0.02).bfloat16()
    b["src"].copy_(first.view(torch.uint8))
    # the header and chunk table are fixed by the shape, so one info serves
    # every replay; the capture needs it on the host before it starts
    ref = zc.compress(first, shared_tables=bool(flags))
    info = dict(zc.read_info(ref))
    # replays make blobs of other lengths: bound the decoder's reads by the
    # blob buffer instead of the first blob's length
    info["blob_bytes"] = b["blob"].numel()
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        zc.compress_into(b["src"], b["blob"], b["nb"], b["ws"], b["st"], dtype=wl.BF16, shape=(n,), stream=s,
                         flags=flags)  # warm-up outside the capture (function attributes, tables)
        zc.decompress_into(b["blob"], info, b["out"], b["st"], stream=s)
    s.synchronize()
    with torch.cuda.graph(graph, stream=s):
        zc.compress_into(b["src"], b["blob"], b["nb"], b["ws"], b["st"], dtype=wl.BF16, shape=(n,), stream=s,
                         flags=flags)
        zc.decompress_into(b["blob"], info, b["out"], b["st"], stream=s)
    for seed in (1, 2, 3):
        g.manual_seed(seed)
        x = (torch.randn(n, generator=g, device=DEV) * 0.02).bfloat16()
        b["src"].copy_(x.view(torch.uint8))
        b["st"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert int(b["st"].item()) == 0
        got = b["blob"][: int(b["nb"].item())]
        assert torch.equal(got, zc.compress(x, shared_tables=bool(flags))), seed
        assert torch.equal(b["out"], x.view(torch.uint8)), seed


def test_concurrent_streams_with_own_workspaces():
    tensors = [wl.llama8b_tensor(i + 1, "gate", (2048, 4096), DEV) for i in range(4)]
    refs = [zc.compress(t) for t in tensors]
    streams = [torch.cuda.Stream(device=DEV) for _ in tensors]
    bufs = [_buffers(t.numel(), torch.bfloat16, wl.BF16) for t in tensors]
    torch.cuda.synchronize()
    for t, b, s in zip(tensors, bufs, streams):
        b["src"].copy_(t.view(-1).view(torch.uint8))
    torch.cuda.synchronize()
    for t, b, s in zip(tensors, bufs, streams):
        zc.compress_into(b["src"], b["blob"], b["nb"], b["ws"], b["st"], dtype=wl.BF16, shape=tuple(t.shape),
                         stream=s)
    torch.cuda.synchronize()
    for r, b in zip(refs, bufs):
        assert int(b["st"].item()) == 0
        assert torch.equal(b["blob"][: int(b["nb"].item())], r)
