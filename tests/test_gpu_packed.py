"""ZC_PACKED (calls packed into few SMs, for calls on several streams at
once): the blobs are the oracle's byte for byte and decode exactly, in every
format, alone and with calls in flight on several streams.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import entropy_coding_gb300 as zc  # noqa: E402
from entropy_coding_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda:0")
FLAGS = {1: 0, 2: zc.SHARED_TABLES, 3: zc.LANE_WORDS}


def _run(src: torch.Tensor, dtype: int, shape, chunk: int, version: int, stream, ws: torch.Tensor):
    """Packed compression on `stream`, then packed decompression; returns the
    blob tensor, its length, the output and the two status words (not
    synchronised)."""
    flags = FLAGS[version] | zc.PACKED
    blob = torch.empty(zc.blob_size(src.numel(), dtype, chunk, 0.95, flags), dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    zc.compress_into(src, blob, nb, ws, st[0:1], chunk, 0.95, stream, dtype=dtype, shape=shape, flags=flags)
    return blob, nb, st


@pytest.mark.parametrize("version", [1, 2, 3])
def test_packed_blobs_match_oracle(zco, version):
    rng = np.random.default_rng(91)
    cases = [(wl.BF16, np.zeros(0, np.uint8), 4096),                       # empty
             (wl.BF16, wl.as_bytes(wl.bf16_1m("cpu")).numpy()[:2], 4096),  # one element
             (wl.U16, rng.integers(0, 256, 2 * 4097, dtype=np.uint8), 64),   # 129 chunks of 64 bytes, ragged
             (wl.BF16, wl.as_bytes(wl.bf16_1m("cpu")).numpy(), 4096),     # 512 chunks: many CTAs of 16
             (wl.FP32, wl.as_bytes(wl.fp32_64m("cpu", rows=32)).numpy(), 8192),
             (wl.FP16, wl.as_bytes(wl.fp16_16m("cpu", rows=64)).numpy(), 131072),
             (wl.U8, rng.integers(0, 16, 300_001, dtype=np.uint8), 65536)]
    stream = torch.cuda.Stream(device=DEV)
    for dtype, raw, chunk in cases:
        W = {wl.BF16: 2, wl.FP32: 4, wl.FP16: 2, wl.U8: 1, wl.U16: 2}[dtype]
        shape = (raw.size // W,)
        src = torch.from_numpy(raw.copy()).to(DEV) if raw.size else torch.empty(16, dtype=torch.uint8, device=DEV)[:0]
        ws = torch.empty(max(16, zc.workspace_size(raw.size, dtype, chunk, FLAGS[version])), dtype=torch.uint8,
                         device=DEV)
        stream.wait_stream(torch.cuda.current_stream())
        blob, nb, st = _run(src, dtype, shape, chunk, version, stream, ws)
        torch.cuda.synchronize()
        assert int(st[0].item()) == 0
        got = blob[: int(nb.item())]
        want = zco.compress(raw, dtype, shape, chunk, 0.95, version)
        assert got.cpu().numpy().tobytes() == want, (dtype, version)
        out = torch.empty_like(src)
        zc.decompress_into(got, zc.read_info(got), out, st[1:2], True, stream, packed=True)
        torch.cuda.synchronize()
        assert int(st[1].item()) == 0 and torch.equal(out, src), (dtype, version)


@pytest.mark.parametrize("version", [1, 3])
def test_packed_calls_on_several_streams(zco, version):
    """A Llama layer's tensors, one packed call each, issued round-robin on 4
    streams with a workspace per stream, as the benchmark issues them."""
    specs = wl.llama8b_specs()[1:10]
    streams = [torch.cuda.Stream(device=DEV) for _ in range(4)]
    srcs = [wl.as_bytes(wl.llama8b_tensor(i + 1, nm, sh, DEV)) for i, (nm, sh) in enumerate(specs)]
    ws_bytes = max(zc.workspace_size(s.numel(), wl.BF16, 131072, FLAGS[version]) for s in srcs)
    ws = [torch.empty(ws_bytes, dtype=torch.uint8, device=DEV) for _ in streams]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    runs = [_run(src, wl.BF16, tuple(sh), 131072, version, streams[k % 4], ws[k % 4])
            for k, (src, (_, sh)) in enumerate(zip(srcs, specs))]
    torch.cuda.synchronize()
    outs = []
    for k, ((blob, nb, st), src) in enumerate(zip(runs, srcs)):
        assert int(st[0].item()) == 0
        got = blob[: int(nb.item())]
        out = torch.empty_like(src)
        zc.decompress_into(got, zc.read_info(got), out, st[1:2], True, streams[k % 4], packed=True)
        outs.append((got, out))
    torch.cuda.synchronize()
    for (got, out), src, (blob, nb, st), (_, sh) in zip(outs, srcs, runs, specs):
        assert int(st[1].item()) == 0 and torch.equal(out, src)
        want = zco.compress(src.cpu().numpy(), wl.BF16, tuple(sh), 131072, 0.95, version)
        assert got.cpu().numpy().tobytes() == want


def test_packed_python_api():
    """compress(..., packed=True) makes the same blob as without, and
    decompress(..., packed=True) restores the tensor."""
    t = wl.llama8b_tensor(3, "layers.0.v", (1024, 4096), DEV)
    for kw in ({}, {"lane_words": True}, {"shared_tables": True}):
        a = zc.compress(t, **kw)
        b = zc.compress(t, packed=True, **kw)
        assert torch.equal(a, b), kw
        assert torch.equal(zc.decompress(b, packed=True).view(torch.int16), t.view(torch.int16)), kw
