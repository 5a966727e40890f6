"""zc_compress_noalloc: compression for callers that cannot allocate device
memory (their memory is owned by another allocator, or allocation is not
allowed after start-up). It runs the same compression as zc_compress on a
fixed scratch array inside the library, so its blobs must be byte-identical
to zc_compress's, and stay so on consecutive calls that reuse the array.

The test calls both entry points through the C ABI with ctypes.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import entropy_coding_gb300 as zc  # noqa: E402
from entropy_coding_gb300 import workloads as wl  # noqa: E402


def _noalloc_fn():
    f = zc.lib().zc_compress_noalloc
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [vp, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                  ctypes.c_uint32, ctypes.c_double, vp, ctypes.c_uint64, vp, vp, vp]
    return f


def _compress_noalloc(t: torch.Tensor, chunk: int, thr: float) -> bytes:
    src = wl.as_bytes(t)
    code = wl.dtype_code(t)
    cap = zc.blob_size(src.numel(), code, chunk, thr)
    blob = torch.full((cap,), 0x77, dtype=torch.uint8, device=t.device)
    nb = torch.zeros(1, dtype=torch.int64, device=t.device)
    st = torch.zeros(1, dtype=torch.int32, device=t.device)
    shape = (ctypes.c_int64 * max(1, t.dim()))(*t.shape)
    rc = _noalloc_fn()(src.data_ptr(), src.numel(), code, t.dim(), shape, chunk, thr, blob.data_ptr(), cap,
                       nb.data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return blob[: int(nb.item())].cpu().numpy().tobytes()


def _compress(t: torch.Tensor, chunk: int, thr: float) -> bytes:
    src = wl.as_bytes(t)
    code = wl.dtype_code(t)
    cap = zc.blob_size(src.numel(), code, chunk, thr)
    blob = torch.empty(cap, dtype=torch.uint8, device=t.device)
    ws = torch.empty(zc.workspace_size(src.numel(), code, chunk), dtype=torch.uint8, device=t.device)
    nb = torch.zeros(1, dtype=torch.int64, device=t.device)
    st = torch.zeros(1, dtype=torch.int32, device=t.device)
    zc.compress_into(src, blob, nb, ws, st, chunk, thr, dtype=code, shape=tuple(t.shape))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return blob[: int(nb.item())].cpu().numpy().tobytes()


def test_noalloc_matches_compress_on_consecutive_calls():
    dev = torch.device("cuda:0")
    cases = [(wl.fp32_64m(dev, rows=2048), 131072, 0.95),     # 64 MiB FP32, 512 chunks
             (wl.bf16_1m(dev), 131072, 0.95),
             (wl.bf16_1m(dev)[:200], 4096, 2.0)]
    # near the chunk limit: 2^20 - 1 chunks of 64 bytes, the last one ragged;
    # constant and random chunks, so both grouped and raw chunks appear. The
    # 8-byte status word per chunk then takes 8 MiB of the array, and the
    # statistics run in many waves
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    n = ((1 << 20) - 1) * 64 - 17
    many = torch.randint(0, 256, (n,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    many.view(-1)[: (n // 128) * 128].view(-1, 128)[:, :64] = 7
    cases.append((many, 64, 0.95))
    for t, chunk, thr in cases:
        ref = _compress(t, chunk, thr)
        first = _compress_noalloc(t, chunk, thr)
        second = _compress_noalloc(t, chunk, thr)
        assert first == ref
        assert second == ref
        back = zc.decompress(torch.frombuffer(bytearray(second), dtype=torch.uint8).to(dev))
        assert torch.equal(back.view(torch.uint8), t.view(torch.uint8))


def test_noalloc_checks_arguments_before_its_limit():
    """An invalid call is reported as invalid (ZC_EINVAL) whatever its size,
    and only a valid one beyond the chunk limit as ZC_ECAPACITY."""
    dev = torch.device("cuda:0")
    t = torch.zeros(16, dtype=torch.uint8, device=dev)
    nb = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    big = (1 << 20) * 64 + 64
    for nbytes, dtype, chunk in ((big, 1, 1), (big, 9, 64), (big + 1, 2, 64)):
        shape = (ctypes.c_int64 * 1)(nbytes)
        rc = _noalloc_fn()(t.data_ptr(), nbytes, dtype, 1, shape, chunk, 0.95, t.data_ptr(), 16,
                           nb.data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == zc.EINVAL, (nbytes, dtype, chunk, rc)


def test_noalloc_rejects_tensors_beyond_its_scratch():
    dev = torch.device("cuda:0")
    t = torch.zeros(16, dtype=torch.uint8, device=dev)
    nb = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    shape = (ctypes.c_int64 * 1)((1 << 20) * 64 + 64)
    # 2^20 + 1 chunks of 64 bytes: refused on the host before any launch
    rc = _noalloc_fn()(t.data_ptr(), (1 << 20) * 64 + 64, 1, 1, shape, 64, 0.95, t.data_ptr(), 16,
                       nb.data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == zc.ECAPACITY
