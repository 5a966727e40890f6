"""Every device wait of the library is bounded and reports ZC_ETIMEOUT
instead of hanging. Test hooks of the library make each wait run out on
purpose, with a short limit: the first chunk's offset is never published,
so the look-back waits of compression give up; the warp that runs a
chunk's rANS lanes stops before it signals, so its partner's barrier wait
in decompression gives up. The kernels must return, report the timeout in
the device status, and leave the context usable: a normal call afterwards
still matches the oracle byte for byte.
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


def _compress_status(t: torch.Tensor, flags: int = 0):
    src = wl.as_bytes(t)
    code = wl.dtype_code(t)
    cap = zc.blob_size(src.numel(), code, flags=flags)
    blob = torch.zeros(cap, dtype=torch.uint8, device=DEV)
    ws = torch.empty(zc.workspace_size(src.numel(), code, flags=flags), dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_into(src, blob, nb, ws, st, dtype=code, shape=tuple(t.shape), flags=flags)
    torch.cuda.synchronize()
    return int(st.item()), blob[: int(nb.item())]


@pytest.mark.parametrize("flags", [0, zc.SHARED_TABLES])
def test_lookback_wait_runs_out(zco, flags):
    t = wl.bf16_1m(DEV)[:256]   # 4 chunks of 128 KiB
    zc.set_test_hooks(zc.HOOK_LOOKBACK_STALL)
    try:
        st, _ = _compress_status(t, flags)
    finally:
        zc.set_test_hooks(0)
    assert st & zc.ETIMEOUT, st
    st, blob = _compress_status(t, flags)
    assert st == 0
    ref = zco.compress(wl.as_bytes(t).cpu().numpy(), wl.BF16, tuple(t.shape), version=2 if flags else 1)
    assert blob.cpu().numpy().tobytes() == ref


@pytest.mark.parametrize("flags", [0, zc.SHARED_TABLES])
def test_decoder_barrier_wait_runs_out(flags):
    t = wl.bf16_1m(DEV)
    blob = zc.compress(t, shared_tables=bool(flags))
    info = zc.read_info(blob)
    out = torch.empty_like(t)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.set_test_hooks(zc.HOOK_PRODUCER_STALL)
    try:
        zc.decompress_into(blob, info, out.view(torch.uint8).view(-1), st)
        torch.cuda.synchronize()
    finally:
        zc.set_test_hooks(0)
    assert int(st.item()) & zc.ETIMEOUT, int(st.item())
    assert torch.equal(zc.decompress(blob).view(torch.int16), t.view(torch.int16))
