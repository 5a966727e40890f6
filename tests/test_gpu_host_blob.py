"""GPU parity with page-locked host buffers (the host-blob mode).

On a Grace-Blackwell node the GPU reaches page-locked host memory over the
coherent host link, so the kernels can write a blob straight into host
memory while they code (a GPU tensor to a CPU blob with no separate copy)
and decode straight from it; sources and outputs may live there too. Blobs
made this way must equal the oracle's byte for byte, and decoding must be
exact, whichever side of the link each buffer is on. Unregistered host
memory is refused before any launch.
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
W_OF = {1: 1, 2: 2, 3: 4, 4: 2, 5: 2, 6: 4}


def _gauss_bytes(seed: int, n: int, dtype: int) -> np.ndarray:
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, generator=g) * 0.02
    t = {4: torch.bfloat16, 5: torch.float16, 6: torch.float32}[dtype]
    return x.to(t).view(torch.uint8).numpy().copy()


def _pinned(nbytes: int, fill: int) -> torch.Tensor:
    return torch.full((nbytes,), fill, dtype=torch.uint8).pin_memory()


@pytest.mark.parametrize("dtype,n,chunk,offset", [(4, 300_001, 131072, 0), (6, 70_000, 16384, 16),
                                                  (5, 1, 4096, 4096 + 16), (4, 0, 131072, 0)])
@pytest.mark.parametrize("src_on_host", [False, True])
def test_host_blob_matches_oracle(zco, dtype, n, chunk, offset, src_on_host):
    raw = _gauss_bytes(dtype * 7 + n, n, dtype)
    shape = (n,)
    nbytes = raw.size
    if src_on_host:
        src = _pinned(nbytes + 16, 0)[:nbytes]
        src.copy_(torch.from_numpy(raw))
    else:
        src = torch.from_numpy(raw).to(DEV)
    cap = zc.blob_size(nbytes, dtype, chunk, 0.95)
    hbuf = _pinned(cap + offset + 16, 0xAB)
    blob = hbuf[offset: offset + cap]
    nb = torch.zeros(1, dtype=torch.int64).pin_memory()
    ws = torch.full((max(16, zc.workspace_size(nbytes, dtype, chunk)),), 0x5A, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_into(src, blob, nb, ws, st, chunk, 0.95, dtype=dtype, shape=shape)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = blob[: int(nb.item())].numpy().tobytes()
    assert got == zco.compress(raw, dtype, shape, chunk, 0.95), "host blob differs from the oracle's"

    # decode straight from the host blob, into device memory and into host memory
    info = zc.blob_info(got)
    hb = blob[: int(nb.item())]
    for out_on_host in (False, True):
        out = _pinned(nbytes + 16, 0xCD)[:nbytes] if out_on_host else \
            torch.full((nbytes,), 0xCD, dtype=torch.uint8, device=DEV)
        st.zero_()
        zc.decompress_into(hb, info, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert out.cpu().numpy().tobytes() == raw.tobytes()


def test_host_blob_python_api():
    t = wl.bf16_1m(DEV)
    hb = zc.compress(t, host_blob=True)
    assert hb.device.type == "cpu" and hb.is_pinned()
    assert torch.equal(hb, zc.compress(t).cpu())
    back = zc.decompress(hb)
    assert back.is_cuda and torch.equal(back.view(torch.int16), t.view(torch.int16))


def test_host_blob_batch():
    specs = [s for s in wl.llama8b_specs(1) if s[0].startswith("layers.0.")][:4] + [("n", (4096,))]
    ts = [wl.llama8b_tensor(1 + i, nm, sh, DEV) for i, (nm, sh) in enumerate(specs)]
    hbs = zc.compress_batch(ts, host_blob=True)
    dbs = zc.compress_batch(ts)
    for h, d in zip(hbs, dbs):
        assert h.device.type == "cpu" and torch.equal(h, d.cpu())
    back = zc.decompress_batch(hbs)
    assert all(torch.equal(r.view(torch.int16), t.view(torch.int16)) for r, t in zip(back, ts))


def test_unregistered_host_memory_is_refused():
    """Pageable host memory is not mapped for the device: the library
    refuses it before any launch."""
    t = torch.zeros(1000, dtype=torch.bfloat16, device=DEV)
    cap = zc.blob_size(2000, wl.BF16)
    blob = torch.empty(cap, dtype=torch.uint8)  # pageable
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.empty(zc.workspace_size(2000, wl.BF16), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(zc.ZcError) as e:
        zc.compress_into(t.view(torch.uint8), blob, nb, ws, st)
    assert e.value.status == zc.EINVAL
    good = zc.compress(t)
    out = torch.empty(2000, dtype=torch.uint8)  # pageable
    with pytest.raises(zc.ZcError) as e:
        zc.decompress_into(good, zc.read_info(good), out, st)
    assert e.value.status == zc.EINVAL
