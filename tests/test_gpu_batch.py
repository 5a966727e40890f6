"""GPU parity of the batched calls (zc_compress_batch, zc_decompress_batch).

A batch codes the chunks of many tensors in one grid; each tensor's blob
must still equal the oracle's blob of that tensor alone, byte for byte, and
decoding a batch must restore every tensor exactly. Cases: ragged and empty
tensors at any position of the list, tensors smaller than a chunk, several
hundred tensors (the descriptor tables then take more than one upload
launch), a workspace small enough to split the batch into waves whose
boundaries fall inside tensors, XOR-delta batches, and a Llama-3.1-8B
layer's tensors against one call per tensor.
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


def _tensor_bytes(rng, dtype: int, n: int) -> np.ndarray:
    """n words of dtype: Gaussian floats (several scales), small integers,
    constants or uniform bytes."""
    W = W_OF[dtype]
    if n == 0:
        return np.zeros(0, np.uint8)
    kind = int(rng.integers(0, 4))
    if kind == 0:
        return rng.integers(0, 256, n * W, dtype=np.uint8)
    if kind == 1:
        return np.full(n * W, rng.integers(0, 256), np.uint8)
    if dtype in (1, 2, 3):
        return rng.integers(0, 16, n * W, dtype=np.uint8)
    x = torch.from_numpy((rng.standard_normal(n) * float(rng.choice([0.02, 1.0, 1e-3]))).astype(np.float32))
    t = {4: torch.bfloat16, 5: torch.float16, 6: torch.float32}[dtype]
    return x.to(t).view(torch.uint8).numpy().copy()


def _batch(raws, dtype, chunk, thr, ws_bytes=None, bases=None):
    """Compress host byte arrays in one batched call; returns the blobs' bytes."""
    n = len(raws)
    W = W_OF[dtype]
    srcs = [torch.from_numpy(r).to(DEV) for r in raws]
    bs = [torch.from_numpy(b).to(DEV) for b in bases] if bases is not None else None
    blobs = [torch.full((zc.blob_size(r.size, dtype, chunk, thr),), 0xAB, dtype=torch.uint8, device=DEV)
             for r in raws]
    full = zc.workspace_size_batch([r.size for r in raws], dtype, chunk)
    assert full > 0
    ws = torch.full((ws_bytes or full,), 0x5A, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(n, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_batch_into(srcs, blobs, nb, ws, st, dtype, [(r.size // W,) for r in raws], chunk, thr, bases=bs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return [b[:k].cpu().numpy().tobytes() for b, k in zip(blobs, nb.tolist())]


def _unbatch(blobs, verify=True, bases=None):
    """Decompress blobs (host bytes) in one batched call; returns host bytes."""
    infos = [zc.blob_info(b) for b in blobs]
    dev_blobs = [torch.from_numpy(np.frombuffer(b, np.uint8).copy()).to(DEV) for b in blobs]
    outs = [torch.full((d["nbytes"],), 0xCD, dtype=torch.uint8, device=DEV) for d in infos]
    bs = [torch.from_numpy(b).to(DEV) for b in bases] if bases is not None else None
    n_ws = zc.decompress_workspace_size_batch(len(blobs))
    ws = torch.full((n_ws,), 0x77, dtype=torch.uint8, device=DEV) if n_ws else None
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.decompress_batch_into(dev_blobs, infos, outs, st, ws, verify, bases=bs)
    torch.cuda.synchronize()
    return int(st.item()), [o.cpu().numpy().tobytes() for o in outs]


def _check(zco, raws, dtype, chunk, thr, ws_bytes=None):
    W = W_OF[dtype]
    got = _batch(raws, dtype, chunk, thr, ws_bytes)
    for t, (r, g) in enumerate(zip(raws, got)):
        ref = zco.compress(r, dtype, (r.size // W,), chunk, thr)
        assert g == ref, f"tensor {t} ({r.size} B): batched blob differs from the oracle's"
    for verify in (True, False):
        st, back = _unbatch(got, verify)
        assert st == 0
        assert all(b == r.tobytes() for b, r in zip(back, raws))
    return got


@pytest.mark.parametrize("dtype,chunk,thr", [(4, 131072, 0.95), (6, 65536, 0.95), (5, 4096, 0.95),
                                             (1, 4096, 2.0), (3, 8192, 0.5)])
def test_batch_matches_oracle(zco, dtype, chunk, thr):
    rng = np.random.default_rng(100 + dtype)
    W = W_OF[dtype]
    words = chunk // W
    sizes = [0, 3 * words + 17, 1, words, 0, 0, words - 1, 5 * words, 2 * words + 1, 0]
    _check(zco, [_tensor_bytes(rng, dtype, n) for n in sizes], dtype, chunk, thr)


def test_batch_of_single_and_all_empty(zco):
    rng = np.random.default_rng(7)
    _check(zco, [_tensor_bytes(rng, 4, 40_000)], 4, 16384, 0.95)
    _check(zco, [np.zeros(0, np.uint8)] * 3, 4, 16384, 0.95)


def test_batch_many_tensors(zco):
    """700 tensors: both descriptor tables span several upload launches and the
    chunks of many tensors share each coding wave."""
    rng = np.random.default_rng(11)
    sizes = [int(s) for s in rng.integers(0, 9000, 700)]
    sizes[::37] = [0] * len(sizes[::37])
    _check(zco, [_tensor_bytes(rng, 4, n) for n in sizes], 4, 4096, 0.95)


def test_batch_small_workspace_waves(zco):
    """A workspace that holds a few chunks of statistics: waves end inside
    tensors and each tensor's offset scan carries across them."""
    rng = np.random.default_rng(13)
    dtype, chunk, W = 6, 4096, 4
    raws = [_tensor_bytes(rng, dtype, n) for n in (9000, 0, 1500, 30000, 100, 12000)]
    nc = sum((r.size + chunk - 1) // chunk for r in raws)
    n_pad = (chunk // W + 31) // 32 * 32
    per_chunk = 32 + W * (512 + n_pad)
    ctrl = 256 + (16 * len(raws) + 255) // 256 * 256
    table = (152 * len(raws) + 255) // 256 * 256
    small = ctrl + table + (8 * nc + 255) // 256 * 256 + 3 * per_chunk + 1024 + 2 * W * (2 * chunk // W + 4096)
    assert small < zc.workspace_size_batch([r.size for r in raws], dtype, chunk)
    _check(zco, raws, dtype, chunk, 0.95, ws_bytes=small)


def test_batch_delta_matches_oracle(zco):
    rng = np.random.default_rng(17)
    bases, news = [], []
    for n in (70_000, 0, 1, 131072, 200_003):
        a = rng.integers(0, 1 << 16, n, dtype=np.uint16)
        b = a.copy()
        k = rng.random(n) < 0.1
        b[k] ^= rng.integers(1, 64, int(k.sum()), dtype=np.uint16)
        bases.append(a.view(np.uint8))
        news.append(b.view(np.uint8))
    got = _batch(news, 2, 131072, 0.95, bases=bases)
    for a, b, g in zip(bases, news, got):
        ref = zco.compress(a ^ b, 2, (a.size // 2,), 131072, 0.95)
        assert g == ref
    st, back = _unbatch(got, bases=bases)
    assert st == 0 and all(x == b.tobytes() for x, b in zip(back, news))


def test_batch_llama_layer_equals_single_calls(zco):
    """One Llama-3.1-8B layer (q, k, v, o, gate, up, down, two RMSNorm
    vectors) compressed in one batch: every blob equals the single-call blob,
    the small tensors equal the oracle's, and decoding restores all exactly."""
    specs = [s for s in wl.llama8b_specs(1) if s[0].startswith("layers.0.")]
    ts = [wl.llama8b_tensor(1 + i, nm, shape, DEV) for i, (nm, shape) in enumerate(specs)]
    blobs = zc.compress_batch(ts)
    for (nm, shape), t, b in zip(specs, ts, blobs):
        single = zc.compress(t)
        assert torch.equal(b, single), f"{nm}: batched blob differs from the single-call blob"
        if t.numel() <= 1024 * 4096:
            raw = wl.as_bytes(t.cpu()).numpy()
            assert b.cpu().numpy().tobytes() == zco.compress(raw, 4, tuple(shape), 131072, 0.95), nm
    back = zc.decompress_batch(blobs)
    for t, r in zip(ts, back):
        assert r.dtype == t.dtype and r.shape == t.shape
        assert torch.equal(r.view(torch.int16), t.view(torch.int16))


def test_batch_python_api_delta_round_trip():
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    bases = [(torch.randn(n, generator=g, device=DEV) * 0.02).bfloat16() for n in (5000, 0, 300_000)]
    news = [(b.float() + torch.randn(b.shape, generator=g, device=DEV) * 1e-4).bfloat16() for b in bases]
    blobs = zc.compress_batch(news, bases=bases)
    for b, n, blob in zip(bases, news, blobs):
        assert torch.equal(blob, zc.compress_delta(b, n))
    back = zc.decompress_batch(blobs, bases=bases)
    assert all(torch.equal(r.view(torch.int16), n.view(torch.int16)) for r, n in zip(back, news))


def test_batch_rejects_mixed_blobs():
    a = zc.compress(torch.zeros(1000, dtype=torch.bfloat16, device=DEV))
    b = zc.compress(torch.zeros(1000, dtype=torch.float32, device=DEV))
    with pytest.raises(zc.ZcError):
        zc.decompress_batch([a, b])
    with pytest.raises(zc.ZcError):
        zc.compress_batch([torch.zeros(4, device=DEV), torch.zeros(4, dtype=torch.bfloat16, device=DEV)])
