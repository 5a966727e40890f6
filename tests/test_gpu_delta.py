"""Fused XOR-delta compression (ZipNN note, Method 6: XOR a checkpoint
against a base, then code the byte groups) against the oracle: the blob of
compress_delta(base, new) must be the oracle's blob of (base XOR new) as
unsigned words, and decompress_delta must give `new` back."""
import numpy as np
import pytest
import torch

import entropy_coding_gb300 as zc
from entropy_coding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
CODE = {1: zc.U8, 2: zc.U16, 4: zc.U32}


def _pair(rng, n, word, frac_changed):
    """A base of n words and an update that changes about frac_changed of
    them in their low bits (a fine-tuning step)."""
    dt = {1: np.uint8, 2: np.uint16, 4: np.uint32}[word]
    base = rng.integers(0, np.iinfo(dt).max, n, dtype=dt, endpoint=True)
    flip = rng.integers(0, 1 << min(8 * word - 1, 12), n).astype(dt)
    mask = rng.random(n) < frac_changed
    new = base ^ np.where(mask, flip, 0).astype(dt)
    return base, new


def _check(zco, base: np.ndarray, new: np.ndarray, chunk=131072, thr=0.95, offset=0):
    word = base.dtype.itemsize
    code = CODE[word]
    x = (base ^ new).view(np.uint8)
    ref = zco.compress(x, code, (base.size,), chunk, thr)
    tb = torch.from_numpy(base.view(np.uint8).copy()).to(DEV)
    tn = torch.from_numpy(new.view(np.uint8).copy()).to(DEV)
    nbytes = x.size
    cap = zc.blob_size(nbytes, code, chunk, thr)
    blob = torch.full((cap,), 0xAB, dtype=torch.uint8, device=DEV)
    ws = torch.full((max(16, zc.workspace_size(nbytes, code, chunk)),), 0x5A, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_delta_into(tb, tn, blob, nb, ws, st, chunk, thr, dtype=code, shape=(base.size,))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = blob[: int(nb.item())].cpu().numpy().tobytes()
    assert got == ref, f"delta blob differs from the oracle's: {len(got)} vs {len(ref)} bytes"
    info = zc.blob_info(got)
    out = torch.full((nbytes,), 0xCD, dtype=torch.uint8, device=DEV)
    st.zero_()
    zc.decompress_delta_into(blob, info, tb, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert out.cpu().numpy().tobytes() == new.view(np.uint8).tobytes()
    # the plain decoder of the same blob gives the difference
    back = torch.full((nbytes,), 0xEF, dtype=torch.uint8, device=DEV)
    st.zero_()
    zc.decompress_into(blob, info, back, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and back.cpu().numpy().tobytes() == x.tobytes()


@pytest.mark.parametrize("word", [1, 2, 4])
@pytest.mark.parametrize("n,chunk,frac", [(1, 131072, 0.5), (1000, 4096, 0.3), (300_001, 131072, 0.3),
                                          (200_000, 65536, 0.0), (70_000, 4096, 1.0)])
def test_delta_matches_oracle(zco, word, n, chunk, frac):
    rng = np.random.default_rng(n + 7 * word)
    base, new = _pair(rng, n, word, frac)
    _check(zco, base, new, chunk)


def test_delta_random_difference_raw_chunks(zco):
    """Unrelated tensors: the difference is incompressible, chunks are RAW."""
    rng = np.random.default_rng(11)
    base = rng.integers(0, 1 << 16, 150_000, dtype=np.uint16)
    new = rng.integers(0, 1 << 16, 150_000, dtype=np.uint16)
    _check(zco, base, new, 16384)


def test_delta_checkpoint_pair(zco):
    """BF16 checkpoint pair in the shape of the pages' fine-tuning deltas."""
    a, b = wl.bf16_delta_pair("cpu", rows=256)
    base = a.view(torch.int16).numpy().view(np.uint16)
    new = b.view(torch.int16).numpy().view(np.uint16)
    _check(zco, base, new, 131072)


def test_delta_python_api():
    a, b = wl.bf16_delta_pair("cuda", rows=128)
    blob = zc.compress_delta(a, b)
    back = zc.decompress_delta(blob, a)
    assert back.dtype == b.dtype and torch.equal(back.view(torch.int16), b.view(torch.int16))
    diff = zc.decompress(blob)
    assert torch.equal(diff.view(torch.int16).view(-1), (a.view(torch.int16) ^ b.view(torch.int16)).view(-1))


def test_delta_rejects_float_dtype_and_misalignment():
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    blob = torch.zeros(1 << 17, dtype=torch.uint8, device=DEV)
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(zc.ZcError):
        zc.compress_delta_into(buf[:4096], buf[4096:8192], blob, nb, ws, st, dtype=zc.BF16, shape=(2048,))
    with pytest.raises(zc.ZcError):
        zc.compress_delta_into(buf[8:4104], buf[4096:8192], blob, nb, ws, st, dtype=zc.U16, shape=(2048,))
