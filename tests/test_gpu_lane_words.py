"""GPU parity of blob format v3 (a word list per rANS lane).

lmzip "On a GPU": a GPU rANS decoder is bound by the dependent chain of each
lane's steps; v3 gives every lane its own word list so that no decoding
step waits on where the other lanes' words end. The GPU's v3 blobs must
equal the oracle's v3 blobs byte for byte, and the v3 decoder must restore
every tensor exactly: every dtype with ragged tails, chunk sizes and
thresholds (every stream coded at threshold 2), the workloads, batches of
many small tensors (two-level tables), XOR deltas, host blobs, oracle-made
blobs, corrupted records (counts, lists, padding) and the blob check.
"""
from __future__ import annotations

import struct

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
V3 = zc.LANE_WORDS


def _bytes(rng, dtype: int, n: int, kind: int) -> np.ndarray:
    W = W_OF[dtype]
    if n == 0:
        return np.zeros(0, np.uint8)
    if kind == 0 and dtype in (4, 5, 6):
        x = torch.from_numpy((rng.standard_normal(n) * float(rng.choice([0.02, 1.0]))).astype(np.float32))
        return x.to({4: torch.bfloat16, 5: torch.float16, 6: torch.float32}[dtype]).view(torch.uint8).numpy().copy()
    if kind == 1:
        return rng.integers(0, 12, n * W, dtype=np.uint8)
    if kind == 2:
        return rng.integers(0, 256, n * W, dtype=np.uint8)
    return np.full(n * W, 7, np.uint8)


def gpu_v3(raw: np.ndarray, dtype: int, chunk: int, thr: float) -> bytes:
    nbytes = raw.size
    src = torch.from_numpy(raw).to(DEV)
    cap = zc.blob_size(nbytes, dtype, chunk, thr, V3)
    blob = torch.full((cap,), 0xAB, dtype=torch.uint8, device=DEV)
    ws = torch.full((max(16, zc.workspace_size(nbytes, dtype, chunk, V3)),), 0x5A, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_into(src, blob, nb, ws, st, chunk, thr, dtype=dtype, shape=(nbytes // W_OF[dtype],), flags=V3)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return blob[: int(nb.item())].cpu().numpy().tobytes()


def gpu_decode(blob: bytes, verify=True) -> tuple[int, bytes]:
    info = zc.blob_info(blob)
    assert info["version"] == 3
    b = torch.from_numpy(np.frombuffer(blob, np.uint8).copy()).to(DEV)
    out = torch.full((info["nbytes"] + 16,), 0xCD, dtype=torch.uint8, device=DEV)[: info["nbytes"]]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.decompress_into(b, info, out, st, verify)
    torch.cuda.synchronize()
    return int(st.item()), out.cpu().numpy().tobytes()


def check(zco, raw, dtype, chunk=131072, thr=0.95):
    ref = zco.compress(raw, dtype, (raw.size // W_OF[dtype],), chunk, thr, version=3)
    got = gpu_v3(raw, dtype, chunk, thr)
    if got != ref:
        pos = next((i for i in range(min(len(got), len(ref))) if got[i] != ref[i]), min(len(got), len(ref)))
        raise AssertionError(f"v3 blob mismatch: gpu {len(got)} B, oracle {len(ref)} B, first diff at {pos}")
    for verify in (True, False):
        st, back = gpu_decode(got, verify)
        assert st == 0 and back == raw.tobytes()
    return got


@pytest.mark.parametrize("dtype", [4, 6, 5, 1, 2, 3])
@pytest.mark.parametrize("chunk,thr", [(131072, 0.95), (4096, 0.95), (16384, 2.0), (1024, 0.5), (64, 2.0)])
def test_v3_matches_oracle(zco, dtype, chunk, thr):
    rng = np.random.default_rng(3000 + dtype + chunk)
    for kind in range(4):
        n = int(rng.integers(1, 200_000 if chunk > 64 else 5000))
        check(zco, _bytes(rng, dtype, n, kind), dtype, chunk, thr)


def test_v3_workloads(zco):
    blob = check(zco, wl.as_bytes(wl.bf16_1m()).numpy(), 4)
    assert len(blob) < 0.67 * (2 << 20)
    check(zco, wl.as_bytes(wl.fp32_64m(rows=512)).numpy(), 6)
    check(zco, wl.as_bytes(wl.fp32clean_64m(rows=512)).numpy(), 6)
    check(zco, wl.as_bytes(wl.fp16_16m(rows=256)).numpy(), 5)
    check(zco, wl.as_bytes(wl.bf16_delta(rows=64)[1]).numpy(), 2)   # both streams coded


def test_v3_full_size_tensors(zco):
    """A Llama gate projection (896 chunks: one-level tables) and a 3072-chunk
    tensor of 4 KiB chunks (two-level tables, many chunks per SM)."""
    t = wl.llama8b_tensor(5, "layers.0.gate", (14336, 4096), DEV)
    raw = wl.as_bytes(t).cpu().numpy()
    got = zc.compress(t, lane_words=True)
    assert got.cpu().numpy().tobytes() == zco.compress(raw, 4, (14336, 4096), version=3)
    assert torch.equal(zc.decompress(got).view(torch.int16), t.view(torch.int16))
    raw = wl.as_bytes(wl.llama8b_tensor(3, "q", (1536, 4096))).numpy()
    check(zco, raw, 4, 4096, 0.95)


def test_v3_batch_and_delta(zco):
    rng = np.random.default_rng(6)
    small = [torch.from_numpy(_bytes(rng, 4, int(n), 0)).to(DEV).view(torch.bfloat16)
             for n in rng.integers(1, 9000, 300)]
    sb = zc.compress_batch(small, chunk_bytes=4096, lane_words=True)
    for t, b in zip(small[:40], sb[:40]):
        raw = t.view(torch.uint8).cpu().numpy()
        assert b.cpu().numpy().tobytes() == zco.compress(raw, 4, (raw.size // 2,), 4096, 0.95, version=3)
    back = zc.decompress_batch(sb)
    assert all(torch.equal(r.view(torch.int16), t.view(torch.int16)) for r, t in zip(back, small))
    a = [(torch.randn(n, device=DEV) * 0.02).bfloat16() for n in (40_000, 300_000)]
    b2 = [(x.float() + torch.randn_like(x.float()) * 1e-4).bfloat16() for x in a]
    db = zc.compress_batch(b2, bases=a, lane_words=True)
    for x, y, blob in zip(a, b2, db):
        d = (x.view(torch.int16) ^ y.view(torch.int16)).view(torch.uint8).cpu().numpy()
        assert blob.cpu().numpy().tobytes() == zco.compress(d, 2, (d.size // 2,), 131072, 0.95, version=3)
    back = zc.decompress_batch(db, bases=a)
    assert all(torch.equal(r.view(torch.int16), y.view(torch.int16)) for r, y in zip(back, b2))


def test_v3_host_blob_and_verify():
    t = wl.bf16_1m(DEV)
    hb = zc.compress(t, host_blob=True, lane_words=True)
    db = zc.compress(t, lane_words=True)
    assert hb.device.type == "cpu" and torch.equal(hb, db.cpu())
    assert zc.read_info(db)["version"] == 3
    assert zc.verify(db) == 0 and zc.verify(hb) == 0
    assert torch.equal(zc.decompress(hb).view(torch.int16), t.view(torch.int16))


def test_v3_oracle_blob_decodes(zco):
    raw = wl.as_bytes(wl.fp32_64m(rows=64)).numpy()
    ref = zco.compress(raw, 6, None, 8192, 0.95, version=3)
    st, back = gpu_decode(ref)
    assert st == 0 and back == raw.tobytes()


def test_v3_corrupted_records(zco):
    """Changed word counts, list words and list padding of a coded record:
    with the CRC check every change is reported as ECRC; without it the
    structure checks (counts that do not describe the record, nonzero
    padding, final states) report the changes that break the record, and no
    read leaves the blob."""
    raw = wl.as_bytes(wl.bf16_1m()[:64]).numpy()
    blob = zco.compress(raw, 4, None, 8192, 0.95, version=3)
    off, sm, _ = struct.unpack_from("<QII", blob, 96)
    assert not sm >> 31
    rec = off + 16                                  # stream 0's record after the directory
    k = sum(bin(b).count("1") for b in blob[rec + 128: rec + 160])
    counts_at = rec + 160 + (2 * k + 15) // 16 * 16
    counts = struct.unpack_from("<32H", blob, counts_at)
    lists_at = counts_at + 64
    first_pad = next(l for l in range(32) if counts[l] % 8)   # a lane whose list is padded
    pad_at = lists_at + 2 * sum((c + 7) // 8 * 8 for c in counts[:first_pad]) + 2 * counts[first_pad]
    cases = {"count": counts_at + 2 * 5, "word": lists_at + 2, "padding": pad_at}
    for name, pos in cases.items():
        bad = bytearray(blob)
        bad[pos] ^= 0x01
        st, _ = gpu_decode(bytes(bad))
        assert st & zc.ECRC, name
        st, out = gpu_decode(bytes(bad), verify=False)
        if name in ("count", "padding"):
            assert st & zc.ECORRUPT, name
        assert st in (0, zc.ECORRUPT), (name, st)
