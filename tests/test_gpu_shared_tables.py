"""GPU parity of blob format v2 (shared plane tables).

lmzip "Building on lmz": one frequency table per plane kind, shared by many
chunks. The GPU's v2 blobs must equal the oracle's v2 blobs byte for byte,
and the v2 decoder (one CTA-wide table per plane) must restore every tensor
exactly: single tensors of every dtype with ragged tails, decode CTAs of
sixteen chunks, batches of many small tensors, XOR deltas, blobs in host
memory, planes that are constant over the whole tensor, and corrupted plane
tables.
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
V2 = zc.SHARED_TABLES


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


def _bf16(raw: np.ndarray) -> torch.Tensor:
    if raw.size == 0:
        return torch.empty(0, dtype=torch.bfloat16, device=DEV)
    return torch.from_numpy(raw).to(DEV).view(torch.bfloat16)


def gpu_v2(raw: np.ndarray, dtype: int, chunk: int, thr: float) -> bytes:
    nbytes = raw.size
    src = torch.from_numpy(raw).to(DEV)
    cap = zc.blob_size(nbytes, dtype, chunk, thr, V2)
    blob = torch.full((cap,), 0xAB, dtype=torch.uint8, device=DEV)
    ws = torch.full((max(16, zc.workspace_size(nbytes, dtype, chunk, V2)),), 0x5A, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_into(src, blob, nb, ws, st, chunk, thr, dtype=dtype, shape=(nbytes // W_OF[dtype],), flags=V2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return blob[: int(nb.item())].cpu().numpy().tobytes()


def gpu_decode(blob: bytes, verify=True) -> tuple[int, bytes]:
    info = zc.blob_info(blob)
    assert info["version"] == 2
    b = torch.from_numpy(np.frombuffer(blob, np.uint8).copy()).to(DEV)
    out = torch.full((info["nbytes"] + 16,), 0xCD, dtype=torch.uint8, device=DEV)[: info["nbytes"]]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.decompress_into(b, info, out, st, verify)
    torch.cuda.synchronize()
    return int(st.item()), out.cpu().numpy().tobytes()


def check(zco, raw, dtype, chunk=131072, thr=0.95):
    ref = zco.compress(raw, dtype, (raw.size // W_OF[dtype],), chunk, thr, version=2)
    got = gpu_v2(raw, dtype, chunk, thr)
    if got != ref:
        pos = next((i for i in range(min(len(got), len(ref))) if got[i] != ref[i]), min(len(got), len(ref)))
        raise AssertionError(f"v2 blob mismatch: gpu {len(got)} B, oracle {len(ref)} B, first diff at {pos}")
    for verify in (True, False):
        st, back = gpu_decode(got, verify)
        assert st == 0 and back == raw.tobytes()
    return got


@pytest.mark.parametrize("dtype", [4, 6, 5, 1, 2, 3])
@pytest.mark.parametrize("chunk,thr", [(131072, 0.95), (4096, 0.95), (16384, 2.0), (1024, 0.5)])
def test_v2_matches_oracle(zco, dtype, chunk, thr):
    rng = np.random.default_rng(1000 + dtype + chunk)
    for kind in range(4):
        n = int(rng.integers(1, 200_000))
        check(zco, _bytes(rng, dtype, n, kind), dtype, chunk, thr)


def test_v2_workloads(zco):
    blob = check(zco, wl.as_bytes(wl.bf16_1m()).numpy(), 4)
    assert len(blob) < 0.67 * (2 << 20)
    check(zco, wl.as_bytes(wl.fp32_64m(rows=512)).numpy(), 6)
    check(zco, wl.as_bytes(wl.fp32clean_64m(rows=512)).numpy(), 6)
    check(zco, wl.as_bytes(wl.fp16_16m(rows=256)).numpy(), 5)


def test_v2_sixteen_chunks_per_cta(zco):
    """3072 chunks of 4 KiB: decode CTAs of sixteen chunks, several per SM."""
    raw = wl.as_bytes(wl.llama8b_tensor(3, "q", (1536, 4096))).numpy()
    check(zco, raw, 4, 4096, 0.95)


def test_v2_constant_planes(zco):
    check(zco, np.zeros(300_000, np.uint8), 4)                  # every plane constant: zero tables
    check(zco, np.full(400_000, 0x3F, np.uint8), 6)
    x = wl.as_bytes(wl.fp32clean_64m(rows=8)).numpy()          # low two planes constant
    check(zco, x, 6, 4096)


def test_v2_batch_and_delta(zco):
    rng = np.random.default_rng(5)
    sizes = [0, 70_000, 1, 131072, 0, 250_001, 5000]
    ts = [_bf16(_bytes(rng, 4, n, k % 3)) for k, n in enumerate(sizes)]
    blobs = zc.compress_batch(ts, shared_tables=True)
    for t, b in zip(ts, blobs):
        raw = t.view(torch.uint8).cpu().numpy() if t.numel() else np.zeros(0, np.uint8)
        assert b.cpu().numpy().tobytes() == zco.compress(raw, 4, (raw.size // 2,), 131072, 0.95, version=2)
    back = zc.decompress_batch(blobs)
    assert all(torch.equal(r.view(torch.int16), t.view(torch.int16)) for r, t in zip(back, ts))
    # many small tensors: decode CTAs stop at every blob boundary
    small = [_bf16(_bytes(rng, 4, int(n), 0)) for n in rng.integers(1, 9000, 300)]
    sb = zc.compress_batch(small, chunk_bytes=4096, shared_tables=True)
    for t, b in zip(small[:40], sb[:40]):
        raw = t.view(torch.uint8).cpu().numpy()
        assert b.cpu().numpy().tobytes() == zco.compress(raw, 4, (raw.size // 2,), 4096, 0.95, version=2)
    back = zc.decompress_batch(sb)
    assert all(torch.equal(r.view(torch.int16), t.view(torch.int16)) for r, t in zip(back, small))
    # XOR deltas in v2
    a = [(torch.randn(n, device=DEV) * 0.02).bfloat16() for n in (40_000, 300_000)]
    b2 = [(x.float() + torch.randn_like(x.float()) * 1e-4).bfloat16() for x in a]
    db = zc.compress_batch(b2, bases=a, shared_tables=True)
    for x, y, blob in zip(a, b2, db):
        d = (x.view(torch.int16) ^ y.view(torch.int16)).view(torch.uint8).cpu().numpy()
        assert blob.cpu().numpy().tobytes() == zco.compress(d, 2, (d.size // 2,), 131072, 0.95, version=2)
    back = zc.decompress_batch(db, bases=a)
    assert all(torch.equal(r.view(torch.int16), y.view(torch.int16)) for r, y in zip(back, b2))


def test_v2_host_blob_and_python_api():
    t = wl.bf16_1m(DEV)
    hb = zc.compress(t, host_blob=True, shared_tables=True)
    db = zc.compress(t, shared_tables=True)
    assert hb.device.type == "cpu" and torch.equal(hb, db.cpu())
    assert zc.read_info(db)["version"] == 2
    assert torch.equal(zc.decompress(hb).view(torch.int16), t.view(torch.int16))
    assert torch.equal(zc.decompress(db).view(torch.int16), t.view(torch.int16))


def test_v2_oracle_blob_decodes(zco):
    raw = wl.as_bytes(wl.fp32_64m(rows=64)).numpy()
    ref = zco.compress(raw, 6, None, 8192, 0.95, version=2)
    st, back = gpu_decode(ref)
    assert st == 0 and back == raw.tobytes()


def test_v2_corrupted_plane_table_is_reported(zco):
    """A plane table changed on the device after the host read the header:
    either no longer a 12-bit table (the chunks are reported corrupt) or a
    different valid table (the chunk CRCs fail)."""
    raw = wl.as_bytes(wl.bf16_1m()).numpy()
    good = gpu_v2(raw, 4, 131072, 0.95)
    info = zc.blob_info(good)
    t0 = 96 + 16 * info["n_chunks"]
    f = np.frombuffer(good[t0: t0 + 512], "<u2").copy()
    top = int(np.argmax(f))
    nxt = int(np.argsort(f)[-2])
    for mutate in ("sum", "swap"):
        g = f.copy()
        if mutate == "sum":
            g[top] += 1
        else:
            g[top] -= 5
            g[nxt] += 5
        bad = bytearray(good)
        bad[t0: t0 + 512] = g.astype("<u2").tobytes()
        b = torch.from_numpy(np.frombuffer(bytes(bad), np.uint8).copy()).to(DEV)
        out = torch.empty(info["nbytes"], dtype=torch.uint8, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        zc.decompress_into(b, info, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) & (zc.ECORRUPT | zc.ECRC), mutate


def test_v2_small_workspace_waves_at_tensor_boundaries(zco):
    """A batch whose workspace holds 40 chunks of statistics and one coding
    warp: the v2 waves hold whole tensors ([9, 0, 2], [30, 1], [12] chunks),
    so every tensor's plane tables are complete before it is coded."""
    rng = np.random.default_rng(23)
    dtype, chunk, W = 6, 4096, 4
    sizes = [9000, 0, 1500, 30000, 100, 12000]
    raws = [_bytes(rng, dtype, n, k % 3) for k, n in enumerate(sizes)]
    n = len(raws)
    nc = sum((r.size + chunk - 1) // chunk for r in raws)
    pad = lambda x: (x + 255) // 256 * 256
    n_pad = (chunk // W + 31) // 32 * 32
    per_chunk = 32 + W * (512 + n_pad)
    fixed = (256 + pad(16 * n)) + pad(152 * n) + pad(2048 * W * n) + pad(512 * W * n) + pad(8 * nc)
    rec = min(160 + 512 + 2 * (chunk // W), int(np.ceil(0.95 * (chunk // W))) + 160 + 512 + 2048)
    slot = pad(W * ((rec + 15) // 16 * 16 + 16))
    small = fixed + 40 * per_chunk + slot + 768
    full = zc.workspace_size_batch([r.size for r in raws], dtype, chunk, V2)
    assert small < full
    srcs = [torch.from_numpy(r).to(DEV) if r.size else torch.empty(0, dtype=torch.uint8, device=DEV) for r in raws]
    blobs = [torch.full((zc.blob_size(r.size, dtype, chunk, 0.95, V2),), 0xAB, dtype=torch.uint8, device=DEV)
             for r in raws]
    ws = torch.full((small,), 0x5A, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(n, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_batch_into(srcs, blobs, nb, ws, st, dtype, [(r.size // W,) for r in raws], chunk, 0.95, flags=V2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for r, b, k in zip(raws, blobs, nb.tolist()):
        got = b[:k].cpu().numpy().tobytes()
        assert got == zco.compress(r, dtype, (r.size // W,), chunk, 0.95, version=2)
        if r.size:
            s2, back = gpu_decode(got)
            assert s2 == 0 and back == r.tobytes()
