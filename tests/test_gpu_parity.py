"""GPU parity: the CUDA path against the oracle, through the C ABI.

Integer/byte work, so the bar is bit-exactness everywhere: GPU blobs equal
oracle blobs byte for byte, GPU decoding restores the input exactly (from
both GPU and oracle blobs), and the oracle decodes GPU blobs. Inputs are the
seeded synthetic workloads (every configuration at full size; the 16 GB
Llama-shaped model, every tensor, is in test_gpu_llama8b_full.py) plus edge
cases: empty, ragged, tiny, constant, NaN-laden,
near the passthrough threshold, many chunks, unaligned pointers, corrupted
blobs.
"""
from __future__ import annotations

import struct
import zlib

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


def gpu_compress_bytes(raw: np.ndarray, dtype: int, shape, chunk=131072, thr=0.95, offset=0) -> bytes:
    """Compress host bytes on the GPU (optionally from a misaligned device
    pointer `offset` bytes into a buffer) and return the blob bytes."""
    nbytes = raw.size
    buf = torch.empty(nbytes + offset + 16, dtype=torch.uint8, device=DEV)
    src = buf[offset:offset + nbytes]
    if nbytes:
        src.copy_(torch.from_numpy(raw))
    cap = zc.blob_size(nbytes, dtype, chunk, thr)
    assert cap > 0
    blob = torch.full((cap,), 0xAB, dtype=torch.uint8, device=DEV)   # stale bytes must not leak
    ws = torch.full((max(16, zc.workspace_size(nbytes, dtype, chunk)),), 0x5A, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_into(src, blob, nb, ws, st, chunk, thr, dtype=dtype, shape=shape)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return blob[: int(nb.item())].cpu().numpy().tobytes()


def gpu_decompress_bytes(blob: bytes, verify=True, offset=0) -> tuple[int, np.ndarray]:
    info = zc.blob_info(blob)
    b = torch.from_numpy(np.frombuffer(blob, np.uint8).copy()).to(DEV)
    out_buf = torch.full((info["nbytes"] + offset + 16,), 0xCD, dtype=torch.uint8, device=DEV)
    out = out_buf[offset:offset + info["nbytes"]]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.decompress_into(b, info, out, st, verify)
    torch.cuda.synchronize()
    return int(st.item()), out.cpu().numpy()


def check_parity(zco, raw: np.ndarray, dtype: int, shape, chunk=131072, thr=0.95, offset=0):
    ref = zco.compress(raw, dtype, shape, chunk, thr)
    got = gpu_compress_bytes(raw, dtype, shape, chunk, thr, offset)
    if got != ref:
        pos = next((i for i in range(min(len(got), len(ref))) if got[i] != ref[i]), min(len(got), len(ref)))
        raise AssertionError(f"blob mismatch: gpu {len(got)} B, oracle {len(ref)} B, first diff at {pos}")
    st, back = gpu_decompress_bytes(got, offset=offset)
    assert st == 0 and back.tobytes() == raw.tobytes()
    st, back = gpu_decompress_bytes(got, verify=False)
    assert st == 0 and back.tobytes() == raw.tobytes()
    return got


# --------------------------------------------------------------- CRC-32

def test_crc32_pieces_match_zlib():
    rng = np.random.default_rng(0)
    for n in (0, 1, 15, 16, 17, 1000, 16384, 16385, 100000, 1 << 20, (1 << 20) + 7):
        data = rng.integers(0, 256, n + 3, dtype=np.uint8)
        for off in (0, 1, 3):
            d = torch.from_numpy(data[off:off + n].copy()).to(DEV) if n else torch.empty(0, dtype=torch.uint8, device=DEV)
            for piece in (0, 16384, 1000, 64):
                if piece and n // piece > 20000:
                    continue
                got = zc.crc32(d, piece).cpu().numpy().tolist()
                b = data[off:off + n].tobytes()
                if piece == 0:
                    want = [zlib.crc32(b)]
                else:
                    want = [zlib.crc32(b[i:i + piece]) for i in range(0, n, piece)]
                assert got == want, (n, off, piece)


def test_crc32_large_whole_buffer():
    t = torch.randint(0, 256, (300_000_000,), dtype=torch.uint8, device=DEV)
    got = int(zc.crc32(t, 0).item())
    assert got == zlib.crc32(t.cpu().numpy().tobytes())


# ------------------------------------------------------- small and ragged

def _rand_tensor(rng, dtype, n):
    W = W_OF[dtype]
    kind = int(rng.integers(0, 6))
    if n == 0:
        return np.zeros(0, np.uint8)
    if kind == 0:
        return rng.integers(0, 256, n * W, dtype=np.uint8)
    if kind == 1:
        return np.full(n * W, rng.integers(0, 256), np.uint8)
    if kind == 2:
        return rng.choice(np.array([7, 9], np.uint8), n * W)
    if dtype in (1, 2, 3):
        return rng.integers(0, 16, n * W, dtype=np.uint8)
    sigma = float(rng.choice([0.02, 0.05, 1.0, 1e-3]))
    x = torch.from_numpy((rng.standard_normal(n) * sigma).astype(np.float32))
    if kind == 4 and n:
        x[torch.from_numpy(rng.integers(0, n, max(1, n // 50)))] = float("nan")
    if dtype == 4:
        x = x.bfloat16()
    elif dtype == 5:
        x = x.half()
    elif kind == 5:
        x = x.bfloat16().float()
    x = x.contiguous()
    return x.numpy().view(np.uint8).copy() if dtype == 6 else x.view(torch.int16).numpy().view(np.uint8).copy()


def test_random_small_tensors(zco):
    rng = np.random.default_rng(77)
    for trial in range(300):
        dtype = int(rng.integers(1, 7))
        n = int(rng.choice([0, 1, 2, 31, 32, 33, 63, 4095, 4097, int(rng.integers(0, 70000))]))
        raw = _rand_tensor(rng, dtype, n)
        chunk = int(rng.choice([64, 128, 4096, 65536, 131072]))
        thr = float(rng.choice([0.5, 0.95, 1.0, 2.0, 1e6]))
        check_parity(zco, raw, dtype, (n,), chunk, thr)


def test_exhaustive_bf16_patterns(zco):
    words = np.arange(65536, dtype=np.uint16).view(np.uint8)
    check_parity(zco, words, 4, (65536,), 131072, 0.95)
    check_parity(zco, words, 4, (65536,), 4096, 0.95)
    sh = np.random.default_rng(7).permutation(65536).astype(np.uint16).view(np.uint8)
    check_parity(zco, sh, 4, (256, 256), 131072, 2.0)
    for dt in (2, 5):
        check_parity(zco, words, dt, (65536,), 8192, 0.95)


def test_unaligned_pointers(zco):
    rng = np.random.default_rng(5)
    x = torch.from_numpy((rng.standard_normal(100_003) * 0.02).astype(np.float32))
    raw32 = x.numpy().view(np.uint8).copy()
    raw16 = x.bfloat16().view(torch.int16).numpy().view(np.uint8).copy()
    # 16 is 16-byte but not 32-byte aligned: the statistics pass's two-load path
    for off in (4, 8, 12, 16):
        check_parity(zco, raw32, 6, (100_003,), 131072, 0.95, offset=off)
    for off in (2, 6, 10, 16):
        check_parity(zco, raw16, 4, (100_003,), 4096, 0.95, offset=off)


def test_near_threshold_streams(zco):
    """Streams whose coded size is close to threshold x raw size: the GPU's
    skip of provably-incompressible streams must never change a decision."""
    rng = np.random.default_rng(3)
    n = 65536
    for k in (160, 180, 200, 230, 256):
        for skew in (0.0, 0.3, 0.6):
            p = np.exp(-skew * np.arange(k) / k)
            p /= p.sum()
            syms = rng.choice(k, n, p=p).astype(np.uint8)
            for thr in (0.85, 0.9, 0.95, 0.97, 1.0, 1.03):
                check_parity(zco, syms, 1, (n,), 65536, thr)


def test_many_chunks_lookback(zco):
    """~200k chunks of 64 bytes exercise the offset scan across many warps."""
    t = wl.bf16_1m("cpu")
    raw = wl.as_bytes(t).numpy()
    raw = np.concatenate([raw] * 6)
    check_parity(zco, raw, 4, (raw.size // 2,), 64, 0.95)


def _compress_with_workspace(raw: np.ndarray, dtype: int, chunk: int, thr: float, ws_bytes: int) -> bytes:
    nbytes = raw.size
    src = torch.from_numpy(raw).to(DEV)
    cap = zc.blob_size(nbytes, dtype, chunk, thr)
    blob = torch.full((cap,), 0xAB, dtype=torch.uint8, device=DEV)
    ws = torch.full((ws_bytes,), 0x5A, dtype=torch.uint8, device=DEV)
    nb = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.compress_into(src, blob, nb, ws, st, chunk, thr, dtype=dtype, shape=(nbytes // W_OF[dtype],))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return blob[: int(nb.item())].cpu().numpy().tobytes()


@pytest.mark.parametrize("dtype,thr", [(6, 0.95), (4, 0.95), (1, 2.0)])
def test_small_workspace_many_waves(zco, dtype, thr):
    """A workspace far below zc_workspace_size: waves of a few chunks each
    (every chunk of a wave with a coding warp of its own, as many as the
    slots that fit), the offset scan running across the waves."""
    rng = np.random.default_rng(5 + dtype)
    raw = _rand_tensor(rng, dtype, 75_000)
    chunk = 4096
    ref = zco.compress(raw, dtype, (raw.size // W_OF[dtype],), chunk, thr)
    nc = (raw.size + chunk - 1) // chunk
    W = W_OF[dtype]
    n_pad = (chunk // W + 31) // 32 * 32
    per_chunk = 32 + W * (512 + n_pad)
    full = zc.workspace_size(raw.size, dtype, chunk)
    # control + status words, room for about 5 chunks of a wave, and about
    # one coding slot (bounded by a generous record size)
    small = 256 + (8 * nc + 255) // 256 * 256 + 5 * per_chunk + 1024 + 2 * W * (2 * chunk // W + 4096)
    assert small < full
    got = _compress_with_workspace(raw, dtype, chunk, thr, small)
    assert got == ref, "blob differs from the oracle's with a small workspace"
    st, back = gpu_decompress_bytes(got)
    assert st == 0 and back.tobytes() == raw.tobytes()


def test_constant_and_special_tensors(zco):
    for dtype, word in ((4, 0x3F80), (6, 0x3F800000), (5, 0x3C00), (4, 0x0000), (6, 0x7FC00001)):
        W = W_OF[dtype]
        raw = np.frombuffer(int(word).to_bytes(W, "little") * 300_001, np.uint8).copy()
        check_parity(zco, raw, dtype, (300_001,), 131072, 0.95)


# ------------------------------------------------------------ workloads

def _check_tensor(zco, t: torch.Tensor, thr=0.95):
    raw = wl.as_bytes(t.cpu()).numpy()
    return check_parity(zco, raw, wl.dtype_code(t), tuple(t.shape), 131072, thr)


def test_workload_bf16_1m(zco):
    blob = _check_tensor(zco, wl.bf16_1m("cpu"))
    assert 0.64 < len(blob) / (2 << 20) < 0.68


def test_workload_fp32_64m(zco):
    _check_tensor(zco, wl.fp32_64m(DEV))


def test_workload_fp32clean_64m(zco):
    _check_tensor(zco, wl.fp32clean_64m(DEV))


def test_workload_fp16_16m(zco):
    _check_tensor(zco, wl.fp16_16m(DEV))


def test_workload_bf16_delta(zco):
    a, x = wl.bf16_delta(DEV)
    _check_tensor(zco, a)
    blob = _check_tensor(zco, x)
    assert len(blob) < 0.4 * x.numel() * 2


# ------------------------------------------------------------ corruption

def test_corrupted_blobs_are_rejected(zco):
    rng = np.random.default_rng(12)
    t = wl.bf16_1m("cpu")[:128]
    raw = wl.as_bytes(t).numpy()
    blob = gpu_compress_bytes(raw, 4, tuple(t.shape), 4096, 0.95)
    table_end = 96 + 16 * struct.unpack_from("<I", blob, 24)[0]
    hits = 0
    for _ in range(200):
        pos = int(rng.integers(table_end, len(blob)))
        bad = bytearray(blob)
        bad[pos] ^= int(rng.integers(1, 256))
        st, out = gpu_decompress_bytes(bytes(bad))
        assert st != 0 or out.tobytes() == raw.tobytes()
        hits += st != 0
        # without the CRC the structure checks still keep every read in bounds
        st2, _ = gpu_decompress_bytes(bytes(bad), verify=False)
        assert st2 in (0, zc.ECORRUPT, zc.EFORMAT)
    assert hits > 150


def test_verify_matches_oracle(zco):
    """zc_verify checks a blob without decoding it (cuZipNN API: verify an
    untrusted blob first). It passes every intact blob, and for a blob with
    one changed byte it reports exactly what the oracle's check reports for
    a payload or padding byte, and an error whenever the oracle does for a
    header or table byte (the device check sees the header CRC fail where the
    oracle may first see a malformed field)."""
    rng = np.random.default_rng(41)
    cases = [(wl.as_bytes(wl.bf16_1m("cpu")[:96]).numpy(), 4, 4096, 1),
             (wl.as_bytes(wl.fp32_64m("cpu", rows=8)).numpy(), 6, 65536, 1),
             (rng.integers(0, 256, 70001, dtype=np.uint8), 1, 4096, 1),   # RAW chunks, ragged tail
             (wl.as_bytes(wl.bf16_1m("cpu")[:64]).numpy(), 4, 8192, 2)]
    for raw, dt, C, ver in cases:
        blob = zco.compress(raw, dt, None, C, 0.95, version=ver)
        info = zc.blob_info(blob)
        table_end = 96 + 16 * info["n_chunks"] + (512 * W_OF[dt] if ver == 2 else 0)
        good = torch.from_numpy(np.frombuffer(blob, np.uint8).copy()).to(DEV)
        assert zc.verify(good, info) == 0 and zco.verify(blob) == 0
        # a GPU blob of the same tensor passes too
        if ver == 1:
            gb = gpu_compress_bytes(raw, dt, (raw.size // W_OF[dt],), C, 0.95)
            assert zc.verify(torch.from_numpy(np.frombuffer(gb, np.uint8).copy()).to(DEV)) == 0
        positions = list(rng.integers(0, len(blob), 120)) + list(range(0, 96, 5)) + [table_end - 1, len(blob) - 1]
        for pos in positions:
            bad = bytearray(blob)
            bad[int(pos)] ^= int(rng.integers(1, 256))
            dev = torch.from_numpy(np.frombuffer(bytes(bad), np.uint8).copy()).to(DEV)
            st = zc.verify(dev, info)
            want = zco.verify(bytes(bad))
            if pos >= table_end:
                assert st == want, (dt, ver, int(pos), st, want)
            else:
                assert (st != 0) == (want != 0) and st & (zc.ECRC | zc.EFORMAT), (dt, ver, int(pos), st, want)
    # a table entry pointing past the blob: a format error, no read
    raw, dt, C, _ = cases[0]
    blob = bytearray(zco.compress(raw, dt, None, C, 0.95))
    info = zc.blob_info(bytes(blob))
    struct.pack_into("<Q", blob, 96 + 16 * 2, 1 << 40)
    dev = torch.from_numpy(np.frombuffer(bytes(blob), np.uint8).copy()).to(DEV)
    assert zc.verify(dev, info) & zc.EFORMAT


def test_decode_reports_changed_payload_as_crc(zco):
    """A changed payload byte fails its chunk's CRC over the stored bytes in
    decoding too; the other chunks decode exactly."""
    rng = np.random.default_rng(43)
    raw = wl.as_bytes(wl.bf16_1m("cpu")[:64]).numpy()
    C = 8192
    blob = zco.compress(raw, 4, None, C, 0.95)
    nc = struct.unpack_from("<I", blob, 24)[0]
    for c in range(0, nc, 3):
        off, sm, _ = struct.unpack_from("<QII", blob, 96 + 16 * c)
        stored = sm & 0x7FFFFFFF
        for pos in (off, off + stored - 1, off + int(rng.integers(0, stored))):
            bad = bytearray(blob)
            bad[pos] ^= 0x10
            st, out = gpu_decompress_bytes(bytes(bad))
            assert st & zc.ECRC, (c, pos)
            keep = np.ones(raw.size, bool)
            keep[c * C:(c + 1) * C] = False
            assert (out[keep] == raw[keep]).all()


@pytest.mark.parametrize("version", [1, 3])
def test_many_chunks_per_sm_report_every_chunk(zco, version):
    """With many chunks per SM (two-level tables, 16 chunks per CTA here) the
    consumer checks the CRC as it reads: a changed byte in any chunk, at
    every position of a CTA's chunk list, is reported, and the blob decodes
    exactly when nothing was changed."""
    t = wl.fp32_64m("cpu", rows=128)  # 4 MiB: 4096 chunks of 1 KiB, 27 per SM
    raw = wl.as_bytes(t).numpy()
    C = 1024
    blob = zco.compress(raw, wl.dtype_code(t), tuple(t.shape), C, 0.95, version)
    st, out = gpu_decompress_bytes(blob)
    assert st == 0 and (out == raw).all()
    nc = struct.unpack_from("<I", blob, 24)[0]
    rng = np.random.default_rng(44)
    for c in list(range(0, 20)) + [nc // 2, nc // 2 + 7, nc - 2, nc - 1]:
        off, sm, _ = struct.unpack_from("<QII", blob, 96 + 16 * c)
        bad = bytearray(blob)
        bad[off + int(rng.integers(0, sm & 0x7FFFFFFF))] ^= 0x04
        st, out = gpu_decompress_bytes(bytes(bad))
        assert st & zc.ECRC, (c, st)
        st, _ = gpu_decompress_bytes(bytes(bad), verify=False)
        assert not st & zc.ECRC, (c, st)


def test_corrupted_table_entry_device_checks():
    """A table entry pointing outside the blob is caught on the device even
    when the host check is bypassed (info taken from the good blob)."""
    t = wl.bf16_1m("cpu")[:64]
    raw = wl.as_bytes(t).numpy()
    blob = bytearray(gpu_compress_bytes(raw, 4, tuple(t.shape), 4096, 0.95))
    info = zc.blob_info(bytes(blob))
    struct.pack_into("<Q", blob, 96 + 16 * 3, 1 << 40)
    b = torch.from_numpy(np.frombuffer(bytes(blob), np.uint8).copy()).to(DEV)
    out = torch.empty(info["nbytes"], dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    zc.decompress_into(b, info, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) & zc.EFORMAT


def test_python_api_roundtrip():
    for t in (wl.bf16_1m(DEV), wl.fp16_16m(DEV, rows=64), torch.zeros(0, 3, device=DEV),
              torch.randn(7, 5, 3, device=DEV), torch.randint(-5, 5, (1000,), dtype=torch.int32, device=DEV)):
        blob = zc.compress(t)
        back = zc.decompress(blob)
        assert back.shape == t.shape and back.dtype == t.dtype
        assert torch.equal(back.view(torch.uint8) if back.numel() else back, t.view(torch.uint8) if t.numel() else t)
