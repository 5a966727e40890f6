"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties the oracle to a fixed point the pages or the mathematics give:
published CRC check values and zlib (cuZipNN, API: checksums match
zlib.crc32), the IEEE field layouts (ZipNN note, Method 1-2), hand-worked
tables and a hand-worked blob, an exact information identity of rANS with
power-of-two tables, the order-0 entropy (ZipNN note, Key insight), Table II
sizes, and an independent pure-Python reader of the format.
"""
from __future__ import annotations

import math
import os
import struct
import zlib

import numpy as np
import pytest
import torch

from entropy_coding_gb300 import workloads
import spec_decoder

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CODES = {"U8": 1, "U16": 2, "U32": 3, "BF16": 4, "FP16": 5, "FP32": 6}
L = 1 << 16


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.rstrip("\n")
            if line.strip() and not line.lstrip().startswith("#"):
                yield line


# ------------------------------------------------------------------ CRC-32

def test_crc32_golden(zco):
    for line in _golden_lines("crc32_check.txt"):
        data_spec, expect = line.rsplit(None, 1)
        data_spec = data_spec.rstrip()
        if data_spec.startswith("ascii:"):
            data = data_spec[len("ascii:"):].encode()
        else:
            data = bytes.fromhex(data_spec[len("hex:"):])
        assert zco.crc32(np.frombuffer(data, np.uint8)) == int(expect, 16), data_spec


def test_crc32_matches_zlib(zco):
    rng = np.random.default_rng(11)
    for n in list(range(0, 300)) + list(range(300, 4097, 97)) + [1 << 20]:
        d = rng.integers(0, 256, n, dtype=np.uint8)
        assert zco.crc32(d) == zlib.crc32(d.tobytes()), n


# ------------------------------------------- exponent extraction + grouping

def test_group_layout_golden(zco):
    for line in _golden_lines("exponent_layout.txt"):
        parts = line.split()
        dtype = CODES[parts[0]]
        W = zco.WORD_BYTES[dtype]
        word = int(parts[1], 16).to_bytes(W, "little")
        expect = [int(b, 16) for b in parts[2:2 + W]]
        got = zco.group_split(np.frombuffer(word, np.uint8), dtype)[:, 0].tolist()
        assert got == expect, line


def _frexp_fields(values: np.ndarray, bias_shift: int):
    m, e = np.frexp(values.astype(np.float64))
    return (e + bias_shift).astype(np.int64), np.signbit(values)


def test_group_exponent_stream_is_ieee_exponent(zco):
    """Stream 0 of BF16/FP32 is the biased exponent that frexp reports, the
    sign is the top bit of stream 1; FP16 stream 0 holds e5|s|m[9:8]."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * 0.02).astype(np.float32)
    x = x[np.abs(x) > 1e-30]
    for t, dt in ((torch.from_numpy(x).bfloat16(), 4), (torch.from_numpy(x), 6)):
        raw = t.view(torch.int16 if dt == 4 else torch.int32).numpy().view(np.uint8)
        st = zco.group_split(raw, dt)
        e, sign = _frexp_fields(t.float().numpy(), 126)
        assert (st[0].astype(np.int64) == e).all()
        assert ((st[1] >> 7).astype(bool) == sign).all()
    h = torch.from_numpy((rng.standard_normal(20000) * 0.05).astype(np.float32)).half()
    h = h[h.float().abs() > 6.2e-5]  # normal FP16 numbers only
    st = zco.group_split(h.view(torch.int16).numpy().view(np.uint8), 5)
    e, sign = _frexp_fields(h.float().numpy(), 14)
    bits = h.view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    assert ((st[0] >> 3).astype(np.int64) == e).all()
    assert (((st[0] >> 2) & 1).astype(bool) == sign).all()
    assert ((st[0] & 3).astype(np.int64) == (bits >> 8) & 3).all()
    assert (st[1].astype(np.int64) == bits & 0xFF).all()


def test_group_split_merge_exhaustive_16bit(zco):
    words = np.arange(65536, dtype=np.uint16).view(np.uint8)
    for dt in (2, 4, 5):
        st = zco.group_split(words, dt)
        assert (zco.group_merge(st, dt) == words).all()
        # a bijection: every (stream0, stream1) pair occurs exactly once
        pairs = st[0].astype(np.int64) * 256 + st[1]
        assert np.unique(pairs).size == 65536


def test_group_split_merge_fp32(zco):
    rng = np.random.default_rng(3)
    w = np.concatenate([rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32),
                        np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00001, 1, 0xFFFFFFFF],
                                 np.uint32)]).view(np.uint8)
    for dt in (3, 6):
        assert (zco.group_merge(zco.group_split(w, dt), dt) == w).all()


# ---------------------------------------------------------- normalisation

def test_normalize_golden(zco):
    for line in _golden_lines("normalize_cases.txt"):
        n_s, counts_s, expect_s, _why = [p.strip() for p in line.split("|")]
        counts = np.zeros(256, np.uint32)
        for kv in counts_s.split():
            k, v = kv.split(":")
            counts[int(k)] = int(v)
        expect = np.zeros(256, np.uint32)
        for kv in expect_s.split():
            k, v = kv.split(":")
            expect[int(k)] = int(v)
        assert (zco.normalize(counts, int(n_s)) == expect).all(), line


def test_normalize_invariants(zco):
    rng = np.random.default_rng(9)
    for trial in range(400):
        k = int(rng.integers(2, 257))
        n = int(rng.integers(k, 70000))
        p = rng.dirichlet(np.full(k, float(rng.choice([0.05, 0.5, 5.0]))))
        syms = rng.choice(256, k, replace=False)
        counts = np.zeros(256, np.uint32)
        np.add.at(counts, syms[rng.choice(k, n, p=p)], 1)
        if (counts > 0).sum() < 2:
            continue
        f = zco.normalize(counts, n)
        assert int(f.sum()) == 4096
        assert ((f > 0) == (counts > 0)).all()
        assert f.max() <= 4095
        # never farther from the exact share than the rounding and the
        # one-symbol correction allow
        exact = counts.astype(np.float64) * 4096 / n
        dev = np.abs(f - exact)
        big = int(np.argmax(counts))
        assert (np.delete(dev, big) <= max(1.0, float(k))).all()


def test_normalize_cost_near_entropy(zco):
    """Cross-entropy of the 12-bit table against the counts stays within 1%
    (plus a few bits) of the counts' own order-0 entropy."""
    rng = np.random.default_rng(2)
    for sigma in (0.02, 0.05, 1.0):
        x = torch.from_numpy((rng.standard_normal(65536) * sigma).astype(np.float32)).bfloat16()
        e = zco.group_split(x.view(torch.int16).numpy().view(np.uint8), 4)[0]
        counts = np.bincount(e, minlength=256).astype(np.uint32)
        f = zco.normalize(counts, e.size)
        nz = counts > 0
        H = float(-(counts[nz] * np.log2(counts[nz] / e.size)).sum())
        cost = float((counts[nz] * np.log2(4096.0 / f[nz])).sum())
        assert H - 1e-6 <= cost <= 1.01 * H + 64


# ------------------------------------------------------------------- rANS

@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_rans_exact_information_power_of_two(zco, bits):
    """With 2^b equally frequent symbols the table is f = 4096 / 2^b, and
    each coded symbol adds exactly b to floor(log2 x) while each word takes
    16 away, so sum_l (floor(log2 x_l) - 16) + 16 * nwords = b * n."""
    rng = np.random.default_rng(bits)
    k = 1 << bits
    for n in (k, 32 * k, 4096, 65536 - (65536 % k), 50000 - (50000 % k)):
        s = np.repeat(np.arange(k, dtype=np.uint8), n // k)
        rng.shuffle(s)
        rec = zco.rans_record(s)
        states = np.frombuffer(rec[:128], np.uint32).astype(np.int64)
        assert ((states >= L) & (states < 2**32)).all()
        words_at = 160 + (2 * k + 15) // 16 * 16
        nwords = (len(rec) - words_at) // 2
        info = sum(int(x).bit_length() - 1 - 16 for x in states) + 16 * nwords
        assert info == bits * n
        assert (zco.rans_decode(rec, n) == s).all()


def test_rans_roundtrip_streams(zco):
    rng = np.random.default_rng(4)
    for n in (2, 3, 31, 32, 33, 63, 64, 65, 1000, 4095, 4096, 4097, 32768, 65536):
        for dist in ("skew", "uniform", "two", "geom"):
            if dist == "skew":
                s = rng.choice(256, n, p=rng.dirichlet(np.full(256, 0.05)))
            elif dist == "uniform":
                s = rng.integers(0, 256, n)
            elif dist == "two":
                s = rng.choice([3, 250], n, p=[0.999, 0.001])
            else:
                s = np.minimum(rng.geometric(0.3, n), 255)
            s = s.astype(np.uint8)
            if np.unique(s).size < 2:
                s[0] ^= 1
            rec = zco.rans_record(s)
            assert (zco.rans_decode(rec, n) == s).all()


def test_tiny_blob_golden(zco):
    g = dict(line.split(None, 1) for line in _golden_lines("tiny_rans_blob.txt"))
    blob = zco.compress(np.array([0, 1], np.uint8), 1, (2,), chunk_bytes=64, threshold=1e6)
    assert len(blob) == int(g["blob_bytes"])
    table_end = int(g["table_end"])
    head = bytearray(96)
    head[0:4] = b"ZCNN"
    struct.pack_into("<HBBIBBHQI", head, 4, 1, int(g["dtype"]), int(g["ndim"]),
                     int(g["chunk_bytes"]), 32, 12, 0, int(g["nbytes"]), int(g["n_chunks"]))
    struct.pack_into("<q", head, 32, int(g["shape0"]))
    states = [int(g["state0"]), int(g["state1"])] + [int(g["state_rest"])] * 30
    rec = struct.pack("<32I", *states) + bytes([int(g["bitmap_byte0"], 16)]) + bytes(31)
    rec += struct.pack("<2H", *map(int, g["freqs"].split())) + bytes(12)
    assert len(rec) == 176 and int(g["nwords"]) == 0
    payload = struct.pack("<I", int(g["dir0"], 16)) + bytes(12) + rec
    assert len(payload) == int(g["chunk0_stored"])
    entry = struct.pack("<QII", int(g["chunk0_offset"]),
                        int(g["chunk0_stored"]) | (int(g["chunk0_raw"]) << 31),
                        zlib.crc32(payload))  # the stored payload bytes
    table = bytes(head) + entry
    assert len(table) == table_end
    hcrc = zlib.crc32(table)
    expect = table[:28] + struct.pack("<I", hcrc) + table[32:] + payload
    assert blob == expect


# ------------------------------------------------------- whole-blob checks

def _rand_tensor(rng, dtype, n):
    W = {1: 1, 2: 2, 3: 4, 4: 2, 5: 2, 6: 4}[dtype]
    kind = rng.integers(0, 6)
    if kind == 0:
        b = rng.integers(0, 256, n * W, dtype=np.uint8)
    elif kind == 1:
        b = np.full(n * W, rng.integers(0, 256), np.uint8)
    elif kind == 2:
        b = rng.choice(np.array([7, 9], np.uint8), n * W)
    else:
        sigma = float(rng.choice([0.02, 0.05, 1.0, 1e-3]))
        x = (rng.standard_normal(n) * sigma).astype(np.float32)
        if kind == 4 and n:
            x[rng.integers(0, n, max(1, n // 50))] = np.nan
        t = torch.from_numpy(x)
        if dtype == 4:
            t = t.bfloat16()
        elif dtype == 5:
            t = t.half()
        elif dtype in (1, 2, 3):
            b = rng.integers(0, 16, n * W, dtype=np.uint8)
            return b
        if kind == 5 and dtype == 6:
            t = t.bfloat16().float()
        b = t.numpy().view(np.uint8) if dtype == 6 else t.view(torch.int16).numpy().view(np.uint8)
    return np.ascontiguousarray(b).reshape(-1)


def test_roundtrip_random_tensors(zco):
    rng = np.random.default_rng(2024)
    for trial in range(240):
        dtype = int(rng.integers(1, 7))
        n = int(rng.choice([0, 1, 31, 32, 33, 4095, 4097, int(rng.integers(0, 5001))]))
        data = _rand_tensor(rng, dtype, n)
        shape = (n,) if trial % 3 else ((1, n) if trial % 2 else (n, 1))
        chunk = int(rng.choice([64, 4096, 131072]))
        thr = float(rng.choice([0.5, 0.95, 1.0, 2.0]))
        blob = zco.compress(data, dtype, shape, chunk, thr)
        assert len(blob) <= zco.blob_size(data.size, dtype, chunk, thr)
        info = zco.blob_info(blob)
        assert info["shape"] == tuple(shape) and info["dtype"] == dtype
        back = zco.decompress(blob)
        assert back.tobytes() == data.tobytes(), (trial, dtype, n, chunk, thr)
        if data.size <= 20000:
            assert spec_decoder.decode(blob) == data.tobytes()


def _chunk_modes(blob, W):
    """(raw chunk flags, per-chunk directory modes) read from a blob."""
    nc, = struct.unpack_from("<I", blob, 24)
    raws, modes = [], []
    for c in range(nc):
        off, sm, _ = struct.unpack_from("<QII", blob, 96 + 16 * c)
        raws.append(sm >> 31)
        modes.append(None if sm >> 31 else
                     [struct.unpack_from("<I", blob, off + 4 * j)[0] >> 30 for j in range(W)])
    return raws, modes


def test_exhaustive_bf16_patterns(zco):
    words = np.arange(65536, dtype=np.uint16).view(np.uint8)
    # (a) in order, one chunk: both streams are uniform, so the chunk is RAW
    blob = zco.compress(words, 4, (65536,), 131072, 0.95)
    raws, _ = _chunk_modes(blob, 2)
    assert raws == [1]
    assert (zco.decompress(blob) == words).all()
    # (b) in order, 4 KiB chunks: the exponent stream holds 16 values per
    # chunk (4 bits) and is coded; the sign|mantissa stream is 7 bits, RAW
    blob = zco.compress(words, 4, (65536,), 4096, 0.95)
    raws, modes = _chunk_modes(blob, 2)
    assert raws == [0] * 32 and all(m == [1, 0] for m in modes)
    assert (zco.decompress(blob) == words).all()
    # (c) shuffled with threshold 2: every stream is rANS-coded
    perm = np.random.default_rng(7).permutation(65536).astype(np.uint16)
    sh = perm.view(np.uint8)
    blob = zco.compress(sh, 4, (256, 256), 131072, 2.0)
    raws, modes = _chunk_modes(blob, 2)
    assert raws == [0] and modes == [[1, 1]]
    assert (zco.decompress(blob) == sh).all()


def test_entropy_bound_exponent_streams(zco):
    """Every coded exponent record: with H = n * (empirical order-0 entropy)
    / 8 bytes, H - 8 <= 2 * nwords + 128 <= 1.01 * H + 8."""
    tensors = [(workloads.bf16_1m(), 4), (workloads.fp32_64m(rows=256), 6),
               (workloads.fp32clean_64m(rows=256), 6)]
    for t, dt in tensors:
        raw = workloads.as_bytes(t).numpy()
        C = 131072
        for c in range(0, raw.size, C):
            chunk = raw[c:c + C]
            e = zco.group_split(chunk, dt)[0]
            counts = np.bincount(e, minlength=256)
            nz = counts[counts > 0]
            H = float(-(nz * np.log2(nz / e.size)).sum()) / 8
            rec = zco.rans_record(e)
            k = int((counts > 0).sum())
            nwords = (len(rec) - 160 - (2 * k + 15) // 16 * 16) // 2
            assert H - 8 <= 2 * nwords + 128 <= 1.01 * H + 8, (dt, c)


def _group_sizes(blob, W, stream_bytes):
    """Per-stream stored bytes (RAW chunks count fully) as % of the input."""
    nc, = struct.unpack_from("<I", blob, 24)
    sizes = [0] * W
    for c in range(nc):
        off, sm, _ = struct.unpack_from("<QII", blob, 96 + 16 * c)
        if sm >> 31:
            for j in range(W):
                sizes[j] += (sm & 0x7FFFFFFF) // W
            continue
        for j in range(W):
            entry, = struct.unpack_from("<I", blob, off + 4 * j)
            mode, v = entry >> 30, entry & 0x3FFFFFFF
            sizes[j] += 0 if mode == 2 else v
    return [100.0 * s / stream_bytes for s in sizes]


def test_sizes_near_table2(zco):
    gens = {"bf16_1m": lambda: workloads.bf16_1m(),
            "fp32_64m": lambda: workloads.fp32_64m(rows=512),
            "fp16_16m": lambda: workloads.fp16_16m(rows=1024),
            "fp32clean_64m": lambda: workloads.fp32clean_64m(rows=512)}
    for line in _golden_lines("table2_sizes.txt"):
        name, _model, total, groups, tol_total, tol_exp = line.split()
        t = gens[name]()
        dt = workloads.dtype_code(t)
        raw = workloads.as_bytes(t).numpy()
        blob = zco.compress(raw, dt, tuple(t.shape))
        W = raw.size // t.numel()
        got_total = 100.0 * len(blob) / raw.size
        assert abs(got_total - float(total)) <= float(tol_total), (name, got_total)
        got = _group_sizes(blob, W, raw.size // W)
        want = [float(g) for g in groups.split(",")]
        assert abs(got[0] - want[0]) <= float(tol_exp), (name, got)
        for g, w in zip(got[1:], want[1:]):
            assert abs(g - w) <= 2.0 or (w == 100 and g >= 99), (name, got)


def test_corruption_detected(zco):
    rng = np.random.default_rng(8)
    t = workloads.bf16_1m()[:64]
    raw = workloads.as_bytes(t).numpy()
    blob = zco.compress(raw, 4, tuple(t.shape), 4096, 0.95)
    for pos in list(range(0, 160)) + list(rng.integers(0, len(blob), 400)):
        bad = bytearray(blob)
        bad[pos] ^= int(rng.integers(1, 256))
        st, out = zco.decompress_status(bytes(bad))
        assert st != 0 or out.tobytes() == raw.tobytes(), pos
    # truncated blobs are rejected, never read past their end
    for cut in (0, 50, 96, 100, len(blob) - 1):
        st, _ = zco.decompress_status(blob[:cut])
        assert st != 0


def test_chunk_crc_is_checked_before_decoding(zco):
    """cuZipNN API: the CRC-32s are taken over pieces of the blob so that an
    untrusted blob can be rejected before it is decoded. A changed payload
    byte fails its chunk's CRC; that chunk is reported and never decoded (so
    no structural error is raised from inside it), the other chunks decode
    exactly, and the check without decoding (verify) reports the same. Bytes
    of the zero padding between payloads are outside every CRC."""
    rng = np.random.default_rng(31)
    t = workloads.bf16_1m()[:48]
    raw = workloads.as_bytes(t).numpy()
    C = 4096
    blob = zco.compress(raw, 4, tuple(t.shape), C, 0.95)
    assert zco.verify(blob) == 0
    nc, = struct.unpack_from("<I", blob, 24)
    entries = [struct.unpack_from("<QII", blob, 96 + 16 * c) for c in range(nc)]
    for c, (off, sm, crc) in enumerate(entries):
        stored = sm & 0x7FFFFFFF
        assert crc == zlib.crc32(blob[off:off + stored]), c
        for pos in (off, off + stored - 1, off + int(rng.integers(0, stored))):
            bad = bytearray(blob)
            bad[pos] ^= int(rng.integers(1, 256))
            st, out = zco.decompress_status(bytes(bad))
            assert st == zco.ECRC, (c, pos)
            assert zco.verify(bytes(bad)) == zco.ECRC
            keep = np.ones(raw.size, bool)
            keep[c * C:(c + 1) * C] = False
            assert (out[keep] == raw[keep]).all()
    # a header or table byte: caught by the header CRC or the layout checks
    for pos in list(range(0, 96, 7)) + [96 + 16 * c + 13 for c in range(nc)]:
        bad = bytearray(blob)
        bad[pos] ^= 0x40
        assert zco.verify(bytes(bad)) & (zco.EFORMAT | zco.ECRC), pos
    # truncated: a payload outside the blob
    assert zco.verify(blob[:-16]) & zco.EFORMAT


def test_no_verify_flag_still_checks_structure(zco):
    t = workloads.bf16_1m()[:16]
    raw = workloads.as_bytes(t).numpy()
    blob = bytearray(zco.compress(raw, 4, tuple(t.shape), 4096, 0.95))
    off, sm, _ = struct.unpack_from("<QII", blob, 96)
    assert not sm >> 31
    struct.pack_into("<I", blob, off, 3 << 30)  # an undefined stream mode
    st, _ = zco.decompress_status(bytes(blob), zco.NO_VERIFY)
    assert st & zco.ECORRUPT


def test_header_rejections(zco):
    blob = zco.compress(np.arange(100, dtype=np.uint8), 1, (100,), 64, 0.95)
    bad = bytearray(blob)
    bad[4] = 2  # another format version
    assert zco.decompress_status(bytes(bad))[0] & zco.EFORMAT
    bad = bytearray(blob)
    bad[0] = ord("X")
    assert zco.decompress_status(bytes(bad))[0] & zco.EFORMAT
    bad = bytearray(blob)
    bad[40] ^= 1  # shape field: caught by the header CRC or the shape check
    assert zco.decompress_status(bytes(bad))[0] != 0


def test_param_validation(zco):
    assert zco.blob_size(10, 4, 131072, 0.95) > 0  # five BF16 words
    assert zco.blob_size(11, 4, 131072, 0.95) == 0
    assert zco.blob_size(64, 1, 100, 0.95) == 0
    assert zco.blob_size(64, 1, 131072 + 64, 0.95) == 0
    assert zco.blob_size(64, 1, 64, 0.0) == 0
    assert zco.blob_size(64, 9, 64, 0.95) == 0
    assert zco.blob_size(0, 1, 64, 0.95) == 96


# ------------------------------------------------- format v2 (shared tables)
# lmz "Building on lmz": one table per plane kind shared by many chunks. The
# v2 pins tie it to the pinned v1 coder (a one-chunk tensor's plane table is
# the table v1 stores in that chunk's record, and the v2 record is the v1
# record without its table), to the independent reader, to the entropy, and
# to the rule's invariants with 64-bit counts.

def _v1_records(blob, W):
    """{stream j: record bytes} of the single grouped chunk of a v1 blob."""
    off, sm, _ = struct.unpack_from("<QII", blob, 96)
    assert not sm >> 31
    pos, recs = 16, {}
    for j in range(W):
        entry, = struct.unpack_from("<I", blob, off + 4 * j)
        mode, v = entry >> 30, entry & 0x3FFFFFFF
        if mode == 1:
            recs[j] = blob[off + pos: off + pos + v]
        if mode != 2:
            pos += (v + 15) // 16 * 16
    return recs


def test_v2_single_chunk_equals_v1_records(zco):
    rng = np.random.default_rng(31)
    cases = [(workloads.as_bytes(workloads.bf16_1m()[:32]).numpy(), 4),
             (workloads.as_bytes(workloads.fp32_64m(rows=1)[:, :4000]).numpy(), 6),
             (rng.integers(0, 9, 20000, dtype=np.uint8), 1),
             ((rng.integers(0, 4, 6000, dtype=np.uint16) * 257).view(np.uint8), 2)]
    for raw, dt in cases:
        W = {1: 1, 2: 2, 4: 2, 6: 4}[dt]
        b1 = zco.compress(raw, dt, None, 131072, 2.0)   # threshold 2: every non-constant stream coded
        b2 = zco.compress(raw, dt, None, 131072, 2.0, version=2)
        planes = zco.plane_tables(raw, dt)
        nc, = struct.unpack_from("<I", b2, 24)
        stored = np.frombuffer(b2[96 + 16 * nc: 96 + 16 * nc + 512 * W], "<u2").reshape(W, 256)
        assert (stored == planes).all()
        recs1 = _v1_records(b1, W)
        off2, _, _ = struct.unpack_from("<QII", b2, 96)
        pos = 16
        for j in range(W):
            entry, = struct.unpack_from("<I", b2, off2 + 4 * j)
            mode, v = entry >> 30, entry & 0x3FFFFFFF
            if j in recs1:
                r1 = recs1[j]
                bitmap = r1[128:160]
                present = [s for s in range(256) if bitmap[s // 8] >> (s % 8) & 1]
                k = len(present)
                f1 = dict(zip(present, struct.unpack_from(f"<{k}H", r1, 160)))
                assert {s: int(planes[j][s]) for s in range(256) if planes[j][s]} == f1
                words1 = r1[160 + (2 * k + 15) // 16 * 16:]
                assert mode == 1 and b2[off2 + pos: off2 + pos + v] == r1[:128] + words1
            if mode != 2:
                pos += (v + 15) // 16 * 16
        assert zco.decompress(b2).tobytes() == raw.tobytes()
        assert spec_decoder.decode(b2) == raw.tobytes()


def test_v2_roundtrip_random_tensors(zco):
    rng = np.random.default_rng(4096)
    for trial in range(160):
        dtype = int(rng.integers(1, 7))
        n = int(rng.choice([0, 1, 31, 33, 4097, int(rng.integers(0, 6001))]))
        data = _rand_tensor(rng, dtype, n)
        chunk = int(rng.choice([64, 1024, 4096, 131072]))
        thr = float(rng.choice([0.5, 0.95, 1.0, 2.0]))
        blob = zco.compress(data, dtype, (n,), chunk, thr, version=2)
        assert len(blob) <= zco.blob_size(data.size, dtype, chunk, thr, version=2)
        info = zco.blob_info(blob)
        assert info["version"] == 2 and info["dtype"] == dtype
        assert zco.decompress(blob).tobytes() == data.tobytes(), (trial, dtype, n, chunk, thr)
        if data.size <= 20000:
            assert spec_decoder.decode(blob) == data.tobytes()


def test_v2_exhaustive_bf16_patterns(zco):
    """All 65,536 BF16 patterns shuffled over 4 KiB chunks, every stream coded
    (threshold 2) with the two plane tables of the whole tensor (each plane is
    uniform over the tensor: f = 16 for all 256 symbols)."""
    perm = np.random.default_rng(9).permutation(65536).astype(np.uint16).view(np.uint8)
    planes = zco.plane_tables(perm, 4, 4096)
    assert (planes == 16).all()
    blob = zco.compress(perm, 4, (65536,), 4096, 2.0, version=2)
    nc, = struct.unpack_from("<I", blob, 24)
    assert nc == 32
    assert zco.decompress(blob).tobytes() == perm.tobytes()
    assert spec_decoder.decode(blob) == perm.tobytes()


def test_v2_plane_tables_invariants(zco):
    rng = np.random.default_rng(77)
    t = workloads.fp32_64m(rows=64)
    raw = workloads.as_bytes(t).numpy()
    planes = zco.plane_tables(raw, 6, 131072)
    streams = zco.group_split(raw, 6)
    for j in range(4):
        counts = np.bincount(streams[j], minlength=256)
        f = planes[j]
        assert f.sum() == 4096 and ((f > 0) == (counts > 0)).all()
        nz = counts > 0
        H = float(-(counts[nz] * np.log2(counts[nz] / counts.sum())).sum())
        cost = float((counts[nz] * np.log2(4096.0 / f[nz])).sum())
        assert H - 1e-6 <= cost <= 1.01 * H + 64
    # a plane with one symbol over the tensor has an all-zero table
    clean = workloads.as_bytes(workloads.fp32clean_64m(rows=4)).numpy()
    p2 = zco.plane_tables(clean, 6, 131072)
    assert (p2[2] == 0).all() and (p2[3] == 0).all() and p2[0].sum() == 4096
    # the 64-bit rule reduces to the 32-bit one, and depends on ratios only
    for _ in range(20):
        counts = rng.integers(0, 5000, 256) * (rng.random(256) < 0.3)
        counts[int(rng.integers(0, 256))] += 1
        counts[int(rng.integers(0, 256))] += 1
        n = int(counts.sum())
        f32 = zco.normalize(counts.astype(np.uint32), n)
        assert (zco.normalize64(counts.astype(np.uint64), n) == f32).all()
        big = counts.astype(np.uint64) << np.uint64(20)
        assert (zco.normalize64(big, n << 20) == f32).all()


def test_v2_entropy_bound_and_size(zco):
    """Coded exponent records are within the cross-entropy under the plane
    table (H_x - 8 <= record <= 1.01 H_x + 8, in bytes), and the shared
    tables cost little against per-chunk tables on a stationary tensor."""
    for t, dt in [(workloads.bf16_1m(), 4), (workloads.fp32_64m(rows=256), 6)]:
        raw = workloads.as_bytes(t).numpy()
        planes = zco.plane_tables(raw, dt)
        f = planes[0].astype(np.float64)
        C = 131072
        for c in range(0, raw.size, C):
            e = zco.group_split(raw[c:c + C], dt)[0]
            counts = np.bincount(e, minlength=256)
            nz = counts > 0
            Hx = float((counts[nz] * np.log2(4096.0 / f[nz])).sum()) / 8
            rec = zco.rans_record_shared(e, planes[0])
            assert Hx - 8 <= len(rec) <= 1.01 * Hx + 8, (dt, c)
            assert (zco.rans_decode_shared(rec, e.size, planes[0]) == e).all()
        b1 = zco.compress(raw, dt, None, C, 0.95)
        b2 = zco.compress(raw, dt, None, C, 0.95, version=2)
        assert len(b2) <= 1.003 * len(b1) + 2048


def test_v2_rejections(zco):
    raw = workloads.as_bytes(workloads.bf16_1m()[:64]).numpy()
    blob = bytearray(zco.compress(raw, 4, None, 131072, 0.95, version=2))
    nc, = struct.unpack_from("<I", blob, 24)
    t0 = 96 + 16 * nc
    bad = bytearray(blob)
    bad[t0 + 2 * 120] ^= 1                      # a plane table no longer sums to 4096
    st, _ = zco.decompress_status(bytes(bad))
    assert st & (zco.EFORMAT | zco.ECRC)
    bad = bytearray(blob)
    bad[4] = 4                                   # unknown version
    st, _ = zco.decompress_status(bytes(bad))
    assert st & zco.EFORMAT


# ------------------------------------------- format v3 (a word list per lane)
# lmz "On a GPU": the decoder is bound by each lane's dependent chain; v3
# gives every lane its own word list so that no step waits on the others.

def _v3_head(rec: bytes) -> int:
    k = sum(bin(b).count("1") for b in rec[128:160])
    return 160 + (2 * k + 15) // 16 * 16


def test_v3_lane_lists_are_the_v1_words_by_lane(zco):
    """A v3 record holds exactly the v1 record's states, table and words,
    with lane l's list the words lane l takes when the v1 record is decoded
    by the independent reader, in reverse order of taking (the order the
    lane emitted them). This ties v3 to the pinned v1 coder."""
    rng = np.random.default_rng(303)
    for n in (2, 31, 32, 33, 100, 1000, 4095, 4097, 32768, 65536):
        for dist in ("skew", "uniform", "geom"):
            if dist == "skew":
                s = rng.choice(256, n, p=rng.dirichlet(np.full(256, 0.05)))
            elif dist == "uniform":
                s = rng.integers(0, 256, n)
            else:
                s = np.minimum(rng.geometric(0.3, n), 255)
            s = s.astype(np.uint8)
            if np.unique(s).size < 2:
                s[0] ^= 1
            r1, r3 = zco.rans_record(s), zco.rans_record_lanes(s)
            head = _v3_head(r1)
            assert r3[:head] == r1[:head]
            owners: list[int] = []
            assert spec_decoder._rans(r1, n, owners=owners) == s.tolist()
            words = struct.unpack_from(f"<{(len(r1) - head) // 2}H", r1, head)
            assert len(owners) == len(words)
            want = [[] for _ in range(32)]
            for i, lane in enumerate(owners):       # the i-th word taken is words[-1 - i]
                want[lane].append(words[len(words) - 1 - i])
            want = [w[::-1] for w in want]
            assert spec_decoder._lane_lists(r3, head) == want
            assert len(r3) == head + 64 + sum(2 * (len(w) + -len(w) % 8) for w in want)
            assert (zco.rans_decode_lanes(r3, n) == s).all()
            assert spec_decoder._rans(r3, n, lanes=True) == s.tolist()


def test_v3_tiny_blob_golden(zco):
    g = dict(line.split(None, 1) for line in _golden_lines("tiny_v3_blob.txt"))
    blob = zco.compress(np.array([0, 1], np.uint8), 1, (2,), chunk_bytes=64, threshold=1e6, version=3)
    assert len(blob) == int(g["blob_bytes"])
    head = bytearray(96)
    head[0:4] = b"ZCNN"
    struct.pack_into("<HBBIBBHQI", head, 4, int(g["version"]), 1, 1, 64, 32, 12, 0, 2, 1)
    struct.pack_into("<q", head, 32, 2)
    states = [int(g["state0"]), int(g["state1"])] + [int(g["state_rest"])] * 30
    rec = struct.pack("<32I", *states) + bytes([int(g["bitmap_byte0"], 16)]) + bytes(31)
    rec += struct.pack("<2H", *map(int, g["freqs"].split())) + bytes(12)
    rec += struct.pack("<32H", *([int(g["counts"])] * 32))
    payload = struct.pack("<I", int(g["dir0"], 16)) + bytes(12) + rec
    assert len(payload) == int(g["chunk0_stored"])
    entry = struct.pack("<QII", int(g["table_end"]), int(g["chunk0_stored"]), zlib.crc32(payload))
    table = bytes(head) + entry
    assert len(table) == int(g["table_end"])
    expect = table[:28] + struct.pack("<I", zlib.crc32(table)) + table[32:] + payload
    assert blob == expect


def test_v3_roundtrip_random_tensors(zco):
    rng = np.random.default_rng(333)
    for trial in range(160):
        dtype = int(rng.integers(1, 7))
        n = int(rng.choice([0, 1, 31, 33, 4097, int(rng.integers(0, 6001))]))
        data = _rand_tensor(rng, dtype, n)
        chunk = int(rng.choice([64, 1024, 4096, 131072]))
        thr = float(rng.choice([0.5, 0.95, 1.0, 2.0]))
        blob = zco.compress(data, dtype, (n,), chunk, thr, version=3)
        assert len(blob) <= zco.blob_size(data.size, dtype, chunk, thr, version=3)
        info = zco.blob_info(blob)
        assert info["version"] == 3 and info["dtype"] == dtype
        assert zco.decompress(blob).tobytes() == data.tobytes(), (trial, dtype, n, chunk, thr)
        assert zco.verify(blob) == 0
        if data.size <= 20000:
            assert spec_decoder.decode(blob) == data.tobytes()


def test_v3_exhaustive_bf16_patterns(zco):
    """All 65,536 BF16 patterns: in order over 4 KiB chunks (exponent coded,
    sign|mantissa RAW) and shuffled with every stream coded (threshold 2)."""
    words = np.arange(65536, dtype=np.uint16).view(np.uint8)
    blob = zco.compress(words, 4, (65536,), 4096, 0.95, version=3)
    raws, modes = _chunk_modes(blob, 2)
    assert raws == [0] * 32 and all(m == [1, 0] for m in modes)
    assert (zco.decompress(blob) == words).all()
    perm = np.random.default_rng(7).permutation(65536).astype(np.uint16).view(np.uint8)
    blob = zco.compress(perm, 4, (256, 256), 131072, 2.0, version=3)
    raws, modes = _chunk_modes(blob, 2)
    assert raws == [0] and modes == [[1, 1]]
    assert (zco.decompress(blob) == perm).all()
    assert spec_decoder.decode(blob) == perm.tobytes()


def test_v3_size_and_corruption(zco):
    """v3 costs at most the counts and the list padding per coded record
    over v1, and a changed byte anywhere is detected (CRC or structure)."""
    raw = workloads.as_bytes(workloads.bf16_1m()).numpy()
    b1 = zco.compress(raw, 4, None, 131072, 0.95)
    b3 = zco.compress(raw, 4, None, 131072, 0.95, version=3)
    nc = raw.size // 131072
    assert len(b1) < len(b3) <= len(b1) + nc * pad16(64 + 14 * 32)
    rng = np.random.default_rng(77)
    small = zco.compress(raw[:8192], 4, None, 4096, 0.95, version=3)
    for pos in list(rng.integers(0, len(small), 200)):
        bad = bytearray(small)
        bad[pos] ^= int(rng.integers(1, 256))
        st, out = zco.decompress_status(bytes(bad))
        assert st != 0 or out.tobytes() == raw[:8192].tobytes(), pos
        # without the CRC check a changed raw byte decodes silently; the
        # structure checks still keep every read within the blob
        zco.decompress_status(bytes(bad), zco.NO_VERIFY)


def pad16(x: int) -> int:
    return (x + 15) // 16 * 16
