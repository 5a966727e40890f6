"""CPU checks of the C-ABI library: it loads, exports every symbol that
include/zc.h declares, and its host-only entry points (sizes, header
parsing) agree with the oracle. No kernel is launched."""
from __future__ import annotations

import os
import re
import struct

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "zc.h")).read()
    return sorted(set(re.findall(r"^\w[\w\s\*]*?\b(zc_\w+)\s*\(", src, re.M)))


def test_library_exports_every_declared_symbol():
    import entropy_coding_gb300 as zc
    L = zc.lib()
    names = _declared()
    assert set(names) >= {"zc_blob_size", "zc_workspace_size", "zc_blob_info", "zc_compress",
                          "zc_decompress", "zc_crc32"}
    for n in names:
        assert hasattr(L, n), n


def test_blob_size_matches_oracle(zco):
    import entropy_coding_gb300 as zc
    for nbytes, dt, C, thr in [(0, 4, 131072, 0.95), (2, 4, 64, 0.95), (2 << 20, 4, 131072, 0.95),
                               (12345 * 4, 6, 4096, 2.0), (777, 1, 64, 1.0), (10, 4, 100, 0.95),
                               (11, 4, 64, 0.95), (64, 1, 64, 0.0), (64, 9, 64, 0.95)]:
        assert zc.blob_size(nbytes, dt, C, thr) == zco.blob_size(nbytes, dt, C, thr)


def test_blob_info_matches_oracle(zco):
    import entropy_coding_gb300 as zc
    rng = np.random.default_rng(1)
    for dt, n, C in [(4, 3000, 4096), (6, 1000, 64), (1, 0, 64), (2, 77, 131072)]:
        W = zco.WORD_BYTES[dt]
        data = rng.integers(0, 8, n * W, dtype=np.uint8)
        blob = zco.compress(data, dt, (n,), C, 0.95)
        got = zc.blob_info(blob)
        ref = zco.blob_info(blob)
        for k in ("dtype", "ndim", "shape", "nbytes", "n_chunks", "chunk_bytes", "blob_bytes"):
            assert got[k] == ref[k], k
        bad = bytearray(blob)
        bad[28] ^= 1
        with pytest.raises(zc.ZcError) as e:
            zc.blob_info(bytes(bad))
        assert e.value.status == zc.ECRC
        bad = bytearray(blob)
        bad[4] = 2
        with pytest.raises(zc.ZcError) as e:
            zc.blob_info(bytes(bad))
        assert e.value.status == zc.EFORMAT


def test_blob_info_rejects_moved_offsets(zco):
    import entropy_coding_gb300 as zc
    import zlib
    data = np.arange(4096, dtype=np.uint8)
    blob = bytearray(zco.compress(data, 1, (4096,), 1024, 0.95))
    off, = struct.unpack_from("<Q", blob, 96 + 16)
    struct.pack_into("<Q", blob, 96 + 16, off + 16)      # second chunk's offset moved
    head = bytearray(blob[:96 + 16 * 4])
    head[28:32] = b"\0\0\0\0"
    struct.pack_into("<I", blob, 28, zlib.crc32(bytes(head)))  # with a valid header CRC
    with pytest.raises(zc.ZcError) as e:
        zc.blob_info(bytes(blob))
    assert e.value.status == zc.EFORMAT
