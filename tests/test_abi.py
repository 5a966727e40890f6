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


def test_delta_entry_points_reject_bad_arguments_on_the_host():
    """The delta entry points check dtype and alignment before any launch
    (the pointers below are never dereferenced)."""
    import ctypes
    import entropy_coding_gb300 as zc
    L = zc.lib()
    shape = (ctypes.c_int64 * 1)(1024)
    aligned, odd = 0x10000, 0x10008
    args = dict(nbytes=2048, ndim=1, shape=shape, chunk=4096, thr=0.95, blob=aligned, cap=1 << 16, nb=aligned,
                ws=aligned, wsb=1 << 20, st=aligned, stream=None)

    def comp(base, new, dtype):
        return L.zc_compress_delta(base, new, args["nbytes"], dtype, args["ndim"], args["shape"], args["chunk"],
                                   args["thr"], args["blob"], args["cap"], args["nb"], args["ws"], args["wsb"],
                                   args["st"], args["stream"])
    for dt in (zc.BF16, zc.FP16, zc.FP32, 0, 9):
        assert comp(aligned, aligned, dt) == zc.EINVAL
    assert comp(odd, aligned, zc.U16) == zc.EINVAL
    assert comp(aligned, odd, zc.U16) == zc.EINVAL
    assert comp(None, aligned, zc.U16) == zc.EINVAL

    info = zc._Info()
    info.dtype, info.ndim, info.nbytes, info.n_chunks, info.chunk_bytes = zc.BF16, 1, 2048, 1, 4096
    info.shape[0] = 1024
    info.blob_bytes = 1 << 12
    assert L.zc_decompress_delta(aligned, ctypes.byref(info), aligned, aligned, 2048, 0, aligned, None) == zc.EINVAL
    info.dtype = zc.U16
    assert L.zc_decompress_delta(aligned, ctypes.byref(info), odd, aligned, 2048, 0, aligned, None) == zc.EINVAL
    assert L.zc_decompress_delta(aligned, ctypes.byref(info), aligned, odd, 2048, 0, aligned, None) == zc.EINVAL
