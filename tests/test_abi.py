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
    info.version = 1
    assert L.zc_decompress_delta(aligned, ctypes.byref(info), aligned, aligned, 2048, 0, aligned, None) == zc.EINVAL
    info.dtype = zc.U16
    assert L.zc_decompress_delta(aligned, ctypes.byref(info), odd, aligned, 2048, 0, aligned, None) == zc.EINVAL
    assert L.zc_decompress_delta(aligned, ctypes.byref(info), aligned, odd, 2048, 0, aligned, None) == zc.EINVAL


def test_batch_entry_points_reject_bad_arguments_on_the_host():
    """The batched entry points check every tensor (blob) before any launch
    (the device pointers below are never dereferenced)."""
    import ctypes
    import entropy_coding_gb300 as zc
    L = zc.lib()
    aligned = 0x10000
    vp2 = ctypes.c_void_p * 2
    u64_2 = ctypes.c_uint64 * 2
    ndims = (ctypes.c_int32 * 2)(1, 1)
    shapes = (ctypes.c_int64 * 16)(*([1024] + [0] * 7 + [1024] + [0] * 7))

    def comp(n, srcs, bases, nbytes, dtype, nd=ndims, flags=0):
        return L.zc_compress_batch(n, srcs, bases, nbytes, dtype, nd, shapes, 4096, 0.95, flags,
                                   vp2(aligned, aligned), u64_2(1 << 16, 1 << 16), aligned, aligned, 1 << 24,
                                   aligned, None)
    assert comp(0, None, None, None, zc.BF16) == zc.OK
    assert comp(0, None, None, None, zc.BF16, flags=16) == zc.EINVAL  # unknown flag
    assert comp(0, None, None, None, zc.BF16, flags=6) == zc.EINVAL   # two formats at once
    assert comp(0, None, None, None, zc.BF16, flags=zc.PACKED | zc.LANE_WORDS) == zc.OK
    assert comp(2, None, None, u64_2(2048, 2048), zc.BF16) == zc.EINVAL
    # deltas only for unsigned word dtypes
    assert comp(2, vp2(aligned, aligned), vp2(aligned, aligned), u64_2(2048, 2048), zc.BF16) == zc.EINVAL
    # the second tensor's shape does not match its size
    assert comp(2, vp2(aligned, aligned), None, u64_2(2048, 4096), zc.BF16) == zc.EINVAL
    # a misaligned second source
    assert comp(2, vp2(aligned, aligned + 1), None, u64_2(2048, 2048), zc.BF16) == zc.EINVAL

    infos = (zc._Info * 2)()
    for i, dt in enumerate((zc.BF16, zc.FP32)):
        infos[i].dtype, infos[i].ndim, infos[i].n_chunks, infos[i].chunk_bytes = dt, 1, 1, 4096
        infos[i].nbytes = 2048 if dt == zc.BF16 else 4096
        infos[i].shape[0] = 1024
        infos[i].blob_bytes = 1 << 12
        infos[i].version = 1
    caps = u64_2(1 << 16, 1 << 16)
    ws = zc.decompress_workspace_size_batch(2)
    assert ws >= 2 * 48 and zc.decompress_workspace_size_batch(1) == 0
    # mixed dtypes in one batch
    assert L.zc_decompress_batch(2, vp2(aligned, aligned), infos, None, vp2(aligned, aligned), caps, 0, aligned,
                                 ws, aligned, None) == zc.EINVAL
    infos[1].dtype, infos[1].nbytes = zc.BF16, 2048
    # no workspace for the descriptor table
    assert L.zc_decompress_batch(2, vp2(aligned, aligned), infos, None, vp2(aligned, aligned), caps, 0, None, 0,
                                 aligned, None) == zc.EINVAL
    # an output too small for the second blob
    assert L.zc_decompress_batch(2, vp2(aligned, aligned), infos, None, vp2(aligned, aligned), u64_2(1 << 16, 16),
                                 0, aligned, ws, aligned, None) == zc.ECAPACITY
    assert L.zc_decompress_batch(0, None, None, None, None, None, 0, None, 0, None, None) == zc.OK
    assert zc.workspace_size_batch([2048, 3], zc.BF16, 4096) == 0
    assert zc.workspace_size_batch([2048, 0], zc.BF16, 4096, zc.SHARED_TABLES) > 0
    assert zc.blob_size(2048, zc.BF16, 4096, 0.95, zc.SHARED_TABLES) == zc.blob_size(2048, zc.BF16, 4096) + 1024
    assert zc.workspace_size_batch([2048, 0], zc.BF16, 4096) > 0


def test_packed_flag_is_a_launch_choice_on_the_host():
    """ZC_PACKED combines with every format and with ZC_NO_VERIFY and sizes
    nothing differently; unknown bits are refused before any launch (the
    device pointers below are never dereferenced)."""
    import ctypes
    import entropy_coding_gb300 as zc
    L = zc.lib()
    for fmt in (0, zc.SHARED_TABLES, zc.LANE_WORDS):
        for nb in (0, 1000, 1 << 20):
            assert L.zc_blob_size_ex(nb, zc.BF16, 4096, 0.95, fmt | zc.PACKED) == L.zc_blob_size_ex(
                nb, zc.BF16, 4096, 0.95, fmt)
            assert L.zc_workspace_size_ex(nb, zc.BF16, 4096, fmt | zc.PACKED) == L.zc_workspace_size_ex(
                nb, zc.BF16, 4096, fmt)
    assert L.zc_blob_size_ex(1000, zc.BF16, 4096, 0.95, 16) == 0
    aligned = 0x10000
    info = zc._info_struct({"version": 1, "dtype": zc.BF16, "ndim": 1, "shape": [512], "nbytes": 1024,
                            "chunk_bytes": 4096, "n_chunks": 1, "blob_bytes": 4096})
    assert L.zc_decompress(aligned, ctypes.byref(info), aligned, 2048, 16, aligned, None) == zc.EINVAL
    assert L.zc_decompress(aligned, ctypes.byref(info), aligned, 2048, 32 | zc.PACKED, aligned, None) == zc.EINVAL
