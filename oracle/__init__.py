"""CPU oracle for the compressor — TEST INFRASTRUCTURE ONLY.

A plain single-threaded C program (``zco.c``) that defines the blob format
and the exact bytes a compressor must produce. Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package; the GPU
library never does, and this package never touches the GPU library.

This module builds ``libzco.so`` with gcc and wraps it with ctypes over numpy
arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zco.c")
_LIB_PATH = os.path.join(_HERE, "libzco.so")
_lock = threading.Lock()
_lib = None

U8, U16, U32, BF16, FP16, FP32 = 1, 2, 3, 4, 5, 6
WORD_BYTES = {U8: 1, U16: 2, U32: 4, BF16: 2, FP16: 2, FP32: 4}
OK, EINVAL, EFORMAT, ECRC, ECORRUPT, ECAPACITY = 0, 1, 2, 4, 8, 32
NO_VERIFY = 1


def build(force: bool = False) -> str:
    """Compile zco.c into libzco.so (plain C, -O2, no vector extensions)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "zco.h"))
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
             "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            c_u8p = ctypes.c_void_p
            L.zco_crc32.restype = ctypes.c_uint32
            L.zco_crc32.argtypes = [c_u8p, ctypes.c_uint64]
            L.zco_word_bytes.restype = ctypes.c_int
            L.zco_word_bytes.argtypes = [ctypes.c_int]
            L.zco_group_split.restype = None
            L.zco_group_split.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_int, c_u8p]
            L.zco_group_merge.restype = None
            L.zco_group_merge.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_int, c_u8p]
            L.zco_normalize.restype = ctypes.c_int
            L.zco_normalize.argtypes = [c_u8p, ctypes.c_uint32, c_u8p]
            L.zco_rans_record.restype = ctypes.c_uint64
            L.zco_rans_record.argtypes = [c_u8p, ctypes.c_uint32, c_u8p, ctypes.c_uint64]
            L.zco_rans_decode.restype = ctypes.c_int
            L.zco_rans_decode.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_uint32, c_u8p]
            L.zco_encode_chunk.restype = ctypes.c_uint64
            L.zco_encode_chunk.argtypes = [c_u8p, ctypes.c_uint32, ctypes.c_int, ctypes.c_double,
                                           c_u8p, ctypes.c_uint64, ctypes.POINTER(ctypes.c_int)]
            L.zco_blob_size.restype = ctypes.c_uint64
            L.zco_blob_size.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_uint32, ctypes.c_double]
            L.zco_compress.restype = ctypes.c_int
            L.zco_compress.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, c_u8p,
                                       ctypes.c_uint32, ctypes.c_double, c_u8p, ctypes.c_uint64,
                                       ctypes.POINTER(ctypes.c_uint64)]
            L.zco_blob_info.restype = ctypes.c_int
            L.zco_blob_info.argtypes = [c_u8p, ctypes.c_uint64, ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(ctypes.c_int), c_u8p,
                                        ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint32),
                                        ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint64)]
            L.zco_decompress.restype = ctypes.c_int
            L.zco_decompress.argtypes = [c_u8p, ctypes.c_uint64, c_u8p, ctypes.c_uint64, ctypes.c_uint32]
            L.zco_rans_record_lanes.restype = ctypes.c_uint64
            L.zco_rans_record_lanes.argtypes = [c_u8p, ctypes.c_uint32, c_u8p, ctypes.c_uint64]
            L.zco_rans_decode_lanes.restype = ctypes.c_int
            L.zco_rans_decode_lanes.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_uint32, c_u8p]
            L.zco_encode_chunk_lanes.restype = ctypes.c_uint64
            L.zco_encode_chunk_lanes.argtypes = [c_u8p, ctypes.c_uint32, ctypes.c_int, ctypes.c_double,
                                                 c_u8p, ctypes.c_uint64, ctypes.POINTER(ctypes.c_int)]
            L.zco_verify.restype = ctypes.c_int
            L.zco_verify.argtypes = [c_u8p, ctypes.c_uint64]
            L.zco_normalize64.restype = ctypes.c_int
            L.zco_normalize64.argtypes = [c_u8p, ctypes.c_uint64, c_u8p]
            L.zco_plane_tables.restype = ctypes.c_int
            L.zco_plane_tables.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_int, ctypes.c_uint32, c_u8p]
            L.zco_rans_record_shared.restype = ctypes.c_uint64
            L.zco_rans_record_shared.argtypes = [c_u8p, ctypes.c_uint32, c_u8p, c_u8p, ctypes.c_uint64]
            L.zco_rans_decode_shared.restype = ctypes.c_int
            L.zco_rans_decode_shared.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_uint32, c_u8p, c_u8p]
            L.zco_blob_size_v.restype = ctypes.c_uint64
            L.zco_blob_size_v.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_uint32, ctypes.c_double,
                                          ctypes.c_int]
            L.zco_compress_v.restype = ctypes.c_int
            L.zco_compress_v.argtypes = [c_u8p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, c_u8p,
                                         ctypes.c_uint32, ctypes.c_double, ctypes.c_int, c_u8p, ctypes.c_uint64,
                                         ctypes.POINTER(ctypes.c_uint64)]
            _lib = L
    return _lib


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(-1)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data if a.size else 0


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status}")
        self.status = status


def crc32(data) -> int:
    d = _u8(data)
    return int(lib().zco_crc32(_ptr(d), d.size))


def group_split(data, dtype: int) -> np.ndarray:
    d = _u8(data)
    W = WORD_BYTES[dtype]
    n = d.size // W
    out = np.empty(W * n, np.uint8)
    lib().zco_group_split(_ptr(d), n, dtype, _ptr(out))
    return out.reshape(W, n)


def group_merge(streams: np.ndarray, dtype: int) -> np.ndarray:
    s = np.ascontiguousarray(streams, dtype=np.uint8)
    W = WORD_BYTES[dtype]
    n = s.size // W
    out = np.empty(W * n, np.uint8)
    lib().zco_group_merge(_ptr(s), n, dtype, _ptr(out))
    return out


def normalize(counts, n: int) -> np.ndarray:
    c = np.ascontiguousarray(counts, dtype=np.uint32)
    assert c.size == 256
    f = np.zeros(256, np.uint32)
    st = lib().zco_normalize(_ptr(c), n, _ptr(f))
    if st:
        raise OracleError(st, "normalize")
    return f


def rans_record(symbols) -> bytes:
    s = _u8(symbols)
    cap = 160 + 512 + 2 * s.size + 16
    rec = np.zeros(cap, np.uint8)
    r = lib().zco_rans_record(_ptr(s), s.size, _ptr(rec), cap)
    if r == 0:
        raise OracleError(EINVAL, "rans_record")
    return rec[:r].tobytes()


def rans_decode(record: bytes, n: int) -> np.ndarray:
    r = np.frombuffer(record, np.uint8).copy()
    out = np.zeros(max(n, 1), np.uint8)
    st = lib().zco_rans_decode(_ptr(r), r.size, n, _ptr(out))
    if st:
        raise OracleError(st, "rans_decode")
    return out[:n]


def rans_record_lanes(symbols) -> bytes:
    """Format v3 record: a word list per lane."""
    s = _u8(symbols)
    cap = 160 + 512 + 64 + 2 * s.size + 16 * 32 + 16
    rec = np.zeros(cap, np.uint8)
    r = lib().zco_rans_record_lanes(_ptr(s), s.size, _ptr(rec), cap)
    if r == 0:
        raise OracleError(EINVAL, "rans_record_lanes")
    return rec[:r].tobytes()


def rans_decode_lanes(record: bytes, n: int) -> np.ndarray:
    r = np.frombuffer(record, np.uint8).copy()
    out = np.zeros(max(n, 1), np.uint8)
    st = lib().zco_rans_decode_lanes(_ptr(r), r.size, n, _ptr(out))
    if st:
        raise OracleError(st, "rans_decode_lanes")
    return out[:n]


def encode_chunk(chunk, dtype: int, threshold: float = 0.95, version: int = 1) -> tuple[bytes, bool]:
    """One chunk's stored payload (unpadded) and whether it is a RAW chunk
    (format v1, or v3 with a word list per lane)."""
    d = _u8(chunk)
    W = WORD_BYTES[dtype]
    cap = 16 + W * (160 + 512 + 64 + 16 * 32 + 2 * (d.size // W) + 16) + d.size
    out = np.zeros(cap, np.uint8)
    raw = ctypes.c_int(0)
    fn = lib().zco_encode_chunk_lanes if version == 3 else lib().zco_encode_chunk
    r = fn(_ptr(d), d.size, dtype, threshold, _ptr(out), cap, ctypes.byref(raw))
    if r == 0:
        raise OracleError(ECAPACITY, "encode_chunk")
    return out[:r].tobytes(), bool(raw.value)


def blob_size(nbytes: int, dtype: int, chunk_bytes: int = 131072, threshold: float = 0.95,
              version: int = 1) -> int:
    return int(lib().zco_blob_size_v(nbytes, dtype, chunk_bytes, threshold, version))


def compress(data, dtype: int, shape=None, chunk_bytes: int = 131072, threshold: float = 0.95,
             version: int = 1) -> bytes:
    """Blob of a tensor in format v1 (a table per coded stream), v2 (shared
    plane tables) or v3 (v1 with a word list per lane in each record)."""
    d = _u8(data)
    W = WORD_BYTES[dtype]
    if shape is None:
        shape = (d.size // W,)
    shp = np.zeros(8, np.int64)
    shp[: len(shape)] = shape
    cap = blob_size(d.size, dtype, chunk_bytes, threshold, version)
    if cap == 0:
        raise OracleError(EINVAL, "blob_size")
    blob = np.zeros(cap, np.uint8)
    nb = ctypes.c_uint64(0)
    st = lib().zco_compress_v(_ptr(d), d.size, dtype, len(shape), _ptr(shp), chunk_bytes, threshold, version,
                              _ptr(blob), cap, ctypes.byref(nb))
    if st:
        raise OracleError(st, "compress")
    return blob[: nb.value].tobytes()


def normalize64(counts, n: int) -> np.ndarray:
    c = np.ascontiguousarray(counts, dtype=np.uint64)
    assert c.size == 256
    f = np.zeros(256, np.uint32)
    st = lib().zco_normalize64(_ptr(c), n, _ptr(f))
    if st:
        raise OracleError(st, "normalize64")
    return f


def plane_tables(data, dtype: int, chunk_bytes: int = 131072) -> np.ndarray:
    """Format v2's W plane tables of a tensor, shape (W, 256)."""
    d = _u8(data)
    W = WORD_BYTES[dtype]
    out = np.zeros(W * 256, np.uint32)
    st = lib().zco_plane_tables(_ptr(d), d.size, dtype, chunk_bytes, _ptr(out))
    if st:
        raise OracleError(st, "plane_tables")
    return out.reshape(W, 256)


def rans_record_shared(symbols, f) -> bytes:
    s = _u8(symbols)
    t = np.ascontiguousarray(f, dtype=np.uint32)
    cap = 128 + 2 * s.size + 16
    rec = np.zeros(cap, np.uint8)
    r = lib().zco_rans_record_shared(_ptr(s), s.size, _ptr(t), _ptr(rec), cap)
    if r == 0:
        raise OracleError(EINVAL, "rans_record_shared")
    return rec[:r].tobytes()


def rans_decode_shared(record: bytes, n: int, f) -> np.ndarray:
    r = np.frombuffer(record, np.uint8).copy()
    t = np.ascontiguousarray(f, dtype=np.uint32)
    out = np.zeros(max(n, 1), np.uint8)
    st = lib().zco_rans_decode_shared(_ptr(r), r.size, n, _ptr(t), _ptr(out))
    if st:
        raise OracleError(st, "rans_decode_shared")
    return out[:n]


def blob_info(blob: bytes) -> dict:
    b = np.frombuffer(blob, np.uint8)
    dt, nd = ctypes.c_int(0), ctypes.c_int(0)
    shp = np.zeros(8, np.int64)
    nbytes, nbb = ctypes.c_uint64(0), ctypes.c_uint64(0)
    nc, cb = ctypes.c_uint32(0), ctypes.c_uint32(0)
    st = lib().zco_blob_info(_ptr(b), b.size, ctypes.byref(dt), ctypes.byref(nd), _ptr(shp),
                             ctypes.byref(nbytes), ctypes.byref(nc), ctypes.byref(cb), ctypes.byref(nbb))
    if st:
        raise OracleError(st, "blob_info")
    return dict(dtype=dt.value, ndim=nd.value, shape=tuple(int(x) for x in shp[: nd.value]),
                nbytes=nbytes.value, n_chunks=nc.value, chunk_bytes=cb.value, blob_bytes=nbb.value,
                version=int(b[4]) | int(b[5]) << 8)


def decompress_status(blob: bytes, flags: int = 0) -> tuple[int, np.ndarray]:
    b = np.frombuffer(blob, np.uint8)
    try:
        info = blob_info(blob)
        n = info["nbytes"]
    except OracleError as e:
        return e.status, np.zeros(0, np.uint8)
    out = np.zeros(max(n, 1), np.uint8)
    st = lib().zco_decompress(_ptr(b), b.size, _ptr(out), n, flags)
    return int(st), out[:n]


def decompress(blob: bytes, flags: int = 0) -> np.ndarray:
    st, out = decompress_status(blob, flags)
    if st:
        raise OracleError(st, "decompress")
    return out


def verify(blob: bytes) -> int:
    """Status of checking a blob's header, table and chunk CRCs without
    decoding it (0 = intact)."""
    b = np.frombuffer(blob, np.uint8)
    if b.size == 0:
        return EFORMAT
    return int(lib().zco_verify(_ptr(b), b.size))
