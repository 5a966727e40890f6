"""GB300-native lossless compression of float model tensors.

ZipNN-style pipeline (nucleation NOTE-241: ZipNN, Method): exponent
extraction and byte grouping, per-chunk order-0 12-bit frequency tables,
32-lane interleaved rANS with raw passthrough (cuZipNN 0.1.0 API:
passthrough_threshold), a chunk-offset prefix scan and per-chunk zlib CRC-32.
Every step runs in the CUDA kernels of ``libzc.so`` (include/zc.h); this
module only marshals arguments through ctypes and uses PyTorch for device
memory and streams. There is no CPU fallback: without the library every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build
from .workloads import BF16, FP16, FP32, U8, U16, U32

__all__ = ["compress", "decompress", "crc32", "verify", "verify_into", "blob_info", "blob_size", "workspace_size",
           "compress_into", "decompress_into", "compress_delta", "decompress_delta", "compress_delta_into",
           "decompress_delta_into", "compress_batch", "compress_batch_into", "decompress_batch",
           "decompress_batch_into", "workspace_size_batch", "decompress_workspace_size_batch", "ZcError", "lib", "SHARED_TABLES", "LANE_WORDS", "OK", "EINVAL", "EFORMAT",
           "ECRC", "ECORRUPT", "ETIMEOUT", "ECAPACITY", "ECUDA", "NO_VERIFY", "PACKED"]

OK, EINVAL, EFORMAT, ECRC, ECORRUPT, ETIMEOUT, ECAPACITY, ECUDA = 0, 1, 2, 4, 8, 16, 32, 64
NO_VERIFY = 1
SHARED_TABLES = 2  # compression flag: blob format v2 (shared plane tables)
LANE_WORDS = 4     # compression flag: blob format v3 (a word list per rANS lane)
PACKED = 8         # compression and decompression flag: pack the call's chunks into few SMs (calls on several streams)
HOOK_LOOKBACK_STALL, HOOK_PRODUCER_STALL = 1, 2  # test hooks (zc_set_test_hooks)
DEFAULT_CHUNK = 131072
DEFAULT_THRESHOLD = 0.95

_TORCH_TO_CODE = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32,
                  torch.uint8: U8, torch.int8: U8, torch.bool: U8,
                  torch.int16: U16, torch.int32: U32}
for _n, _c in (("uint16", U16), ("uint32", U32)):
    if hasattr(torch, _n):
        _TORCH_TO_CODE[getattr(torch, _n)] = _c
_CODE_TO_TORCH = {BF16: torch.bfloat16, FP16: torch.float16, FP32: torch.float32,
                  U8: torch.uint8, U16: torch.int16, U32: torch.int32}
_WORD = {U8: 1, U16: 2, U32: 4, BF16: 2, FP16: 2, FP32: 4}


class ZcError(RuntimeError):
    def __init__(self, status: int, what: str):
        names = [n for n, b in (("EINVAL", EINVAL), ("EFORMAT", EFORMAT), ("ECRC", ECRC),
                                ("ECORRUPT", ECORRUPT), ("ETIMEOUT", ETIMEOUT),
                                ("ECAPACITY", ECAPACITY), ("ECUDA", ECUDA)) if status & b]
        super().__init__(f"{what}: status {status} ({'|'.join(names) or 'OK'})")
        self.status = status


class _Info(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * 8),
                ("nbytes", ctypes.c_uint64), ("blob_bytes", ctypes.c_uint64),
                ("n_chunks", ctypes.c_uint32), ("chunk_bytes", ctypes.c_uint32),
                ("version", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libzc.so (built with nvcc on first use if absent)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            vp, u64, u32, i32, dbl = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_double
            L.zc_blob_size.restype = u64
            L.zc_blob_size.argtypes = [u64, i32, u32, dbl]
            L.zc_workspace_size.restype = u64
            L.zc_workspace_size.argtypes = [u64, i32, u32]
            L.zc_blob_info.restype = i32
            L.zc_blob_info.argtypes = [vp, u64, ctypes.POINTER(_Info)]
            L.zc_compress.restype = i32
            L.zc_compress.argtypes = [vp, u64, i32, i32, ctypes.POINTER(ctypes.c_int64), u32, dbl,
                                      vp, u64, vp, vp, u64, vp, vp]
            L.zc_compress_ex.restype = i32
            L.zc_compress_ex.argtypes = [vp, u64, i32, i32, ctypes.POINTER(ctypes.c_int64), u32, dbl, u32,
                                         vp, u64, vp, vp, u64, vp, vp]
            L.zc_workspace_size_ex.restype = u64
            L.zc_workspace_size_ex.argtypes = [u64, i32, u32, u32]
            L.zc_blob_size_ex.restype = u64
            L.zc_blob_size_ex.argtypes = [u64, i32, u32, dbl, u32]
            L.zc_decompress.restype = i32
            L.zc_decompress.argtypes = [vp, ctypes.POINTER(_Info), vp, u64, u32, vp, vp]
            L.zc_compress_delta.restype = i32
            L.zc_compress_delta.argtypes = [vp, vp, u64, i32, i32, ctypes.POINTER(ctypes.c_int64), u32, dbl,
                                            vp, u64, vp, vp, u64, vp, vp]
            L.zc_decompress_delta.restype = i32
            L.zc_decompress_delta.argtypes = [vp, ctypes.POINTER(_Info), vp, vp, u64, u32, vp, vp]
            L.zc_crc32.restype = i32
            L.zc_crc32.argtypes = [vp, u64, u64, vp, vp]
            L.zc_set_test_hooks.restype = None
            L.zc_set_test_hooks.argtypes = [u32]
            L.zc_verify.restype = i32
            L.zc_verify.argtypes = [vp, ctypes.POINTER(_Info), vp, vp]
            pu64, pi64, pi32 = ctypes.POINTER(u64), ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
            L.zc_workspace_size_batch.restype = u64
            L.zc_workspace_size_batch.argtypes = [pu64, u32, i32, u32, u32]
            L.zc_decompress_workspace_size_batch.restype = u64
            L.zc_decompress_workspace_size_batch.argtypes = [u32]
            L.zc_compress_batch.restype = i32
            L.zc_compress_batch.argtypes = [u32, vp, vp, pu64, i32, pi32, pi64, u32, dbl, u32, vp, pu64, vp, vp,
                                            u64, vp, vp]
            L.zc_decompress_batch.restype = i32
            L.zc_decompress_batch.argtypes = [u32, vp, ctypes.POINTER(_Info), vp, vp, pu64, u32, vp, u64, vp, vp]
            _lib = L
    return _lib


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dtype_code(t: torch.Tensor) -> int:
    try:
        return _TORCH_TO_CODE[t.dtype]
    except KeyError:
        raise ZcError(EINVAL, f"unsupported dtype {t.dtype}") from None


def blob_size(nbytes: int, dtype: int, chunk_bytes: int = DEFAULT_CHUNK, threshold: float = DEFAULT_THRESHOLD,
              flags: int = 0) -> int:
    return int(lib().zc_blob_size_ex(nbytes, dtype, chunk_bytes, threshold, flags))


def workspace_size(nbytes: int, dtype: int, chunk_bytes: int = DEFAULT_CHUNK, flags: int = 0) -> int:
    return int(lib().zc_workspace_size_ex(nbytes, dtype, chunk_bytes, flags))


def _check(st: int, what: str):
    if st:
        raise ZcError(st, what)


def compress_into(src: torch.Tensor, blob: torch.Tensor, blob_bytes: torch.Tensor, workspace: torch.Tensor,
                  status: torch.Tensor, chunk_bytes: int = DEFAULT_CHUNK,
                  threshold: float = DEFAULT_THRESHOLD, stream=None, dtype: int | None = None,
                  shape=None, flags: int = 0) -> None:
    """Launch compression into caller buffers; no allocation, no sync.

    ``blob_bytes`` is a 1-element int64 CUDA tensor that receives the blob
    length; ``status`` a 1-element int32 CUDA tensor the caller zeroes."""
    code = dtype_code(src) if dtype is None else dtype
    shape = tuple(src.shape) if shape is None else tuple(shape)
    shp = (ctypes.c_int64 * max(1, len(shape)))(*shape)
    nbytes = src.numel() * src.element_size()
    st = lib().zc_compress_ex(src.data_ptr() if nbytes else None, nbytes, code, len(shape), shp, chunk_bytes,
                              threshold, flags, blob.data_ptr(), blob.numel(), blob_bytes.data_ptr(),
                              workspace.data_ptr(), workspace.numel(), status.data_ptr(), _stream(stream))
    _check(st, "zc_compress")


def compress(t: torch.Tensor, chunk_bytes: int = DEFAULT_CHUNK, threshold: float = DEFAULT_THRESHOLD,
             stream=None, host_blob: bool = False, shared_tables: bool = False,
             lane_words: bool = False, packed: bool = False) -> torch.Tensor:
    """Compress a CUDA tensor into a self-describing blob (1-D uint8 tensor).

    The blob is a CUDA tensor, or with ``host_blob`` a page-locked CPU tensor
    that the kernels write directly over the host link (no separate copy).
    ``shared_tables`` writes format v2 (one table per byte plane of the
    tensor), ``lane_words`` format v3 (a word list per rANS lane, which the
    decoder steps through without waiting on the other lanes). ``packed``
    (ZC_PACKED) fills few SMs, for calls on several streams at once; it
    changes no byte of the blob. Synchronises once, to read the blob
    length."""
    flags = (SHARED_TABLES if shared_tables else 0) | (LANE_WORDS if lane_words else 0) | (PACKED if packed else 0)
    if not t.is_cuda:
        raise ZcError(EINVAL, "compress expects a CUDA tensor")
    src = t.contiguous()
    code = dtype_code(src)
    nbytes = src.numel() * src.element_size()
    cap = blob_size(nbytes, code, chunk_bytes, threshold, flags)
    if cap == 0:
        raise ZcError(EINVAL, "invalid compression parameters")
    dev = src.device
    if host_blob:
        blob = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
        nb = torch.zeros(1, dtype=torch.int64, pin_memory=True)
    else:
        blob = torch.empty(cap, dtype=torch.uint8, device=dev)
        nb = torch.zeros(1, dtype=torch.int64, device=dev)
    ws = torch.empty(max(16, workspace_size(nbytes, code, chunk_bytes, flags)), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flat = src.view(-1).view(torch.uint8)
    compress_into(flat, blob, nb, ws, status, chunk_bytes, threshold, stream, dtype=code, shape=tuple(t.shape),
                  flags=flags)
    if host_blob:
        torch.cuda.synchronize(dev)  # the length is written to host memory by the kernel
    _check(int(status.item()), "zc_compress (device)")
    return blob[: int(nb.item())]


def blob_info(prefix) -> dict:
    """Header and chunk table of a blob, from host bytes (or a CPU tensor)."""
    if isinstance(prefix, torch.Tensor):
        prefix = prefix.detach().cpu().contiguous().numpy().tobytes()
    buf = ctypes.create_string_buffer(bytes(prefix), len(prefix))
    info = _Info()
    _check(lib().zc_blob_info(buf, len(prefix), ctypes.byref(info)), "zc_blob_info")
    return _info_dict(info)


def _info_dict(info: _Info) -> dict:
    return dict(dtype=info.dtype, ndim=info.ndim, shape=tuple(info.shape[: info.ndim]),
                nbytes=info.nbytes, blob_bytes=info.blob_bytes, n_chunks=info.n_chunks,
                chunk_bytes=info.chunk_bytes, version=info.version)


def _info_struct(d: dict) -> _Info:
    info = _Info()
    info.dtype, info.ndim = d["dtype"], d["ndim"]
    for i, v in enumerate(d["shape"]):
        info.shape[i] = v
    info.nbytes, info.blob_bytes = d["nbytes"], d["blob_bytes"]
    info.n_chunks, info.chunk_bytes = d["n_chunks"], d["chunk_bytes"]
    info.version = d.get("version", 1)
    return info


def read_info(blob: torch.Tensor) -> dict:
    """blob_info of a device or host blob (the header and table on the host)."""
    head = bytes(blob[:96].cpu().numpy())
    n_chunks = int.from_bytes(head[24:28], "little")
    version = head[4] | head[5] << 8
    planes = 512 * _WORD.get(head[6], 0) if version == 2 else 0  # v2: the plane tables follow the chunk table
    return blob_info(blob[: 96 + 16 * n_chunks + planes].cpu())


def decompress_into(blob: torch.Tensor, info: dict, out: torch.Tensor, status: torch.Tensor,
                    verify: bool = True, stream=None, packed: bool = False) -> None:
    """Launch decompression into a caller buffer; no allocation, no sync.
    ``packed`` (ZC_PACKED) fills few SMs, for calls on several streams."""
    flags = (0 if verify else NO_VERIFY) | (PACKED if packed else 0)
    st = lib().zc_decompress(blob.data_ptr(), ctypes.byref(_info_struct(info)), out.data_ptr(),
                             out.numel() * out.element_size(), flags, status.data_ptr(), _stream(stream))
    _check(st, "zc_decompress")


def _readable(blob: torch.Tensor) -> bool:
    return blob.is_cuda or (blob.device.type == "cpu" and blob.is_pinned())


def decompress(blob: torch.Tensor, info: dict | None = None, verify: bool = True, stream=None,
               device=None, packed: bool = False) -> torch.Tensor:
    """Restore the exact tensor (dtype and shape from the blob header). The
    blob is a CUDA tensor or a page-locked CPU tensor, which the kernel reads
    directly; the tensor is made on the blob's device (CUDA blob) or on
    ``device`` (default: the current CUDA device). ``packed`` as in
    compress()."""
    if not _readable(blob):
        raise ZcError(EINVAL, "decompress expects a CUDA or page-locked CPU blob")
    info = read_info(blob) if info is None else info
    dev = blob.device if blob.is_cuda else torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    dt = _CODE_TO_TORCH[info["dtype"]]
    out = torch.empty(info["shape"], dtype=dt, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    decompress_into(blob, info, out, status, verify, stream, packed)
    _check(int(status.item()), "zc_decompress (device)")
    return out


_WORD_CODE = {1: U8, 2: U16, 4: U32}


def compress_delta_into(base: torch.Tensor, new: torch.Tensor, blob: torch.Tensor, blob_bytes: torch.Tensor,
                        workspace: torch.Tensor, status: torch.Tensor, chunk_bytes: int = DEFAULT_CHUNK,
                        threshold: float = DEFAULT_THRESHOLD, stream=None, dtype: int | None = None,
                        shape=None) -> None:
    """Launch fused delta compression of (base XOR new) into caller buffers;
    no allocation, no sync. dtype: U8/U16/U32 (default: by element size)."""
    if base.numel() * base.element_size() != new.numel() * new.element_size():
        raise ZcError(EINVAL, "base and new differ in size")
    code = _WORD_CODE[new.element_size()] if dtype is None else dtype
    shape = tuple(new.shape) if shape is None else tuple(shape)
    shp = (ctypes.c_int64 * max(1, len(shape)))(*shape)
    nbytes = new.numel() * new.element_size()
    st = lib().zc_compress_delta(base.data_ptr() if nbytes else None, new.data_ptr() if nbytes else None, nbytes,
                                 code, len(shape), shp, chunk_bytes, threshold, blob.data_ptr(), blob.numel(),
                                 blob_bytes.data_ptr(), workspace.data_ptr(), workspace.numel(), status.data_ptr(),
                                 _stream(stream))
    _check(st, "zc_compress_delta")


def compress_delta(base: torch.Tensor, new: torch.Tensor, chunk_bytes: int = DEFAULT_CHUNK,
                   threshold: float = DEFAULT_THRESHOLD, stream=None) -> torch.Tensor:
    """Blob of the XOR difference of two same-shape CUDA tensors (a checkpoint
    against its base), formed on the fly; synchronises once for the length."""
    if not (base.is_cuda and new.is_cuda) or base.shape != new.shape or base.dtype != new.dtype:
        raise ZcError(EINVAL, "compress_delta expects two CUDA tensors of one shape and dtype")
    b, n = base.contiguous(), new.contiguous()
    code = _WORD_CODE.get(n.element_size())
    if code is None:
        raise ZcError(EINVAL, f"unsupported element size {n.element_size()}")
    nbytes = n.numel() * n.element_size()
    cap = blob_size(nbytes, code, chunk_bytes, threshold)
    if cap == 0:
        raise ZcError(EINVAL, "invalid compression parameters")
    dev = n.device
    blob = torch.empty(cap, dtype=torch.uint8, device=dev)
    ws = torch.empty(max(16, workspace_size(nbytes, code, chunk_bytes)), dtype=torch.uint8, device=dev)
    nb = torch.zeros(1, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    compress_delta_into(b.view(-1).view(torch.uint8), n.view(-1).view(torch.uint8), blob, nb, ws, status,
                        chunk_bytes, threshold, stream, dtype=code, shape=tuple(n.shape))
    _check(int(status.item()), "zc_compress_delta (device)")
    return blob[: int(nb.item())]


def decompress_delta_into(blob: torch.Tensor, info: dict, base: torch.Tensor, out: torch.Tensor,
                          status: torch.Tensor, verify: bool = True, stream=None, packed: bool = False) -> None:
    """Launch decompression of a difference blob XOR-ed with base into out."""
    st = lib().zc_decompress_delta(blob.data_ptr(), ctypes.byref(_info_struct(info)), base.data_ptr(),
                                   out.data_ptr(), out.numel() * out.element_size(),
                                   (0 if verify else NO_VERIFY) | (PACKED if packed else 0),
                                   status.data_ptr(), _stream(stream))
    _check(st, "zc_decompress_delta")


def decompress_delta(blob: torch.Tensor, base: torch.Tensor, info: dict | None = None, verify: bool = True,
                     stream=None) -> torch.Tensor:
    """The checkpoint `new` from its difference blob and the base tensor."""
    if not (blob.is_cuda and base.is_cuda):
        raise ZcError(EINVAL, "decompress_delta expects a CUDA blob and base")
    info = read_info(blob) if info is None else info
    b = base.contiguous()
    if b.numel() * b.element_size() != info["nbytes"]:
        raise ZcError(EINVAL, "base size does not match the blob")
    out = torch.empty_like(b)
    status = torch.zeros(1, dtype=torch.int32, device=blob.device)
    decompress_delta_into(blob, info, b.view(-1).view(torch.uint8), out.view(-1).view(torch.uint8), status,
                          verify, stream)
    _check(int(status.item()), "zc_decompress_delta (device)")
    return out


def set_test_hooks(hooks: int) -> None:
    """Test hooks that make a bounded device wait run out (tests only; 0 =
    none): HOOK_LOOKBACK_STALL, HOOK_PRODUCER_STALL."""
    lib().zc_set_test_hooks(hooks)


def verify_into(blob: torch.Tensor, info: dict, status: torch.Tensor, stream=None) -> None:
    """Launch the check of a blob's header CRC and chunk CRCs without
    decoding it (OR-ed into the device int32 ``status``); no sync."""
    _check(lib().zc_verify(blob.data_ptr(), ctypes.byref(_info_struct(info)), status.data_ptr(), _stream(stream)),
           "zc_verify")


def verify(blob: torch.Tensor, info: dict | None = None, stream=None) -> int:
    """Status of checking a CUDA or page-locked CPU blob without decoding it
    (cuZipNN API: verify an untrusted blob before decompressing it): 0 when
    the header CRC and every chunk CRC match, else ECRC / EFORMAT bits."""
    if not _readable(blob):
        raise ZcError(EINVAL, "verify expects a CUDA or page-locked CPU blob")
    info = read_info(blob) if info is None else info
    dev = blob.device if blob.is_cuda else torch.device("cuda", torch.cuda.current_device())
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    verify_into(blob, info, status, stream)
    return int(status.item())


def crc32(t: torch.Tensor, piece_bytes: int = 16384, stream=None) -> torch.Tensor:
    """zlib CRC-32 of every piece_bytes piece of a CUDA tensor's bytes
    (int64 CUDA tensor of values in [0, 2^32)); piece_bytes=0: one CRC."""
    if not t.is_cuda:
        raise ZcError(EINVAL, "crc32 expects a CUDA tensor")
    src = t.contiguous()
    nbytes = src.numel() * src.element_size()
    pieces = (nbytes + piece_bytes - 1) // piece_bytes if piece_bytes else 1
    out = torch.empty(max(1, pieces), dtype=torch.int32, device=src.device)
    _check(lib().zc_crc32(src.data_ptr() if nbytes else None, nbytes, piece_bytes, out.data_ptr(),
                          _stream(stream)), "zc_crc32")
    return out[:pieces].to(torch.int64) & 0xFFFFFFFF


def _ptrs(ts) -> ctypes.Array:
    return (ctypes.c_void_p * max(1, len(ts)))(*[t.data_ptr() if t.numel() else None for t in ts])


def _u64s(vals) -> ctypes.Array:
    return (ctypes.c_uint64 * max(1, len(vals)))(*vals)


def workspace_size_batch(nbytes, dtype: int, chunk_bytes: int = DEFAULT_CHUNK, flags: int = 0) -> int:
    """Workspace bytes for compress_batch_into over tensors of these sizes."""
    return int(lib().zc_workspace_size_batch(_u64s(nbytes), len(nbytes), dtype, chunk_bytes, flags))


def decompress_workspace_size_batch(n: int) -> int:
    return int(lib().zc_decompress_workspace_size_batch(n))


def compress_batch_into(srcs, blobs, blob_bytes: torch.Tensor, workspace: torch.Tensor, status: torch.Tensor,
                        dtype: int, shapes, chunk_bytes: int = DEFAULT_CHUNK, threshold: float = DEFAULT_THRESHOLD,
                        stream=None, bases=None, flags: int = 0) -> None:
    """Launch compression of n tensors (flat byte views ``srcs``) into the
    blobs ``blobs`` in one grid; ``blob_bytes`` is an n-element int64 CUDA
    tensor receiving the blob lengths. With ``bases``, tensor t is coded as
    srcs[t] XOR bases[t]. No allocation, no sync."""
    n = len(srcs)
    if len(blobs) != n or len(shapes) != n or (bases is not None and len(bases) != n) or blob_bytes.numel() < n:
        raise ZcError(EINVAL, "compress_batch_into: argument lists differ in length")
    nbytes = [t.numel() * t.element_size() for t in srcs]
    ndims = (ctypes.c_int32 * max(1, n))(*[len(sh) for sh in shapes])
    flat = []
    for sh in shapes:
        if len(sh) > 8:
            raise ZcError(EINVAL, "at most 8 dimensions")
        flat += list(sh) + [0] * (8 - len(sh))
    shp = (ctypes.c_int64 * max(8, len(flat)))(*flat)
    st = lib().zc_compress_batch(n, _ptrs(srcs), _ptrs(bases) if bases is not None else None, _u64s(nbytes), dtype,
                                 ndims, shp, chunk_bytes, threshold, flags, _ptrs(blobs),
                                 _u64s([b.numel() for b in blobs]),
                                 blob_bytes.data_ptr(), workspace.data_ptr(), workspace.numel(), status.data_ptr(),
                                 _stream(stream))
    _check(st, "zc_compress_batch")


def compress_batch(tensors, chunk_bytes: int = DEFAULT_CHUNK, threshold: float = DEFAULT_THRESHOLD, stream=None,
                   bases=None, host_blob: bool = False, shared_tables: bool = False,
                   lane_words: bool = False) -> list:
    """Compress a list of CUDA tensors of one dtype in one call; returns one
    blob per tensor, each equal to compress() of that tensor (with ``bases``:
    to compress_delta(bases[t], tensors[t])); with ``host_blob`` the blobs are
    views of one page-locked CPU buffer written by the kernels. Synchronises
    once."""
    n = len(tensors)
    if n == 0:
        return []
    if not all(t.is_cuda for t in tensors) or len({t.dtype for t in tensors}) != 1:
        raise ZcError(EINVAL, "compress_batch expects CUDA tensors of one dtype")
    ts = [t.contiguous() for t in tensors]
    if bases is not None:
        bs = [b.contiguous() for b in bases]
        if len(bs) != n or any(b.shape != t.shape or b.dtype != t.dtype or not b.is_cuda for b, t in zip(bs, ts)):
            raise ZcError(EINVAL, "compress_batch: bases must match the tensors")
        code = _WORD_CODE.get(ts[0].element_size())
        if code is None:
            raise ZcError(EINVAL, f"unsupported element size {ts[0].element_size()}")
    else:
        code = dtype_code(ts[0])
    flags = (SHARED_TABLES if shared_tables else 0) | (LANE_WORDS if lane_words else 0)
    nbytes = [t.numel() * t.element_size() for t in ts]
    caps = [blob_size(nb, code, chunk_bytes, threshold, flags) for nb in nbytes]
    if 0 in caps:
        raise ZcError(EINVAL, "invalid compression parameters")
    offs, o = [], 0
    for c in caps:
        offs.append(o)
        o += (c + 255) // 256 * 256
    dev = ts[0].device
    buf = torch.empty(o, dtype=torch.uint8, pin_memory=True) if host_blob else \
        torch.empty(o, dtype=torch.uint8, device=dev)
    blobs = [buf[a: a + c] for a, c in zip(offs, caps)]
    ws = torch.empty(max(16, workspace_size_batch(nbytes, code, chunk_bytes, flags)), dtype=torch.uint8, device=dev)
    nb = torch.zeros(n, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flat = [t.view(-1).view(torch.uint8) for t in ts]
    compress_batch_into(flat, blobs, nb, ws, status, code, [tuple(t.shape) for t in tensors], chunk_bytes,
                        threshold, stream, bases=[b.view(-1).view(torch.uint8) for b in bs] if bases is not None
                        else None, flags=flags)
    if host_blob:
        torch.cuda.synchronize(dev)
    _check(int(status.item()), "zc_compress_batch (device)")
    return [b[: int(k)] for b, k in zip(blobs, nb.tolist())]


def decompress_batch_into(blobs, infos, outs, status: torch.Tensor, workspace: torch.Tensor | None = None,
                          verify: bool = True, stream=None, bases=None) -> None:
    """Launch decompression of n blobs (one dtype and chunk size) into
    ``outs`` in one grid; with ``bases``, output t is the decoded bytes XOR
    bases[t]. ``workspace`` holds decompress_workspace_size_batch(n) bytes
    (None when n <= 1). No allocation, no sync."""
    n = len(blobs)
    if len(infos) != n or len(outs) != n or (bases is not None and len(bases) != n):
        raise ZcError(EINVAL, "decompress_batch_into: argument lists differ in length")
    arr = (_Info * max(1, n))(*[_info_struct(d) for d in infos])
    caps = _u64s([t.numel() * t.element_size() for t in outs])
    st = lib().zc_decompress_batch(n, _ptrs(blobs), arr, _ptrs(bases) if bases is not None else None, _ptrs(outs),
                                   caps, 0 if verify else NO_VERIFY,
                                   workspace.data_ptr() if workspace is not None else None,
                                   workspace.numel() if workspace is not None else 0, status.data_ptr(),
                                   _stream(stream))
    _check(st, "zc_decompress_batch")


def decompress_batch(blobs, infos=None, verify: bool = True, stream=None, bases=None) -> list:
    """Restore a list of tensors from their blobs in one call (each equal to
    decompress(), or with ``bases`` to decompress_delta(), of its blob)."""
    n = len(blobs)
    if n == 0:
        return []
    if not all(_readable(b) for b in blobs):
        raise ZcError(EINVAL, "decompress_batch expects CUDA or page-locked CPU blobs")
    infos = [read_info(b) for b in blobs] if infos is None else list(infos)
    dev = blobs[0].device if blobs[0].is_cuda else torch.device("cuda", torch.cuda.current_device())
    if bases is not None:
        outs = [torch.empty_like(b.contiguous()) for b in bases]
        bflat = [b.contiguous().view(-1).view(torch.uint8) for b in bases]
    else:
        outs = [torch.empty(d["shape"], dtype=_CODE_TO_TORCH[d["dtype"]], device=dev) for d in infos]
        bflat = None
    ws_n = decompress_workspace_size_batch(n)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev) if ws_n else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    decompress_batch_into(blobs, infos, [o.view(-1).view(torch.uint8) for o in outs], status, ws, verify, stream,
                          bases=bflat)
    _check(int(status.item()), "zc_decompress_batch (device)")
    return outs
