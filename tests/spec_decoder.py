"""An independent, pure-Python reader of the blob format, for tests.

Written from the format description (header, chunk table, grouped-chunk
directory, rANS record), not from the oracle's code, and sharing nothing with
either implementation. It decodes small blobs (tens of KiB) only, in
format v1 (a table in every record), v2 (one table per plane after the
chunk table, records of states and words) or v3 (v1 with a word list per
lane in every record). A blob that
this reader and the oracle both turn back into the input is a valid encoding
of the documented format, which pins the oracle's layout choices from the
outside.

Bit-level conventions it reads (ZipNN note, Method 1-2 readings): for the
float dtypes the permuted word holds exponent | sign | mantissa from the top;
stream j is byte j counted from the most significant byte.
"""
from __future__ import annotations

import struct
import zlib

WORD = {1: 1, 2: 2, 3: 4, 4: 2, 5: 2, 6: 4}
EXP = {4: 8, 5: 5, 6: 8}


class SpecError(ValueError):
    pass


def _unpermute(p: int, dtype: int) -> int:
    E = EXP.get(dtype)
    if E is None:
        return p
    B = 8 * WORD[dtype]
    e = p >> (B - E)
    s = (p >> (B - E - 1)) & 1
    m = p & ((1 << (B - 1 - E)) - 1)
    return (s << (B - 1)) | (e << (B - 1 - E)) | m


def _lane_lists(rec: bytes, at: int) -> list[list[int]]:
    """v3: 32 u16 counts at `at`, then each lane's words (padded to 8)."""
    counts = struct.unpack_from("<32H", rec, at)
    lists, pos = [], at + 64
    for c in counts:
        lists.append(list(struct.unpack_from(f"<{c}H", rec, pos)))
        if any(struct.unpack_from(f"<{-c % 8}H", rec, pos + 2 * c)):
            raise SpecError("nonzero list padding")
        pos += 2 * (c + -c % 8)
    if pos != len(rec):
        raise SpecError("lane lists do not fill the record")
    return lists


def _rans(rec: bytes, n: int, plane=None, lanes: bool = False, owners: list | None = None) -> list[int]:
    """Decode a record: v1 carries its table (bitmap + frequencies) and one
    word list; a v2 record is states + words and uses its plane's table (256
    frequencies); a v3 record (lanes) is v1's head, then a word list per lane.
    With `owners` (v1), the lane that takes each word is appended to it in
    the order the words are taken."""
    states = list(struct.unpack_from("<32I", rec, 0))
    if plane is None:
        bitmap = rec[128:160]
        present = [s for s in range(256) if bitmap[s // 8] >> (s % 8) & 1]
        k = len(present)
        freqs = struct.unpack_from(f"<{k}H", rec, 160)
        words_at = 160 + (2 * k + 15) // 16 * 16
    else:
        present = [s for s in range(256) if plane[s]]
        freqs = [plane[s] for s in present]
        words_at = 128
    lists = _lane_lists(rec, words_at) if lanes else None
    words = [] if lanes else struct.unpack_from(f"<{(len(rec) - words_at) // 2}H", rec, words_at)
    # slot -> symbol map, built by laying the symbols' slot ranges end to end
    slot_sym, start = [], {}
    for s, f in zip(present, freqs):
        start[s] = len(slot_sym)
        slot_sym += [s] * f
    if len(slot_sym) != 4096:
        raise SpecError("frequencies do not sum to 4096")
    freq = dict(zip(present, freqs))
    out = [0] * n
    nxt = len(words)  # the words are consumed from the last one backwards
    for i in range(n):
        lane = i % 32
        x = states[lane]
        slot = x % 4096
        s = slot_sym[slot]
        x = freq[s] * (x // 4096) + slot - start[s]
        if x < 65536:
            if lanes:  # the lane's own list, from its end backwards
                if not lists[lane]:
                    raise SpecError("ran out of words")
                x = x * 65536 + lists[lane].pop()
            else:
                nxt -= 1
                if nxt < 0:
                    raise SpecError("ran out of words")
                x = x * 65536 + words[nxt]
                if owners is not None:
                    owners.append(lane)
        states[lane] = x
        out[i] = s
    if nxt != 0 or any(x != 65536 for x in states) or (lanes and any(lists)):
        raise SpecError("bad final state")
    return out


def decode(blob: bytes) -> bytes:
    version, = struct.unpack_from("<H", blob, 4)
    if blob[:4] != b"ZCNN" or version not in (1, 2, 3):
        raise SpecError("magic/version")
    dtype, ndim = blob[6], blob[7]
    chunk_bytes, = struct.unpack_from("<I", blob, 8)
    nbytes, = struct.unpack_from("<Q", blob, 16)
    n_chunks, hcrc = struct.unpack_from("<II", blob, 24)
    table_end = 96 + 16 * n_chunks
    planes = None
    if version == 2:  # W plane tables of 256 u16 follow the chunk table
        W = WORD[dtype]
        planes = [struct.unpack_from("<256H", blob, table_end + 512 * j) for j in range(W)]
        table_end += 512 * W
    head = bytearray(blob[:table_end])
    head[28:32] = b"\0\0\0\0"
    if zlib.crc32(bytes(head)) != hcrc:
        raise SpecError("header crc")
    out = bytearray()
    for c in range(n_chunks):
        off, sm, crc = struct.unpack_from("<QII", blob, 96 + 16 * c)
        stored, raw = sm & 0x7FFFFFFF, sm >> 31
        payload = blob[off:off + stored]
        if zlib.crc32(bytes(payload)) != crc:   # CRC of the stored bytes, checked first
            raise SpecError(f"chunk {c} crc")
        length = min(chunk_bytes, nbytes - c * chunk_bytes)
        if raw:
            out += payload
        else:
            out += _grouped(payload, length, dtype, planes, lanes=version == 3)
    return bytes(out)


def _grouped(payload: bytes, length: int, dtype: int, planes=None, lanes: bool = False) -> bytes:
    W = WORD[dtype]
    n = length // W
    pos = (4 * W + 15) // 16 * 16
    streams = []
    for j in range(W):
        entry, = struct.unpack_from("<I", payload, 4 * j)
        mode, v = entry >> 30, entry & 0x3FFFFFFF
        if mode == 2:
            streams.append([v] * n)
            continue
        rec = payload[pos:pos + v]
        streams.append(list(rec) if mode == 0 else _rans(rec, n, None if planes is None else planes[j], lanes))
        pos += (v + 15) // 16 * 16
    out = bytearray()
    for i in range(n):
        p = 0
        for j in range(W):
            p = (p << 8) | streams[j][i]
        out += _unpermute(p, dtype).to_bytes(W, "little")
    return bytes(out)
