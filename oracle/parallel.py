"""Process-pool helpers for checking large workloads against the oracle —
TEST INFRASTRUCTURE ONLY (used by the test suite).

Workers are started with the ``spawn`` method by the caller; each one loads
the oracle library and returns only a digest of the blob it made, so that a
large tensor's blob never travels back through a pipe.
"""
from __future__ import annotations

import hashlib


def blob_digest(raw, dtype: int, shape, chunk_bytes: int, threshold: float, version: int = 1):
    """(length, sha256 hex) of the oracle's blob of ``raw`` (uint8 array)."""
    import oracle
    blob = oracle.compress(raw, dtype, tuple(shape), chunk_bytes, threshold, version=version)
    return len(blob), hashlib.sha256(blob).hexdigest()
