"""Every tensor of the Llama-3.1-8B-shaped BF16 model (290 tensors, 16.06
GB; lmzip README "What it saves": the Llama-3.1-8B safetensors shards;
ZipNN note, Table II) compressed on the GPU one call per tensor, each blob
compared byte for byte with the oracle's blob of the same tensor, and each
blob decoded on the GPU back to the exact tensor.

The oracle is single-threaded, so the comparisons run in a process pool over
the host's cores (started with spawn); a worker returns the length and the
SHA-256 of its blob, compared with the GPU blob's. The two 1 GB tensors
(embedding, LM head) go first so that they do not become the tail.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import multiprocessing as mp
import os

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import entropy_coding_gb300 as zc  # noqa: E402
from entropy_coding_gb300 import workloads as wl  # noqa: E402

DEV = torch.device("cuda:0")


def test_llama8b_every_tensor_matches_oracle(zco):
    from oracle.parallel import blob_digest

    specs = wl.llama8b_specs()
    order = [0, len(specs) - 1] + list(range(1, len(specs) - 1))
    cores = max(1, len(os.sched_getaffinity(0)))
    pending: dict = {}
    checked = total_bytes = total_blob = 0

    def settle(block: bool):
        nonlocal checked
        done = [f for f in pending if f.done()]
        if block and not done:
            done = list(cf.wait(pending, return_when=cf.FIRST_COMPLETED).done)
        for f in done:
            name, want = pending.pop(f)
            assert f.result() == want, f"{name}: GPU blob differs from the oracle's"
            checked += 1

    with cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
        for idx in order:
            name, shape = specs[idx]
            t = wl.llama8b_tensor(idx, name, shape, DEV)
            blob = zc.compress(t)
            back = zc.decompress(blob)
            assert torch.equal(back.view(torch.int16), t.view(torch.int16)), name
            gpu = blob.cpu().numpy().tobytes()
            raw = wl.as_bytes(t).cpu().numpy()
            total_bytes += raw.size
            total_blob += len(gpu)
            want = (len(gpu), hashlib.sha256(gpu).hexdigest())
            del t, blob, back, gpu
            pending[ex.submit(blob_digest, raw, wl.BF16, shape, 131072, 0.95, 1)] = (name, want)
            while len(pending) > 2 * cores:
                settle(block=True)
        while pending:
            settle(block=True)
    assert checked == len(specs) == 290
    assert total_bytes == 16_060_514_304
    assert 0.65 < total_blob / total_bytes < 0.67
