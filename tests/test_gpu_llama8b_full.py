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


@pytest.mark.parametrize("version,streams", [(1, 1), (3, 8)])
def test_llama8b_every_tensor_matches_oracle(zco, version, streams):
    """Format v1 one call after another, and format v3 (a word list per lane)
    with the calls issued round-robin on 8 streams, each with its own
    workspace and packed into few SMs (ZC_PACKED): the launch configuration
    the benchmark times."""
    from oracle.parallel import blob_digest

    flags = {1: 0, 3: zc.LANE_WORDS}[version]
    packed = streams > 1
    C, thr = 131072, 0.95
    specs = wl.llama8b_specs()
    order = [0, len(specs) - 1] + list(range(1, len(specs) - 1))
    cores = max(1, len(os.sched_getaffinity(0)))
    workers = [torch.cuda.Stream(device=DEV) for _ in range(streams)]
    ws_bytes = max(zc.workspace_size(2 * torch.Size(sh).numel(), wl.BF16, C, flags) for _, sh in specs)
    ws = [torch.empty(ws_bytes, dtype=torch.uint8, device=DEV) for _ in range(streams)]
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
        for i0 in range(0, len(order), streams):
            group = []
            for k, idx in enumerate(order[i0:i0 + streams]):
                name, shape = specs[idx]
                src = wl.as_bytes(wl.llama8b_tensor(idx, name, shape, DEV))
                blob = torch.empty(zc.blob_size(src.numel(), wl.BF16, C, thr, flags), dtype=torch.uint8, device=DEV)
                nb = torch.zeros(1, dtype=torch.int64, device=DEV)
                st = torch.zeros(1, dtype=torch.int32, device=DEV)
                workers[k].wait_stream(torch.cuda.current_stream())  # the inputs were made there
                zc.compress_into(src, blob, nb, ws[k], st, C, thr, workers[k], dtype=wl.BF16, shape=tuple(shape),
                                 flags=flags | (zc.PACKED if packed else 0))
                group.append((k, name, shape, src, blob, nb, st))
            torch.cuda.synchronize()
            outs = []
            for k, name, shape, src, blob, nb, st in group:
                assert int(st.item()) == 0, name
                b = blob[: int(nb.item())]
                out = torch.empty_like(src)
                zc.decompress_into(b, zc.read_info(b), out, st, True, workers[k], packed=packed)
                outs.append((name, shape, src, b, out, st))
            torch.cuda.synchronize()
            for name, shape, src, b, out, st in outs:
                assert int(st.item()) == 0 and torch.equal(out, src), name
                gpu = b.cpu().numpy().tobytes()
                raw = src.cpu().numpy()
                total_bytes += raw.size
                total_blob += len(gpu)
                want = (len(gpu), hashlib.sha256(gpu).hexdigest())
                pending[ex.submit(blob_digest, raw, wl.BF16, shape, C, thr, version)] = (name, want)
            del group, outs
            while len(pending) > 2 * cores:
                settle(block=True)
        while pending:
            settle(block=True)
    assert checked == len(specs) == 290
    assert total_bytes == 16_060_514_304
    assert 0.65 < total_blob / total_bytes < 0.67
