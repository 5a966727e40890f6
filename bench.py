#!/usr/bin/env python
"""Benchmark: encode and decode throughput (GB/s of original bytes) of the
compressor on one GB300, with the HBM roofline fraction and the size ratio.

A step is one pass of the whole hot path over the workload: compression
(byte grouping, per-chunk tables, rANS with passthrough, offset scan, CRC-32)
and decompression of the blobs it made (rANS decode, merge, CRC check). The
default workload is the Llama-3.1-8B-shaped BF16 model (290 tensors, 16.06
GB), compressed and decompressed tensor by tensor from device memory; the
same model in one batched call each way is reported beside it. Inputs are
device-resident when the timed region starts; inputs smaller than 256 MiB get
the L2 flushed before every timed call. `value` = original bytes of all ranks
/ (encode + decode time); encode and decode are also reported on their own.

`--impl reference` times the CPU oracle (plain C, one thread) on a bounded
sample of the same workload, as the reference arm.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one independent replica per GPU (the path shards by
tensor and needs no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e specification


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="llama8b",
                   choices=["fp32_64m", "bf16_1m", "fp32clean_64m", "fp16_16m", "bf16_delta", "bf16_delta_fused",
                            "bf16_llama_gate", "llama8b", "llama8b_batch"])
    p.add_argument("--chunk-bytes", type=int, default=131072)
    p.add_argument("--threshold", type=float, default=0.95)
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--no-verify", action="store_true", help="decode without the CRC check")
    p.add_argument("--shared-tables", action="store_true",
                   help="blob format v2: one table per byte plane of each tensor (ZC_SHARED_TABLES)")
    p.add_argument("--streams", type=int, default=8,
                   help="llama8b: the per-tensor calls are issued round-robin on this many CUDA streams, each "
                        "with its own workspace, and packed into few SMs (ZC_PACKED) when there are several "
                        "(1: one stream, every call after the previous one)")
    p.add_argument("--packed", action="store_true",
                   help="single-tensor workloads: pack each call into few SMs (ZC_PACKED), the launch shape the "
                        "model's calls on several streams use")
    p.add_argument("--format", type=int, default=None, choices=[1, 2, 3],
                   help="blob format: 1 (a table and one word list per coded stream), 2 (shared plane "
                        "tables, as --shared-tables), 3 (a word list per rANS lane, ZC_LANE_WORDS; the "
                        "default)")
    return p.parse_args()


FORMAT_NAMES = {1: "v1 (a table and one word list per coded stream)", 2: "v2 (shared plane tables)",
                3: "v3 (v1 with a word list per rANS lane)"}


def format_version(a) -> int:
    if a.format is not None:
        return a.format
    return 2 if a.shared_tables else 3


def format_flags(a, zc) -> int:
    return {1: 0, 2: zc.SHARED_TABLES, 3: zc.LANE_WORDS}[format_version(a)]


def make_workload(name: str, device):
    from entropy_coding_gb300 import workloads as wl
    if name == "fp32_64m":
        return wl.fp32_64m(device), "FP32 8192x8192 N(0,0.02) seed 1"
    if name == "bf16_1m":
        return wl.bf16_1m(device), "BF16 1024x1024 N(0,0.02) seed 0"
    if name == "fp32clean_64m":
        return wl.fp32clean_64m(device), "clean FP32 8192x8192 (BF16-rounded) seed 2"
    if name == "fp16_16m":
        return wl.fp16_16m(device), "FP16 4096x4096 N(0,0.05) seed 3"
    if name == "bf16_delta":
        return wl.bf16_delta(device)[1], "U16 XOR of two BF16 4096x14336 checkpoints, seed 4"
    if name == "bf16_delta_fused":
        # the coded bytes are the XOR difference (what the oracle codes); the
        # GPU arm forms it inside the kernels from the two checkpoints
        return (wl.bf16_delta(device)[1], "two BF16 4096x14336 checkpoints, seed 4, XOR difference formed in "
                                          "the kernels (compress_delta / decompress_delta)")
    if name in MODEL_WORKLOADS:
        # the reference arm samples the model from its start (the embedding)
        nm, shape = wl.llama8b_specs()[0]
        return wl.llama8b_tensor(0, nm, shape, device), MODEL_WORKLOADS[name]
    if name == "bf16_llama_gate":
        specs = wl.llama8b_specs()
        nm, shape = specs[5]
        return wl.llama8b_tensor(5, nm, shape, device), "Llama-3.1-8B layer-0 gate_proj BF16 14336x4096"
    raise ValueError(name)


MODEL_WORKLOADS = {
    "llama8b": "Llama-3.1-8B-shaped BF16 model (290 tensors, 16.06 GB), N(0,0.02) per tensor, RMSNorm vectors of "
               "ones; one compression and one decompression call per tensor (issued round-robin on the "
               "configured number of CUDA streams)",
    "llama8b_batch": "Llama-3.1-8B-shaped BF16 model (290 tensors, 16.06 GB), N(0,0.02) per tensor, RMSNorm "
                     "vectors of ones; all tensors in one batched compression and one batched decompression call",
}


def encode_launches(tensor_chunks, word: int, chunk_bytes: int, v2: bool = False) -> int:
    """Kernels one compression call over tensors of these chunk counts
    launches, as the library plans it with a full-size workspace: a wave
    holds at most 2 GiB of per-chunk statistics (32 + W (512 + n_pad) bytes a
    chunk; v2: at least the largest tensor, and only whole tensors); each wave
    is a statistics and a coding kernel (v2: and a plane-table kernel); the
    empty tensors' blobs take one more kernel."""
    nc = sum(tensor_chunks)
    empty = 1 if 0 in tensor_chunks else 0
    if nc == 0:
        return empty
    n_pad = (chunk_bytes // word + 31) // 32 * 32
    wave = min(nc, (2048 << 20) // (32 + word * (512 + n_pad)))
    if not v2:
        return empty + 2 * ((nc + wave - 1) // wave)
    wave = max(wave, max(tensor_chunks))
    waves, t, n = 0, 0, len(tensor_chunks)
    while t < n:
        t0, chunks = t, 0
        while t < n and (t == t0 or chunks + tensor_chunks[t] <= wave):
            chunks += tensor_chunks[t]
            t += 1
        waves += 1 if chunks else 0
    return empty + 3 * waves


def max_over_ranks(vals, device) -> list:
    """Per-rank timings reduced to their maximum over all ranks (replicas:
    the job takes as long as its slowest rank), followed by a barrier; the
    values unchanged with one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(vals)
    t = torch.tensor(list(vals), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return t.tolist()


def replica_value(units_per_rank: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job throughput of independent replicas: the units every rank
    processed over the slowest rank's time."""
    return world * units_per_rank * steps / seconds


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if k in d:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "entropy_coding_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as fh:
                h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, version: int, packed: bool):
    """DRAM bytes of the timed unit (one call; for the model, one phase) from
    the committed ncu summaries of this kernel, workload, blob format and
    launch shape, if they were taken from the current kernel sources. For
    code_kernel the unit is the compression call (stats_kernel too)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            d = json.load(fh)
        e = d[f"{kernel}:{workload}:v{version}" + (":packed" if packed else "")]
        if e.get("source_hash") == kernel_source_hash():
            return int(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clock and throttle sampling during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--id={self.index}",
               "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[0]) for r in self.rows if r and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) > 1 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 3 + i and r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(self.rows)}


def _oracle_round_trip(job):
    """One pool worker's share of a reference step: the oracle, as it stands,
    compresses and decompresses its sample; returns the bytes and whether the
    round trip was exact."""
    raw, code, chunk_bytes, threshold, version = job
    import oracle
    blob = oracle.compress(raw, code, None, chunk_bytes, threshold, version)
    return raw.size, oracle.decompress(blob).tobytes() == raw.tobytes()


def run_reference_model(a):
    """The oracle over the Llama-shaped model through a process pool on every
    host core (the workload is 290 independent tensors): each step, every
    worker compresses and decompresses a 2 MiB slice of a different layer
    tensor (bounded so the run takes minutes, not the 16 GB)."""
    import multiprocessing as mp
    import oracle
    from entropy_coding_gb300 import workloads as wl
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    specs = wl.llama8b_specs()
    jobs = []
    for i in range(1, 1 + cores):  # layer 0, 1, ... tensors after the embedding
        nm, shape = specs[i]
        raw = wl.as_bytes(wl.llama8b_tensor(i, nm, shape)).numpy()
        jobs.append((raw[: 16 * a.chunk_bytes].copy(), wl.BF16, a.chunk_bytes, a.threshold, format_version(a)))
    sample = sum(j[0].size for j in jobs)
    with mp.get_context("spawn").Pool(cores) as pool:
        for _ in range(max(1, a.warmup)):
            pool.map(_oracle_round_trip, jobs)
        t = 0.0
        for _ in range(a.steps):
            t0 = time.perf_counter()
            res = pool.map(_oracle_round_trip, jobs)
            t += time.perf_counter() - t0
            assert all(ok for _, ok in res)
    value = sample * a.steps / t / 1e9
    desc = MODEL_WORKLOADS[a.workload]
    line = {"metric": "round-trip GB/s (original bytes; encode + decode)", "value": round(value, 4),
            "unit": "GB/s", "impl": "reference", "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": round(1e3 * t / a.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": a.workload, "desc": desc, "chunk_bytes": a.chunk_bytes,
                       "threshold": a.threshold},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{len(jobs)} slices of 2 MiB (16 chunks) from the first {len(jobs)} "
                                       f"layer tensors per step, one per process, {cores} processes "
                                       f"(os.sched_getaffinity), single-threaded C oracle in each"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(a):
    """The CPU oracle on a bounded sample of the workload (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if a.workload in MODEL_WORKLOADS:
        run_reference_model(a)
        return
    import numpy as np
    import torch
    import oracle
    from entropy_coding_gb300 import workloads as wl
    oracle.build()
    t, desc = make_workload(a.workload, "cpu")
    raw = wl.as_bytes(t).numpy()
    code = wl.dtype_code(t)
    W = raw.size // max(1, t.numel())
    sample = min(raw.size, 16 * a.chunk_bytes)     # 2 MiB per step: a few seconds of CPU work
    part = raw[:sample]
    blob = oracle.compress(part, code, (sample // W,), a.chunk_bytes, a.threshold, format_version(a))  # warm-up
    oracle.decompress(blob)
    t_enc = t_dec = 0.0
    size = 0
    for _ in range(a.steps):
        t0 = time.perf_counter()
        blob = oracle.compress(part, code, (sample // W,), a.chunk_bytes, a.threshold, format_version(a))
        t1 = time.perf_counter()
        out = oracle.decompress(blob)
        t2 = time.perf_counter()
        t_enc += t1 - t0
        t_dec += t2 - t1
        size = len(blob)
    assert out.tobytes() == part.tobytes()
    n = sample * a.steps
    value = n / (t_enc + t_dec) / 1e9
    line = {"metric": "round-trip GB/s (original bytes; encode + decode)", "value": round(value, 4),
            "unit": "GB/s", "impl": "reference", "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": round(1e3 * (t_enc + t_dec) / a.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": a.workload, "desc": desc, "chunk_bytes": a.chunk_bytes,
                       "threshold": a.threshold},
            "encode_gbs": round(n / t_enc / 1e9, 4), "decode_gbs": round(n / t_dec / 1e9, 4),
            "size_pct": round(100.0 * size / sample, 3),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"first {sample} bytes ({sample // a.chunk_bytes} chunks) of the "
                                       f"workload per step, single-threaded C oracle"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(t, code, a):
    """Single-thread oracle on a bounded sample (about ten seconds)."""
    import oracle
    from entropy_coding_gb300 import workloads as wl
    oracle.build()
    raw = wl.as_bytes(t.cpu()).numpy()
    W = raw.size // max(1, t.numel())
    budget, done, t_total, chunks = 8.0, 0, 0.0, 0
    step = min(raw.size, 8 * a.chunk_bytes)
    while t_total < budget and done < raw.size:
        part = raw[done:done + step]
        t0 = time.perf_counter()
        blob = oracle.compress(part, code, (part.size // W,), a.chunk_bytes, a.threshold, format_version(a))
        out = oracle.decompress(blob)
        t_total += time.perf_counter() - t0
        assert out.tobytes() == part.tobytes()
        done += part.size
        chunks += (part.size + a.chunk_bytes - 1) // a.chunk_bytes
    return {"value": round(done / t_total / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} bytes ({chunks} chunks) from the start of the workload, compressed and "
                      f"decompressed once, single-threaded C oracle, {t_total:.1f} s"}


def run_model(a, world, rank, local, dev, stream):
    """The Llama-shaped model: every tensor compressed and decompressed, by one
    call per tensor (llama8b) or one batched call each way (llama8b_batch)."""
    import torch
    import torch.distributed as dist
    import entropy_coding_gb300 as zc
    from entropy_coding_gb300 import workloads as wl

    batched = a.workload == "llama8b_batch"
    also_batched = not batched  # the per-tensor line also reports the batched calls
    flags = format_flags(a, zc)
    specs = wl.llama8b_specs()
    C, thr, code, Wd = a.chunk_bytes, a.threshold, wl.BF16, 2
    sizes = [2 * int(torch.Size(sh).numel()) for _, sh in specs]
    n = len(specs)

    def layout(lens):
        offs, o = [], 0
        for x in lens:
            offs.append(o)
            o += (x + 255) // 256 * 256
        return offs, o

    s_offs, s_total = layout(sizes)
    src_all = torch.empty(s_total, dtype=torch.uint8, device=dev)
    srcs = [src_all[o: o + x] for o, x in zip(s_offs, sizes)]
    for i, ((nm, sh), d) in enumerate(zip(specs, srcs)):
        d.copy_(wl.as_bytes(wl.llama8b_tensor(i, nm, sh, dev)))
    out_all = torch.empty(s_total, dtype=torch.uint8, device=dev)
    outs = [out_all[o: o + x] for o, x in zip(s_offs, sizes)]
    caps = [zc.blob_size(x, code, C, thr, flags) for x in sizes]
    b_offs, b_total = layout(caps)
    blob_all = torch.empty(b_total, dtype=torch.uint8, device=dev)
    blobs = [blob_all[o: o + x] for o, x in zip(b_offs, caps)]
    shapes = [tuple(sh) for _, sh in specs]
    nb = torch.zeros(n, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_b = dws = ws_1 = None
    if batched or also_batched:
        ws_b = torch.empty(zc.workspace_size_batch(sizes, code, C, flags), dtype=torch.uint8, device=dev)
        n_dws = zc.decompress_workspace_size_batch(n)
        dws = torch.empty(max(16, n_dws), dtype=torch.uint8, device=dev)
    # per-tensor calls: round-robin on n_streams streams, each with its own
    # workspace; the calls of one step start after an event on `stream` and
    # `stream` waits for all of them at the end of the step
    n_streams = 1 if batched else max(1, a.streams)
    workers = [stream] if n_streams == 1 else [torch.cuda.Stream(device=dev) for _ in range(n_streams)]
    ws_1 = []
    if not batched:
        ws_bytes_1 = max(zc.workspace_size(x, code, C, flags) for x in sizes)
        ws_1 = [torch.empty(ws_bytes_1, dtype=torch.uint8, device=dev) for _ in range(n_streams)]
    N = sum(sizes)
    verify = not a.no_verify

    def fan_out():
        if n_streams > 1:
            ev = torch.cuda.Event()
            ev.record(stream)
            for w in workers:
                w.wait_event(ev)

    def fan_in():
        if n_streams > 1:
            for w in workers:
                ev = torch.cuda.Event()
                ev.record(w)
                stream.wait_event(ev)

    # calls on several streams pack their chunks into few SMs (ZC_PACKED), so
    # that the calls in flight share the GPU instead of each spreading over it
    packed = n_streams > 1

    def comp(inputs, blobs=blobs, nb=nb, one_call=batched):
        if one_call:
            zc.compress_batch_into(inputs, blobs, nb, ws_b, st, code, shapes, C, thr, stream, flags=flags)
        else:
            fan_out()
            for t in range(n):
                k = t % n_streams
                zc.compress_into(inputs[t], blobs[t], nb[t:t + 1], ws_1[k], st, C, thr, workers[k], dtype=code,
                                 shape=shapes[t], flags=flags | (zc.PACKED if packed else 0))
            fan_in()

    def decomp(infos, blobs=blobs, one_call=batched):
        if one_call:
            zc.decompress_batch_into(blobs, infos, outs, st, dws, verify, stream)
        else:
            fan_out()
            for t in range(n):
                zc.decompress_into(blobs[t], infos[t], outs[t], st, verify, workers[t % n_streams], packed=packed)
            fan_in()

    with torch.cuda.stream(stream):
        comp(srcs)
    stream.synchronize()
    assert int(st.item()) == 0
    lens = nb.tolist()
    S = sum(lens)
    planes = 512 * Wd if flags & zc.SHARED_TABLES else 0  # v2: the plane tables follow the chunk table
    infos = [zc.blob_info(b[: 96 + 16 * ((x + C - 1) // C) + planes].cpu()) for b, x in zip(blobs, sizes)]
    with torch.cuda.stream(stream):
        decomp(infos)
    stream.synchronize()
    assert int(st.item()) == 0 and torch.equal(out_all, src_all), "round trip failed"

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            comp(srcs)
            decomp(infos)
    stream.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for ev in evs:
                ev[0].record(stream)
                comp(srcs)
                ev[1].record(stream)
                decomp(infos)
                ev[2].record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    t_enc = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    t_dec = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    assert int(st.item()) == 0 and nb.tolist() == lens
    total = t_enc + t_dec
    total, t_enc, t_dec = max_over_ranks([total, t_enc, t_dec], dev)

    # the same model in one batched call each way, beside the per-tensor line
    batched_line = None
    if also_batched:
        with torch.cuda.stream(stream):
            for _ in range(max(1, a.warmup)):
                comp(srcs, one_call=True)
                decomp(infos, one_call=True)
        stream.synchronize()
        assert int(st.item()) == 0 and nb.tolist() == lens and torch.equal(out_all, src_all)
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
        with torch.cuda.stream(stream):
            for ev in bev:
                ev[0].record(stream)
                comp(srcs, one_call=True)
                ev[1].record(stream)
                decomp(infos, one_call=True)
                ev[2].record(stream)
        stream.synchronize()
        bt_enc = sum(e[0].elapsed_time(e[1]) for e in bev) / 1e3
        bt_dec = sum(e[1].elapsed_time(e[2]) for e in bev) / 1e3
        assert int(st.item()) == 0 and nb.tolist() == lens
        bt_enc, bt_dec = max_over_ranks([bt_enc, bt_dec], dev)
        batched_line = (bt_enc, bt_dec)

    # end to end through the public calls: the model from pinned host memory,
    # the blobs back to the host and up again, the restored model to the host
    e2e_steps = max(1, min(a.e2e_steps, 2))
    h_src = torch.empty(s_total, dtype=torch.uint8, pin_memory=True)
    h_src.copy_(src_all)
    h_blob = torch.empty(b_total, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(s_total, dtype=torch.uint8, pin_memory=True)
    h2d = d2h = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            src_all.copy_(h_src, non_blocking=True)
            comp(srcs)
            got = nb.tolist()
            for o, k in zip(b_offs, got):
                h_blob[o: o + k].copy_(blob_all[o: o + k], non_blocking=True)
            for o, k in zip(b_offs, got):
                blob_all[o: o + k].copy_(h_blob[o: o + k], non_blocking=True)
            decomp(infos)
            h_out.copy_(out_all, non_blocking=True)
        stream.synchronize()
        h2d += s_total + sum(got)
        d2h += sum(got) + 8 * n + s_total
    t_e2e = time.perf_counter() - t0
    assert int(st.item()) == 0 and torch.equal(h_out, h_src)

    # end to end with the blobs in page-locked host memory, written and read
    # by the kernels; the host parses every header and table between the calls
    del h_blob
    hb_all = torch.empty(b_total, dtype=torch.uint8, pin_memory=True)
    hb_blobs = [hb_all[o: o + x] for o, x in zip(b_offs, caps)]
    hb_nb = torch.zeros(n, dtype=torch.int64, pin_memory=True)
    h_out.zero_()
    hb_h2d = hb_d2h = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            src_all.copy_(h_src, non_blocking=True)
            comp(srcs, hb_blobs, hb_nb)
        stream.synchronize()
        got = hb_nb.tolist()
        hb_infos = [zc.blob_info(b[: 96 + 16 * ((x + C - 1) // C) + planes]) for b, x in zip(hb_blobs, sizes)]
        with torch.cuda.stream(stream):
            decomp(hb_infos, [b[:k] for b, k in zip(hb_blobs, got)])
            h_out.copy_(out_all, non_blocking=True)
        stream.synchronize()
        hb_h2d += s_total + sum(got)
        hb_d2h += sum(got) + 8 * n + s_total
    t_hb = time.perf_counter() - t0
    assert int(st.item()) == 0 and torch.equal(h_out, h_src)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    hbm, peak_kind = peaks()
    alg = N + S
    enc_ach = alg * a.steps / t_enc / 1e9
    dec_ach = alg * a.steps / t_dec / 1e9
    chunks = [(x + C - 1) // C for x in sizes]
    dec_kernel = "decode_v2_kernel" if flags & zc.SHARED_TABLES else "decode_kernel"
    # the roofline of the phase that takes longer: compression (stats_kernel
    # then code_kernel per call; code_kernel is most of its kernel time) or
    # decompression (decode_kernel)
    enc_dom = t_enc >= t_dec
    dom_kernel, dom_ach = ("code_kernel", enc_ach) if enc_dom else (dec_kernel, dec_ach)
    if batched:
        table_launches = lambda words: (words + 7679) // 7680
        per_step = (encode_launches(chunks, Wd, C, bool(flags & zc.SHARED_TABLES)) + table_launches(38 * n)
                    + 1 + table_launches(14 * n))
    else:
        per_step = sum(encode_launches([c], Wd, C, bool(flags & zc.SHARED_TABLES)) + (1 if c else 0) for c in chunks)
    line = {
        "metric": "round-trip GB/s (original bytes; encode + decode)",
        "value": round(replica_value(N, a.steps, world, total) / 1e9, 3), "unit": "GB/s",
        "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(1e3 * total / a.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": a.workload, "desc": MODEL_WORKLOADS[a.workload], "nbytes": N, "tensors": n,
                   "streams": n_streams, "packed_launches": packed,
                   "chunk_bytes": C, "threshold": thr, "verify_crc_on_decode": verify,
                   "format": FORMAT_NAMES[format_version(a)],
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"},
        "encode": {"gbs": round(N * a.steps / t_enc / 1e9, 2), "roofline_frac": round(enc_ach / hbm, 4),
                   "ms": round(1e3 * t_enc / a.steps, 4)},
        "decode": {"gbs": round(N * a.steps / t_dec / 1e9, 2), "roofline_frac": round(dec_ach / hbm, 4),
                   "ms": round(1e3 * t_dec / a.steps, 4)},
        "size_pct": round(100.0 * S / N, 3),
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "achieved": round(dom_ach, 1), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dom_ach / hbm, 4),
                     "frac_of_nominal": round(dom_ach / NOMINAL_HBM_GBS, 4),
                     "traffic": profiled_traffic(dom_kernel, a.workload, format_version(a), packed),
                     "algorithmic_bytes_per_launch": alg,
                     "note": ("compression" if enc_dom else "decompression") + " phase of the whole model ("
                             + ("one batched call" if batched else f"{n} calls on {n_streams} streams") + "): its "
                             "algorithmic bytes (original + blob) over its time; traffic likewise per phase"},
        "clocks": clk.summary(),
        "e2e": {"value": round(N * e2e_steps / t_hb / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": hb_h2d // e2e_steps, "d2h_bytes_per_step": hb_d2h // e2e_steps,
                "mode": "model copied from pinned host memory, blobs written to and decoded from pinned host "
                        "memory by the kernels, result copied back"},
        "e2e_device_blob": {"value": round(N * e2e_steps / t_e2e / 1e9, 3), "unit": "GB/s",
                            "h2d_bytes_per_step": h2d // e2e_steps, "d2h_bytes_per_step": d2h // e2e_steps,
                            "mode": "device blobs, copied to pinned host memory and back"},
        "gpu_launches": per_step * a.steps,
    }
    if batched_line is not None:
        bt_enc, bt_dec = batched_line
        line["batched"] = {
            "desc": "the same model, all tensors in one zc_compress_batch and one zc_decompress_batch call",
            "value": round(replica_value(N, a.steps, world, bt_enc + bt_dec) / 1e9, 3), "unit": "GB/s",
            "encode": {"gbs": round(N * a.steps / bt_enc / 1e9, 2), "ms": round(1e3 * bt_enc / a.steps, 4),
                       "roofline_frac": round(alg * a.steps / bt_enc / 1e9 / hbm, 4)},
            "decode": {"gbs": round(N * a.steps / bt_dec / 1e9, 2), "ms": round(1e3 * bt_dec / a.steps, 4),
                       "roofline_frac": round(alg * a.steps / bt_dec / 1e9 / hbm, 4)}}
    del src_all, out_all, blob_all
    first = wl.llama8b_tensor(0, *specs[0])
    line["cpu_baseline"] = cpu_baseline(first, code, a)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    a = _args()
    if a.impl == "reference":
        run_reference(a)
        return
    import torch
    import torch.distributed as dist
    import entropy_coding_gb300 as zc
    from entropy_coding_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    if a.workload in MODEL_WORKLOADS:
        run_model(a, world, rank, local, dev, stream)
        return

    t, desc = make_workload(a.workload, dev)
    code = wl.dtype_code(t)
    src = wl.as_bytes(t)
    base = None
    if a.workload == "bf16_delta_fused":
        ta, tb = wl.bf16_delta_pair(dev)
        base, src = wl.as_bytes(ta), wl.as_bytes(tb)
    N = src.numel()
    C, thr = a.chunk_bytes, a.threshold
    flags = format_flags(a, zc) | (zc.PACKED if a.packed else 0)
    planes = 512 * (N // max(1, t.numel())) if flags & zc.SHARED_TABLES else 0  # v2: the plane tables follow the chunk table
    cap = zc.blob_size(N, code, C, thr, flags)
    blob = torch.empty(cap, dtype=torch.uint8, device=dev)
    ws = torch.empty(zc.workspace_size(N, code, C, flags), dtype=torch.uint8, device=dev)
    nb = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(N, dtype=torch.uint8, device=dev)
    shape = tuple(t.shape)

    def comp(inp, blob=blob, nb=nb):
        if base is None:
            zc.compress_into(inp, blob, nb, ws, st, C, thr, stream, dtype=code, shape=shape, flags=flags)
        elif flags & ~zc.PACKED:  # a v2 or v3 delta goes through the batched entry point (a batch of one)
            zc.compress_batch_into([inp], [blob], nb, ws, st, code, [shape], C, thr, stream, bases=[base], flags=flags)
        else:
            zc.compress_delta_into(base, inp, blob, nb, ws, st, C, thr, stream, dtype=code, shape=shape)

    def decomp(info, blob=blob, out=out):
        if base is None:
            zc.decompress_into(blob, info, out, st, not a.no_verify, stream, packed=a.packed)
        else:
            zc.decompress_delta_into(blob, info, base, out, st, not a.no_verify, stream)

    # first pass outside timing: blob length, header, correctness
    with torch.cuda.stream(stream):
        comp(src)
    stream.synchronize()
    S = int(nb.item())
    assert int(st.item()) == 0
    info = zc.blob_info(blob[: 96 + 16 * ((N + C - 1) // C) + planes].cpu())
    with torch.cuda.stream(stream):
        decomp(info)
    stream.synchronize()
    assert int(st.item()) == 0 and torch.equal(out, src), "round trip failed"

    # inputs below 256 MiB would leave the tensor or the blob in the 129 MB L2
    # between iterations: write a 512 MiB buffer before each compression and
    # each decompression (outside the timed intervals)
    flush_l2 = N < (256 << 20)
    l2_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if flush_l2 else None

    def flush():
        if l2_buf is not None:
            l2_buf.zero_()

    def one_step(ev):
        flush()
        ev[0].record(stream)
        comp(src)
        ev[1].record(stream)
        flush()
        ev[2].record(stream)
        decomp(info)
        ev[3].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            one_step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    stream.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(a.steps)]
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for ev in evs:
                one_step(ev)
        stream.synchronize()
    torch.cuda.synchronize()
    t_enc = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    t_dec = sum(e[2].elapsed_time(e[3]) for e in evs) / 1e3
    assert int(st.item()) == 0 and int(nb.item()) == S
    total = t_enc + t_dec
    total, t_enc, t_dec = max_over_ranks([total, t_enc, t_dec], dev)

    # end to end through the public calls, host (pinned) buffers in and out
    h_src = torch.empty(N, dtype=torch.uint8, pin_memory=True)
    h_src.copy_(src.cpu())
    h_blob = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(N, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty_like(src)
    h2d = d2h = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if base is not None:  # the base checkpoint travels with each step too
        h_base = torch.empty(N, dtype=torch.uint8, pin_memory=True)
        h_base.copy_(base.cpu())
    for _ in range(a.e2e_steps):
        with torch.cuda.stream(stream):
            if base is not None:
                base.copy_(h_base, non_blocking=True)
            d_in.copy_(h_src, non_blocking=True)
            comp(d_in)
            s_bytes = int(nb.item())
            h_blob[:s_bytes].copy_(blob[:s_bytes], non_blocking=True)
            blob[:s_bytes].copy_(h_blob[:s_bytes], non_blocking=True)
            decomp(info)
            h_out.copy_(out, non_blocking=True)
        stream.synchronize()
        h2d += N + s_bytes + (N if base is not None else 0)
        d2h += s_bytes + 8 + N
    t_e2e = time.perf_counter() - t0
    assert torch.equal(h_out, h_src)

    # end to end with the blob in page-locked host memory: the coding kernel
    # writes it over the host link and the decoder reads it from there (no
    # blob copies); the host parses the header and table between the calls
    hb_blob = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
    hb_nb = torch.zeros(1, dtype=torch.int64, pin_memory=True)
    h_out.zero_()
    hb_h2d = hb_d2h = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(a.e2e_steps):
        with torch.cuda.stream(stream):
            if base is not None:
                base.copy_(h_base, non_blocking=True)
            d_in.copy_(h_src, non_blocking=True)
            comp(d_in, hb_blob, hb_nb)
        stream.synchronize()
        s_bytes = int(hb_nb.item())
        hb_info = zc.blob_info(hb_blob[: 96 + 16 * ((N + C - 1) // C) + planes])
        with torch.cuda.stream(stream):
            decomp(hb_info, hb_blob[:s_bytes])
            h_out.copy_(out, non_blocking=True)
        stream.synchronize()
        hb_h2d += N + s_bytes + (N if base is not None else 0)
        hb_d2h += s_bytes + 8 + N
    t_hb = time.perf_counter() - t0
    assert torch.equal(h_out, h_src)

    # zero copy: the tensor, the blob and the restored tensor all stay in
    # page-locked host memory; the kernels read and write them over the link
    zc_line = None
    if base is None:
        h_out.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(a.e2e_steps):
            with torch.cuda.stream(stream):
                comp(h_src, hb_blob, hb_nb)
            stream.synchronize()
            s_bytes = int(hb_nb.item())
            hb_info = zc.blob_info(hb_blob[: 96 + 16 * ((N + C - 1) // C) + planes])
            with torch.cuda.stream(stream):
                decomp(hb_info, hb_blob[:s_bytes], h_out)
            stream.synchronize()
        t_zc = time.perf_counter() - t0
        assert int(st.item()) == 0 and torch.equal(h_out, h_src)
        zc_line = {"value": round(N * a.e2e_steps / t_zc / 1e9, 3), "unit": "GB/s",
                   "h2d_bytes_per_step": hb_h2d // a.e2e_steps, "d2h_bytes_per_step": hb_d2h // a.e2e_steps,
                   "mode": "tensor, blob and restored tensor in pinned host memory, read and written by the "
                           "kernels (no copies)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    hbm, peak_kind = peaks()
    enc_gbs = N * a.steps / t_enc / 1e9
    dec_gbs = N * a.steps / t_dec / 1e9
    # algorithmic bytes per call: the input and the blob (a delta also reads
    # the base checkpoint, in both directions)
    alg = N + S + (N if base is not None else 0)
    enc_ach = alg * a.steps / t_enc / 1e9
    dec_ach = alg * a.steps / t_dec / 1e9
    # the roofline of the call that takes longer: compression (stats_kernel
    # then code_kernel; code_kernel is most of its time) or decompression
    # (one decode_kernel launch)
    enc_dom = t_enc >= t_dec
    dominant = "code_kernel" if enc_dom else ("decode_v2_kernel" if flags & zc.SHARED_TABLES else "decode_kernel")
    ach = enc_ach if enc_dom else dec_ach
    traffic = profiled_traffic(dominant, a.workload, format_version(a), a.packed)
    line = {
        "metric": "round-trip GB/s (original bytes; encode + decode)",
        "value": round(replica_value(N, a.steps, world, total) / 1e9, 3), "unit": "GB/s",
        "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(1e3 * total / a.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": a.workload, "desc": desc, "nbytes": N, "chunk_bytes": C, "threshold": thr,
                   "verify_crc_on_decode": not a.no_verify,
                   "l2": "512 MiB written before each compression and decompression (not timed)" if flush_l2
                   else "inputs larger than L2 (no flush)",
                   "format": FORMAT_NAMES[format_version(a)], "packed_launches": a.packed,
                   "parallelism": f"replicas x{world}"},
        "encode": {"gbs": round(enc_gbs, 2), "roofline_frac": round(enc_ach / hbm, 4),
                   "ms": round(1e3 * t_enc / a.steps, 4)},
        "decode": {"gbs": round(dec_gbs, 2), "roofline_frac": round(dec_ach / hbm, 4),
                   "ms": round(1e3 * t_dec / a.steps, 4)},
        "size_pct": round(100.0 * S / N, 3),
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(ach / hbm, 4),
                     "frac_of_nominal": round(ach / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": alg},
        "clocks": clk.summary(),
        # end to end through the public calls (cuZipNN's measured mode: a tensor
        # to a CPU blob and back): the tensor copied up from pinned memory, the
        # blob written to and decoded from pinned host memory by the kernels,
        # the result copied back
        "e2e": {"value": round(N * a.e2e_steps / t_hb / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": hb_h2d // a.e2e_steps, "d2h_bytes_per_step": hb_d2h // a.e2e_steps,
                "mode": "tensor copied from pinned host memory, blob written to and decoded from pinned host "
                        "memory by the kernels, result copied back"},
        "e2e_device_blob": {"value": round(N * a.e2e_steps / t_e2e / 1e9, 3), "unit": "GB/s",
                            "h2d_bytes_per_step": h2d // a.e2e_steps, "d2h_bytes_per_step": d2h // a.e2e_steps,
                            "mode": "device blob, copied to pinned host memory and back"},
        "e2e_zero_copy": zc_line,
        # stats_kernel + code_kernel (v2: + plane_kernel) + decode_kernel per step
        "gpu_launches": (encode_launches([(N + C - 1) // C], N // max(1, t.numel()), C, bool(flags & zc.SHARED_TABLES)) + 1) * a.steps,
    }
    line["cpu_baseline"] = cpu_baseline(t, code, a)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
