"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random tensors; it holds none of the compression
arithmetic, so both the GPU path's callers and the oracle's tests can use it.

Workloads (ZipNN note, Table II models; lmzip README, Llama-3.1-8B shards):

* ``bf16_1m``      BF16 1024x1024, N(0, 0.02), seed 0
* ``fp32_64m``     FP32 8192x8192, N(0, 0.02), seed 1 ("regular" FP32)
* ``fp32clean_64m`` FP32 8192x8192, N(0, 0.02) seed 2 rounded to BF16 and
  widened back ("clean" FP32: the two low bytes of every word are zero)
* ``fp16_16m``     FP16 4096x4096, N(0, 0.05), seed 3
* ``bf16_delta``   two BF16 4096x14336 tensors, the second the first plus
  N(0, 1e-4), seed 4; the XOR of their bit patterns is compressed as U16
* ``llama8b``      Llama-3.1-8B-shaped BF16 tensors, N(0, 0.02) per tensor
  (seed 1000 + index), RMSNorm vectors of ones
"""
from __future__ import annotations

import torch

# dtype codes of the blob header
U8, U16, U32, BF16, FP16, FP32 = 1, 2, 3, 4, 5, 6
TORCH_CODE = {torch.uint8: U8, torch.int16: U16, torch.uint16: U16, torch.int32: U32,
              torch.uint32: U32, torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}


def _randn(shape, seed: int, device, std: float) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std


def bf16_1m(device="cpu") -> torch.Tensor:
    return _randn((1024, 1024), 0, device, 0.02).bfloat16()


def fp32_64m(device="cpu", rows: int = 8192) -> torch.Tensor:
    return _randn((rows, 8192), 1, device, 0.02)


def fp32clean_64m(device="cpu", rows: int = 8192) -> torch.Tensor:
    return _randn((rows, 8192), 2, device, 0.02).bfloat16().float()


def fp16_16m(device="cpu", rows: int = 4096) -> torch.Tensor:
    return _randn((rows, 4096), 3, device, 0.05).half()


def bf16_delta(device="cpu", rows: int = 4096) -> tuple[torch.Tensor, torch.Tensor]:
    """(a, x): the base BF16 tensor and the U16 XOR of a with its update."""
    g = torch.Generator(device=device)
    g.manual_seed(4)
    a = (torch.randn(rows, 14336, generator=g, device=device) * 0.02).bfloat16()
    b = (a.float() + torch.randn(rows, 14336, generator=g, device=device) * 1e-4).bfloat16()
    x = a.view(torch.int16) ^ b.view(torch.int16)
    return a, x


def bf16_delta_pair(device="cpu", rows: int = 4096) -> tuple[torch.Tensor, torch.Tensor]:
    """(a, b): a base BF16 checkpoint tensor and its update (same draws as
    bf16_delta, which returns their XOR instead of b)."""
    g = torch.Generator(device=device)
    g.manual_seed(4)
    a = (torch.randn(rows, 14336, generator=g, device=device) * 0.02).bfloat16()
    b = (a.float() + torch.randn(rows, 14336, generator=g, device=device) * 1e-4).bfloat16()
    return a, b


LLAMA_LAYERS = 32
LLAMA_LAYER_SHAPES = [("q", (4096, 4096)), ("k", (1024, 4096)), ("v", (1024, 4096)),
                      ("o", (4096, 4096)), ("gate", (14336, 4096)), ("up", (14336, 4096)),
                      ("down", (4096, 14336)), ("input_norm", (4096,)), ("post_norm", (4096,))]


def llama8b_specs(layers: int = LLAMA_LAYERS) -> list[tuple[str, tuple[int, ...]]]:
    """Tensor names and shapes in compression order."""
    specs = [("embed", (128256, 4096))]
    for i in range(layers):
        specs += [(f"layers.{i}.{n}", s) for n, s in LLAMA_LAYER_SHAPES]
    specs.append(("lm_head", (4096, 128256)))
    return specs


def llama8b_tensor(index: int, name: str, shape, device="cpu") -> torch.Tensor:
    if name.endswith("norm"):
        return torch.ones(shape, dtype=torch.bfloat16, device=device)
    return _randn(shape, 1000 + index, device, 0.02).bfloat16()


def dtype_code(t: torch.Tensor) -> int:
    return TORCH_CODE[t.dtype]


def as_bytes(t: torch.Tensor) -> torch.Tensor:
    """The tensor's bytes as a flat uint8 view (row-major)."""
    return t.contiguous().view(-1).view(torch.uint8)
