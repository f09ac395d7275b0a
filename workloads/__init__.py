"""Seeded synthetic inputs for the emulated sum all-reduce.

This module is shared by the tests, the smoke check and the bench. It holds
no part of the method's arithmetic: it only draws numbers and lays them out
as raw bit patterns (``np.uint16`` for bf16/fp16, ``np.float32`` for fp32).

The workloads stand in for the ones the pages measure on:
- the nccl-tests doubling size sweep ("all_reduce_perf -b 8 -e 1G -f 2",
  handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §读懂 nccl-tests);
- tensor-parallel decode and prefill all-reduces at hidden 4096/8192 in bf16
  (handbook "多 GPU 与 NCCL", §练习 exercise 1: 1 token x 8192 x 2 B for decode,
  8192 tokens x 8192 x 2 B for prefill);
- the fill pattern ``g + i % 7`` of the NCCL example program (same chapter,
  §NCCL 编程, ``fill`` kernel).

Recipe: rank r of a call seeded ``seed`` draws from
``np.random.default_rng(np.random.SeedSequence(seed).spawn(n)[r])``.
Values are drawn as float32 and then laid out in the payload type:
- bf16: the upper 16 bits of the float32 (truncation toward zero; the draw
  is only a distribution, so no rounding rule is implied);
- fp16: ``numpy.ndarray.astype(np.float16)``;
- fp32: as drawn.
Integer-valued draws are exact in every payload type.
"""

from __future__ import annotations

import numpy as np

DTYPES = ("f32", "bf16", "f16")
ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2}
STORAGE = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16}

KiB = 1 << 10
MiB = 1 << 20


def _layout(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 draw -> payload bit pattern (see module docstring)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return (x.view(np.uint32) >> 16).astype(np.uint16)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def _draw(rng: np.random.Generator, dist: str, count: int, n: int, rank: int) -> np.ndarray:
    if dist == "int8":  # integers uniform in {-8, ..., 8}
        return rng.integers(-8, 9, size=count).astype(np.float32)
    if dist == "normal":  # N(0, 1)
        return rng.standard_normal(count, dtype=np.float32)
    if dist == "normal_over_n":  # N(0, 1) / n  (n is a power of two in every config)
        return rng.standard_normal(count, dtype=np.float32) / np.float32(n)
    if dist == "uniform":  # U[-1, 1]
        return rng.uniform(-1.0, 1.0, size=count).astype(np.float32)
    if dist == "fill7":  # the NCCL example's pattern: rank g holds g + i % 7
        return (np.float32(rank) + (np.arange(count) % 7)).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def rank_inputs(n: int, count: int, dtype: str, dist: str, seed: int) -> list[np.ndarray]:
    """n seeded rank buffers of ``count`` elements each, as payload bit patterns."""
    children = np.random.SeedSequence(seed).spawn(n)
    out = []
    for r in range(n):
        rng = np.random.default_rng(children[r])
        out.append(_layout(_draw(rng, dist, count, n, r), dtype))
    return out


def payload_f32(n: int, count: int, seed: int, dist: str = "uniform") -> list[np.ndarray]:
    """fp32 payloads for the LL / LL128 protocol rows."""
    return rank_inputs(n, count, "f32", dist, seed)


# The five workloads.  ``seed = 1000 + number``.
CONFIGS = {
    1: dict(name="n2_f32_int", n=2, dtype="f32", dist="int8", counts=[1024],
            algos=("one_shot", "two_shot", "ring")),
    2: dict(name="n8_bf16_decode", n=8, dtype="bf16", dist="normal",
            counts=[t * h for t in (1, 8, 32, 64) for h in (4096, 8192)],
            algos=("one_shot", "two_shot")),
    3: dict(name="n8_bf16_prefill", n=8, dtype="bf16", dist="normal",
            counts=[s // 2 for s in (8 * MiB, 16 * MiB, 32 * MiB, 64 * MiB)],
            algos=("two_shot", "one_shot")),
    4: dict(name="n8_f32_ll", n=8, dtype="f32", dist="uniform",
            counts=[(8 << k) // 4 for k in range(18)],  # payload 8 B .. 1 MiB
            algos=("ll", "ll128")),
    5: dict(name="n16_sweep", n=16, dtype=("bf16", "f16"), dist="normal_over_n",
            counts=[(KiB << k) // 2 for k in range(19)],  # 1 KiB .. 256 MiB
            algos=("ring", "one_shot", "two_shot")),
}


def seed_of(config: int) -> int:
    return 1000 + config


def rank_inputs_device(n: int, count: int, dtype: str, dist: str, seed: int, device="cuda"):
    """Large seeded rank buffers drawn on the device (torch's Philox
    generator, seeded per rank with ``seed * 1000 + r``), laid out with the
    same recipe as ``rank_inputs``; returns torch tensors of payload bits
    (int16 for bf16/fp16, float32 for fp32).  Used where host generation of
    gigabytes would dominate the run; the oracle then reads sampled columns
    of these inputs back from the device."""
    import torch

    out = []
    for r in range(n):
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + r)
        if dist == "normal":
            x = torch.randn(count, generator=g, device=device, dtype=torch.float32)
        elif dist == "normal_over_n":
            x = torch.randn(count, generator=g, device=device, dtype=torch.float32) / n
        elif dist == "uniform":
            x = torch.rand(count, generator=g, device=device, dtype=torch.float32) * 2 - 1
        elif dist == "int8":
            x = torch.randint(-8, 9, (count,), generator=g, device=device).to(torch.float32)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        if dtype == "f32":
            out.append(x)
        elif dtype == "bf16":
            out.append(torch.bitwise_right_shift(x.view(torch.int32), 16).to(torch.int16))
        elif dtype == "f16":
            out.append(x.to(torch.float16).view(torch.int16))
        else:
            raise ValueError(f"unknown dtype {dtype!r}")
        del x
    return out
