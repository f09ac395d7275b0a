"""Helpers for the GPU tests: rank buffers with guard bands, uploads of
payload bit patterns, downloads back to numpy.  Torch only provides device
memory and streams here; all arithmetic runs in libar_gb300.so."""

from __future__ import annotations

import numpy as np
import torch

import all_reduce_reduction_rank_gb300 as ar

GUARD = 256          # bytes of canary before and after every buffer
CANARY = 0xA5


class Buf:
    """One device buffer of `nbytes` with canary bands on both sides."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = nbytes
        body = (nbytes + 255) // 256 * 256
        self.raw = torch.full((GUARD + body + GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.ptr = self.raw.data_ptr() + GUARD
        assert self.ptr % 256 == 0 or self.ptr % 16 == 0

    def body(self) -> torch.Tensor:
        return self.raw[GUARD:GUARD + self.nbytes]

    def upload(self, a: np.ndarray) -> "Buf":
        b = np.ascontiguousarray(a).view(np.uint8)
        assert b.size == self.nbytes
        self.body().copy_(torch.from_numpy(b.copy()))
        return self

    def fill(self, byte: int) -> "Buf":
        self.body().fill_(byte)
        return self

    def download(self, dtype) -> np.ndarray:
        return self.body().cpu().numpy().view(dtype)

    def guards_intact(self) -> bool:
        head = self.raw[:GUARD]
        body = (self.nbytes + 255) // 256 * 256
        tail = self.raw[GUARD + self.nbytes:]
        assert tail.numel() == body - self.nbytes + GUARD
        return bool((head == CANARY).all()) and bool((tail == CANARY).all())


def payload_np_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def upload_ranks(arrays) -> list[Buf]:
    return [Buf(a.nbytes).upload(a) for a in arrays]


def empty_ranks(n: int, nbytes: int, byte: int = 0x5A) -> list[Buf]:
    return [Buf(nbytes).fill(byte) for _ in range(n)]


def ptrs(bufs) -> list[int]:
    return [b.ptr for b in bufs]


class Handle:
    """Context manager around ar_create / ar_destroy."""

    def __init__(self, n: int, max_bytes: int, **options):
        self.n, self.max_bytes, self.options = n, max_bytes, options

    def __enter__(self) -> int:
        self.h = ar.ar_create(self.n, self.max_bytes)
        for k, v in self.options.items():
            ar.check(ar.ar_set_option(self.h, getattr(ar, "AR_OPT_" + k.upper()), v), k)
        return self.h

    def __exit__(self, *exc):
        rc = ar.ar_destroy(self.h)
        assert rc == ar.AR_OK, ar.ar_strerror(rc)
        return False


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint16)
