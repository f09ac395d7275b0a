"""CPU oracle of the emulated sum all-reduce -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The CUDA library neither
imports nor calls it, and the two share no code.

``ar_oracle.c`` holds the arithmetic (plain C loops, one IEEE binary32 add
per step); this module only builds it with gcc and marshals numpy arrays.
``model`` holds the pages' closed forms (traffic, busbw, the alpha-beta
model).  Arrays are payload bit patterns: ``np.uint16`` for bf16/fp16,
``np.float32`` for fp32, ``np.uint8`` for LL/LL128 lines.

Every function is pinned by ``tests/test_oracle_*.py`` against what the pages
and the mathematics fix; no function is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess
import threading

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SRC = _HERE / "ar_oracle.c"
_SO = _HERE / "_build" / "libar_oracle.so"
_DT = {"f32": 0, "bf16": 1, "f16": 2}
_ESZ = {"f32": 4, "bf16": 2, "f16": 2}
_lock = threading.Lock()
_lib = None

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> pathlib.Path:
    """Compile ar_oracle.c into _build/libar_oracle.so (gcc, host only)."""
    _SO.parent.mkdir(exist_ok=True)
    if force or not _SO.exists() or _SO.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _SO.with_suffix(f".{os.getpid()}.tmp")
        subprocess.run(["gcc", *CFLAGS, str(_SRC), "-o", str(tmp), "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(str(build()))
            vp, sz, i32, u32, u64 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                     ctypes.c_uint32, ctypes.c_uint64)
            pp = ctypes.POINTER(ctypes.c_void_p)
            sig = {
                "orc_bf16_to_f32_n": ([vp, vp, sz], None),
                "orc_f32_to_bf16_n": ([vp, vp, sz], None),
                "orc_f16_to_f32_n": ([vp, vp, sz], None),
                "orc_f32_to_f16_n": ([vp, vp, sz], None),
                "orc_all_reduce": ([i32, pp, pp, sz, i32], None),
                "orc_chunk_elems": ([i32, sz, i32], sz),
                "orc_reduce_scatter": ([i32, pp, pp, sz, i32], None),
                "orc_all_gather": ([i32, pp, sz, i32], None),
                "orc_ring": ([i32, pp, pp, sz, i32], i32),
                "orc_ring_order_sum": ([i32, pp, vp, vp, sz, i32], None),
                "orc_ll_bytes": ([sz], sz),
                "orc_ll_pack": ([vp, vp, sz, u32], None),
                "orc_ll_unpack": ([vp, vp, sz, u32], sz),
                "orc_ll_reduce": ([i32, pp, pp, sz, u32], sz),
                "orc_ll128_lines": ([sz], sz),
                "orc_ll128_bytes": ([sz], sz),
                "orc_ll128_pack": ([vp, vp, sz, u64], None),
                "orc_ll128_unpack": ([vp, vp, sz, u64], sz),
                "orc_ll128_reduce": ([i32, pp, pp, sz, u64], sz),
                "orc_ring_rounded": ([i32, pp, pp, sz, i32], i32),
                "orc_tree": ([i32, pp, pp, sz, i32], i32),
                "orc_all_gather_ring": ([i32, pp, sz, i32], i32),
                "orc_allreduce_rmsnorm": ([i32, pp, vp, vp, ctypes.c_double, vp, vp, sz, sz, i32], None),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptrs(arrs) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def _check(arrs, dtype):
    want = np.float32 if dtype == "f32" else np.uint16
    for a in arrs:
        if a.dtype != want or a.ndim != 1 or not a.flags["C_CONTIGUOUS"]:
            raise TypeError(f"{dtype} payload must be contiguous 1-D {np.dtype(want).name}")
    if len({a.size for a in arrs}) > 1:
        raise ValueError("rank buffers differ in length")


# --- payload conversions ---------------------------------------------------

def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    f = np.empty(h.size, np.float32)
    lib().orc_bf16_to_f32_n(_ptr(h), _ptr(f), h.size)
    return f


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    h = np.empty(f.size, np.uint16)
    lib().orc_f32_to_bf16_n(_ptr(f), _ptr(h), f.size)
    return h


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    f = np.empty(h.size, np.float32)
    lib().orc_f16_to_f32_n(_ptr(h), _ptr(f), h.size)
    return f


def f32_to_f16(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    h = np.empty(f.size, np.uint16)
    lib().orc_f32_to_f16_n(_ptr(f), _ptr(h), f.size)
    return h


def to_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of a payload array to float32."""
    if dtype == "f32":
        return np.asarray(a, np.float32)
    return bf16_to_f32(a) if dtype == "bf16" else f16_to_f32(a)


# --- all-reduce ------------------------------------------------------------

def _outs(inputs, n):
    return [np.empty_like(inputs[0]) for _ in range(n)]


def all_reduce(inputs: list, dtype: str) -> list:
    """One-shot definition: every rank gets the rank-order fp32 sum, rounded once."""
    _check(inputs, dtype)
    n, N = len(inputs), inputs[0].size
    out = _outs(inputs, n)
    lib().orc_all_reduce(n, _ptrs(inputs), _ptrs(out), N, _DT[dtype])
    return out


def chunk_elems(n: int, N: int, dtype: str) -> int:
    return lib().orc_chunk_elems(n, N, _DT[dtype])


def reduce_scatter(inputs: list, dtype: str, out: list | None = None) -> list:
    """out[r][chunk r] = rank-order sum of chunk r; the rest of out[r] is untouched."""
    _check(inputs, dtype)
    n, N = len(inputs), inputs[0].size
    if out is None:
        out = [np.zeros_like(inputs[0]) for _ in range(n)]
    lib().orc_reduce_scatter(n, _ptrs(inputs), _ptrs(out), N, _DT[dtype])
    return out


def all_gather(out: list, dtype: str) -> list:
    """In place: every rank copies chunk j from rank j."""
    _check(out, dtype)
    lib().orc_all_gather(len(out), _ptrs(out), out[0].size, _DT[dtype])
    return out


def ring(inputs: list, dtype: str) -> list:
    """The 2(n-1)-step chunked ring, simulated step by step with fp32 partials."""
    _check(inputs, dtype)
    n, N = len(inputs), inputs[0].size
    out = _outs(inputs, n)
    rc = lib().orc_ring(n, _ptrs(inputs), _ptrs(out), N, _DT[dtype])
    if rc != 0:
        raise MemoryError("oracle ring: out of host memory")
    return out


def ring_rounded(inputs: list, dtype: str) -> list:
    """The ring with partials rounded to the payload type at every hop."""
    _check(inputs, dtype)
    n, N = len(inputs), inputs[0].size
    out = _outs(inputs, n)
    if lib().orc_ring_rounded(n, _ptrs(inputs), _ptrs(out), N, _DT[dtype]) != 0:
        raise MemoryError("oracle ring: out of host memory")
    return out


def tree(inputs: list, dtype: str) -> list:
    """The pairwise (recursive-doubling) tree, each level rounded to the payload type."""
    _check(inputs, dtype)
    n, N = len(inputs), inputs[0].size
    out = _outs(inputs, n)
    rc = lib().orc_tree(n, _ptrs(inputs), _ptrs(out), N, _DT[dtype])
    if rc == -1:
        raise ValueError("the pairwise tree needs a power-of-two number of ranks")
    if rc != 0:
        raise MemoryError("oracle tree: out of host memory")
    return out


def ring_order_sum(cols: list, chunk: np.ndarray, dtype: str) -> np.ndarray:
    """Per sampled element k: RN(x_c + x_{c+1} + ... + x_{c+n-1}), c = chunk[k]."""
    _check(cols, dtype)
    chunk = np.ascontiguousarray(chunk, dtype=np.int32)
    res = np.empty_like(cols[0])
    lib().orc_ring_order_sum(len(cols), _ptrs(cols), _ptr(chunk), _ptr(res), cols[0].size, _DT[dtype])
    return res


def sampled_all_reduce(inputs: list, idx: np.ndarray, dtype: str) -> np.ndarray:
    """The one-shot result at the element indices ``idx`` only."""
    cols = [np.ascontiguousarray(a[idx]) for a in inputs]
    return all_reduce(cols, dtype)[0]


# --- LL / LL128 ------------------------------------------------------------

def ll_bytes(count: int) -> int:
    return lib().orc_ll_bytes(count)


def ll128_lines(count: int) -> int:
    return lib().orc_ll128_lines(count)


def ll128_bytes(count: int) -> int:
    return lib().orc_ll128_bytes(count)


def _f32(src):
    src = np.ascontiguousarray(src)
    if src.dtype != np.float32 or src.ndim != 1:
        raise TypeError("LL payload must be 1-D float32")
    return src


def ll_pack(src: np.ndarray, step: int) -> np.ndarray:
    src = _f32(src)
    lines = np.empty(ll_bytes(src.size), np.uint8)
    lib().orc_ll_pack(_ptr(src), _ptr(lines), src.size, step)
    return lines


def ll_unpack(lines: np.ndarray, count: int, step: int, dst: np.ndarray | None = None):
    """Returns (dst, number of lines whose flag was not ``step``)."""
    dst = np.zeros(count, np.float32) if dst is None else dst
    bad = lib().orc_ll_unpack(_ptr(lines), _ptr(dst), count, step)
    return dst, bad


def ll_reduce(lines_in: list, count: int, step: int, lines_out: list | None = None):
    n = len(lines_in)
    if lines_out is None:
        lines_out = [np.zeros_like(lines_in[0]) for _ in range(n)]
    bad = lib().orc_ll_reduce(n, _ptrs(lines_in), _ptrs(lines_out), count, step)
    return lines_out, bad


def ll128_pack(src: np.ndarray, step: int) -> np.ndarray:
    src = _f32(src)
    lines = np.empty(ll128_bytes(src.size), np.uint8)
    lib().orc_ll128_pack(_ptr(src), _ptr(lines), src.size, step)
    return lines


def ll128_unpack(lines: np.ndarray, count: int, step: int, dst: np.ndarray | None = None):
    dst = np.zeros(count, np.float32) if dst is None else dst
    bad = lib().orc_ll128_unpack(_ptr(lines), _ptr(dst), count, step)
    return dst, bad


def ll128_reduce(lines_in: list, count: int, step: int, lines_out: list | None = None):
    n = len(lines_in)
    if lines_out is None:
        lines_out = [np.zeros_like(lines_in[0]) for _ in range(n)]
    bad = lib().orc_ll128_reduce(n, _ptrs(lines_in), _ptrs(lines_out), count, step)
    return lines_out, bad


# --- fused all-reduce + residual add + RMSNorm ------------------------------

def allreduce_rmsnorm(inputs: list, residual: np.ndarray, weight: np.ndarray, eps: float, tokens: int,
                      hidden: int, dtype: str):
    """Returns (norm_out, residual_out), each [tokens * hidden] in the payload type."""
    _check(inputs, dtype)
    _check([residual], dtype)
    _check([weight], dtype)
    assert inputs[0].size == residual.size == tokens * hidden and weight.size == hidden
    norm = np.empty_like(residual)
    res_out = np.empty_like(residual)
    lib().orc_allreduce_rmsnorm(len(inputs), _ptrs(inputs), _ptr(residual), _ptr(weight), eps, _ptr(norm),
                                _ptr(res_out), tokens, hidden, _DT[dtype])
    return norm, res_out
