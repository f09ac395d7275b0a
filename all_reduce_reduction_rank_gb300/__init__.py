"""Python binding of libar_gb300.so (include/ar.h): argument marshalling only.

Every step of the all-reduce runs in the library's CUDA kernels; this module
turns torch tensors (or raw device addresses) and torch streams into the
pointers and sizes of the C-ABI and returns its codes.  It never falls back
to another implementation: if the library is missing, importing
``lib()`` raises.

Functions keep the C names: ``ar_create``, ``ar_one_shot``, ... .  Rank
buffers may be given as torch tensors (their ``data_ptr()``) or as integer
device addresses; ``stream`` may be a ``torch.cuda.Stream``, an integer
``cudaStream_t`` or ``None`` (the legacy default stream).
"""

from __future__ import annotations

import ctypes
import pathlib
import threading

_PKG = pathlib.Path(__file__).resolve().parent
LIB_PATH = _PKG / "libar_gb300.so"

AR_F32, AR_BF16, AR_F16 = 0, 1, 2
DTYPES = {"f32": AR_F32, "bf16": AR_BF16, "f16": AR_F16}
AR_OK, AR_ERR_INVALID, AR_ERR_ALIGN, AR_ERR_TOO_LARGE, AR_ERR_CUDA, AR_ERR_FLAG_TIMEOUT, AR_ERR_WAIT_TIMEOUT = (
    0, -1, -2, -3, -4, -5, -6)
(AR_OP_NONE, AR_OP_ONE_SHOT, AR_OP_TWO_SHOT, AR_OP_RING, AR_OP_LL_PACK, AR_OP_LL_UNPACK, AR_OP_LL_REDUCE,
 AR_OP_LL128_PACK, AR_OP_LL128_UNPACK, AR_OP_LL128_REDUCE, AR_OP_ALLREDUCE_RMSNORM, AR_OP_ONE_SHOT_PUSH,
 AR_OP_ONE_SHOT_COPYIN, AR_OP_RING_ROUNDED, AR_OP_TREE, AR_OP_RING_PERSISTENT, AR_OP_RING_CLUSTER,
 AR_OP_TREE_FUSED, AR_OP_RING_FUSED, AR_OP_RING_ROUNDED_FUSED) = range(20)
AR_OPT_CTAS_PER_SM, AR_OPT_SPIN_NS, AR_OPT_ONE_SHOT_IMPL, AR_OPT_TIMING, AR_OPT_TIMING_PAUSE, AR_OPT_PDL = 1, 2, 3, 4, 5, 6
AR_OPT_AUTO_POLICY, AR_OPT_AUTO_ALPHA_NS, AR_OPT_AUTO_BETA_MBS, AR_OPT_AUTO_HANDOFF = 7, 8, 9, 10
AR_OPT_PUSH_STAGING, AR_OPT_REGISTERED, AR_OPT_PERSISTENT, AR_OPT_ABSENT_RANK = 11, 12, 13, 14
AR_OPT_TWO_SHOT_IMPL = 15
AR_AUTO_MODEL, AR_AUTO_EMULATED = 0, 1
KERNELS = {1: "one_shot", 2: "reduce_scatter", 3: "all_gather", 4: "ring_rs_step", 5: "ring_ag_step",
           6: "ll_pack", 7: "ll_unpack", 8: "ll_reduce", 9: "ll128_pack", 10: "ll128_unpack",
           11: "ll128_reduce", 12: "allreduce_rmsnorm", 13: "push", 14: "push_reduce",
           15: "ring_rs_step_rounded", 16: "tree_level", 17: "ring_persistent",
           18: "copyin", 19: "ring_cluster", 20: "tree_fused", 21: "ring_fused", 22: "ring_rounded_fused",
           23: "two_shot"}

# C symbols the header declares (checked by the CPU tests against include/ar.h)
EXPORTS = (
    "ar_create", "ar_destroy", "ar_set_option", "ar_one_shot", "ar_two_shot", "ar_ring",
    "ar_ll_bytes", "ar_ll128_bytes", "ar_ll_pack", "ar_ll_unpack", "ar_ll128_pack", "ar_ll128_unpack",
    "ar_ll_reduce", "ar_ll128_reduce", "ar_status", "ar_status_info", "ar_traffic", "ar_plan",
    "ar_check_args", "ar_strerror", "ar_timing", "ar_ll_pack_n", "ar_ll_unpack_n", "ar_ll128_pack_n",
    "ar_ll128_unpack_n", "ar_ring_noalloc", "ar_select", "ar_auto", "ar_allreduce_rmsnorm",
    "ar_one_shot_push", "ar_one_shot_copyin", "ar_ring_rounded", "ar_tree", "ar_ring_persistent",
    "ar_ring_cluster", "ar_tree_fused", "ar_ring_fused", "ar_ring_rounded_fused",
)


class Traffic(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int), ("n_ranks", ctypes.c_int), ("count", ctypes.c_size_t),
                ("elem_bytes", ctypes.c_size_t), ("link_bytes_per_rank", ctypes.c_double),
                ("steps", ctypes.c_int), ("launches", ctypes.c_int),
                ("hbm_read_bytes", ctypes.c_uint64), ("hbm_write_bytes", ctypes.c_uint64)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class StatusInfo(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int), ("rank", ctypes.c_int), ("line", ctypes.c_uint64),
                ("lines_skipped", ctypes.c_uint64)]


class LaunchTime(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("op", ctypes.c_int), ("ms", ctypes.c_float),
                ("hbm_bytes", ctypes.c_uint64), ("launches", ctypes.c_int)]


class ArError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {ar_strerror(code)} ({code})" if what else f"{ar_strerror(code)} ({code})")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libar_gb300.so from the package directory (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise ImportError(f"{LIB_PATH} is not built; run all_reduce_reduction_rank_gb300.build.build()")
            L = ctypes.CDLL(str(LIB_PATH))
            vp, sz, i32, u32, u64, i64 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32,
                                          ctypes.c_uint64, ctypes.c_int64)
            pp = ctypes.POINTER(ctypes.c_void_p)
            sig = {
                "ar_create": ([i32, sz, ctypes.POINTER(vp)], i32),
                "ar_destroy": ([vp], i32),
                "ar_set_option": ([vp, i32, i64], i32),
                "ar_one_shot": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_two_shot": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ring": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ring_noalloc": ([i32, pp, pp, sz, i32, vp], i32),
                "ar_select": ([i32, i32, sz, ctypes.c_double, ctypes.c_double, sz], i32),
                "ar_auto": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_allreduce_rmsnorm": ([vp, pp, vp, vp, ctypes.c_float, pp, vp, sz, sz, i32, vp], i32),
                "ar_one_shot_push": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_one_shot_copyin": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ring_rounded": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_tree": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ring_persistent": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ring_cluster": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_tree_fused": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ring_fused": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ring_rounded_fused": ([vp, pp, pp, sz, i32, vp], i32),
                "ar_ll_bytes": ([sz], sz),
                "ar_ll128_bytes": ([sz], sz),
                "ar_ll_pack": ([vp, vp, vp, sz, u32, vp], i32),
                "ar_ll_unpack": ([vp, vp, vp, sz, u32, vp], i32),
                "ar_ll128_pack": ([vp, vp, vp, sz, u64, vp], i32),
                "ar_ll128_unpack": ([vp, vp, vp, sz, u64, vp], i32),
                "ar_ll_pack_n": ([vp, pp, pp, sz, u32, vp], i32),
                "ar_ll_unpack_n": ([vp, pp, pp, sz, u32, vp], i32),
                "ar_ll128_pack_n": ([vp, pp, pp, sz, u64, vp], i32),
                "ar_ll128_unpack_n": ([vp, pp, pp, sz, u64, vp], i32),
                "ar_ll_reduce": ([vp, pp, pp, sz, u32, vp], i32),
                "ar_ll128_reduce": ([vp, pp, pp, sz, u64, vp], i32),
                "ar_status": ([vp], i32),
                "ar_status_info": ([vp, ctypes.POINTER(StatusInfo)], i32),
                "ar_traffic": ([vp, ctypes.POINTER(Traffic)], i32),
                "ar_plan": ([i32, i32, sz, i32, ctypes.POINTER(Traffic)], i32),
                "ar_check_args": ([i32, i32, sz, pp, pp, sz, i32], i32),
                "ar_strerror": ([i32], ctypes.c_char_p),
                "ar_timing": ([vp, ctypes.POINTER(LaunchTime), i32, ctypes.POINTER(i32)], i32),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


# ---- marshalling helpers ----------------------------------------------------

def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())  # torch.Tensor


def _ptr_array(bufs) -> ctypes.Array:
    return (ctypes.c_void_p * len(bufs))(*[_addr(b) for b in bufs])


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return int(s.cuda_stream) or None  # torch.cuda.Stream


def _dtype(dt) -> int:
    return DTYPES[dt] if isinstance(dt, str) else int(dt)


# ---- the C-ABI, same names ----------------------------------------------------

def ar_strerror(code: int) -> str:
    return lib().ar_strerror(code).decode()


def ar_create(n_ranks: int, max_bytes: int) -> int:
    """Returns the handle (an opaque address); raises ArError on failure."""
    h = ctypes.c_void_p()
    rc = lib().ar_create(n_ranks, max_bytes, ctypes.byref(h))
    if rc != AR_OK:
        raise ArError(rc, "ar_create")
    return h.value


def ar_destroy(h: int) -> int:
    return lib().ar_destroy(h)


def ar_set_option(h: int, option: int, value: int) -> int:
    return lib().ar_set_option(h, option, value)


def ar_one_shot(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_one_shot(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_two_shot(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_two_shot(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_one_shot_push(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_one_shot_push(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_one_shot_copyin(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_one_shot_copyin(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_ring_rounded(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_ring_rounded(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_tree(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_tree(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_ring_persistent(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_ring_persistent(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_ring_cluster(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_ring_cluster(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_tree_fused(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_tree_fused(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_ring_fused(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_ring_fused(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_ring_rounded_fused(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_ring_rounded_fused(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype),
                                       _stream(stream))


def ar_ring(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_ring(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_select(policy: int, n_ranks: int, bytes_per_rank: int, alpha_s: float = 1.5e-6,
              beta_bytes_per_s: float = 450e9, handoff_bytes: int = 8 << 20) -> int:
    return lib().ar_select(policy, n_ranks, bytes_per_rank, alpha_s, beta_bytes_per_s, handoff_bytes)


def ar_auto(h, ins, outs, count: int, dtype, stream=None) -> int:
    return lib().ar_auto(h, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_allreduce_rmsnorm(h, ins, residual, weight, eps: float, norm_outs, residual_out, tokens: int,
                         hidden: int, dtype, stream=None) -> int:
    return lib().ar_allreduce_rmsnorm(h, _ptr_array(ins), _addr(residual), _addr(weight), eps, _ptr_array(norm_outs),
                                      _addr(residual_out), tokens, hidden, _dtype(dtype), _stream(stream))


def ar_ring_noalloc(n_ranks: int, ins, outs, count: int, dtype, stream=None) -> int:
    """ar_ring without a handle or any allocation (static 32 MiB scratch in the library)."""
    return lib().ar_ring_noalloc(n_ranks, _ptr_array(ins), _ptr_array(outs), count, _dtype(dtype), _stream(stream))


def ar_ll_bytes(payload_bytes: int) -> int:
    return lib().ar_ll_bytes(payload_bytes)


def ar_ll128_bytes(payload_bytes: int) -> int:
    return lib().ar_ll128_bytes(payload_bytes)


def ar_ll_pack(h, src, lines, count: int, step: int, stream=None) -> int:
    return lib().ar_ll_pack(h, _addr(src), _addr(lines), count, step, _stream(stream))


def ar_ll_unpack(h, lines, dst, count: int, step: int, stream=None) -> int:
    return lib().ar_ll_unpack(h, _addr(lines), _addr(dst), count, step, _stream(stream))


def ar_ll128_pack(h, src, lines, count: int, step: int, stream=None) -> int:
    return lib().ar_ll128_pack(h, _addr(src), _addr(lines), count, step, _stream(stream))


def ar_ll128_unpack(h, lines, dst, count: int, step: int, stream=None) -> int:
    return lib().ar_ll128_unpack(h, _addr(lines), _addr(dst), count, step, _stream(stream))


def ar_ll_pack_n(h, srcs, lines, count: int, step: int, stream=None) -> int:
    return lib().ar_ll_pack_n(h, _ptr_array(srcs), _ptr_array(lines), count, step, _stream(stream))


def ar_ll_unpack_n(h, lines, dsts, count: int, step: int, stream=None) -> int:
    return lib().ar_ll_unpack_n(h, _ptr_array(lines), _ptr_array(dsts), count, step, _stream(stream))


def ar_ll128_pack_n(h, srcs, lines, count: int, step: int, stream=None) -> int:
    return lib().ar_ll128_pack_n(h, _ptr_array(srcs), _ptr_array(lines), count, step, _stream(stream))


def ar_ll128_unpack_n(h, lines, dsts, count: int, step: int, stream=None) -> int:
    return lib().ar_ll128_unpack_n(h, _ptr_array(lines), _ptr_array(dsts), count, step, _stream(stream))


def ar_ll_reduce(h, lines_in, lines_out, count: int, step: int, stream=None) -> int:
    return lib().ar_ll_reduce(h, _ptr_array(lines_in), _ptr_array(lines_out), count, step, _stream(stream))


def ar_ll128_reduce(h, lines_in, lines_out, count: int, step: int, stream=None) -> int:
    return lib().ar_ll128_reduce(h, _ptr_array(lines_in), _ptr_array(lines_out), count, step, _stream(stream))


def ar_status(h) -> int:
    return lib().ar_status(h)


def ar_status_info(h) -> tuple[int, StatusInfo]:
    info = StatusInfo()
    rc = lib().ar_status_info(h, ctypes.byref(info))
    return rc, info


def ar_traffic(h) -> Traffic:
    t = Traffic()
    rc = lib().ar_traffic(h, ctypes.byref(t))
    if rc != AR_OK:
        raise ArError(rc, "ar_traffic")
    return t


def ar_plan(op: int, n_ranks: int, count: int, dtype) -> Traffic:
    t = Traffic()
    rc = lib().ar_plan(op, n_ranks, count, _dtype(dtype), ctypes.byref(t))
    if rc != AR_OK:
        raise ArError(rc, "ar_plan")
    return t


def ar_check_args(op: int, n_ranks: int, max_bytes: int, ins, outs, count: int, dtype) -> int:
    pin = _ptr_array(ins) if ins is not None else None
    pout = _ptr_array(outs) if outs is not None else None
    return lib().ar_check_args(op, n_ranks, max_bytes, pin, pout, count, _dtype(dtype))


def ar_timing(h, max_records: int = 1 << 20) -> list[tuple[str, int, float, int, int]]:
    """Timing records, oldest first: (kernel name, op, ms, hbm bytes, launches)."""
    buf = (LaunchTime * max_records)()
    n = ctypes.c_int(0)
    rc = lib().ar_timing(h, buf, max_records, ctypes.byref(n))
    if rc != AR_OK:
        raise ArError(rc, "ar_timing")
    return [(KERNELS.get(buf[i].kernel, str(buf[i].kernel)), buf[i].op, buf[i].ms, buf[i].hbm_bytes,
             buf[i].launches) for i in range(n.value)]


def check(rc: int, what: str = "") -> None:
    """Raise ArError for a non-zero code."""
    if rc != AR_OK:
        raise ArError(rc, what)
