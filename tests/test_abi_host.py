"""The C-ABI library without a GPU: it loads, exports every symbol that
include/ar.h declares, and its host-only logic (sizes, traffic plan,
argument checks, error codes) matches the pages' closed forms."""

import os
import re

import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
from all_reduce_reduction_rank_gb300 import build as arbuild
from oracle import model
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    arbuild.build()
    return ar.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "ar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ar_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(ar.EXPORTS) == names


def test_strerror_names_every_code(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert ar.ar_strerror(code) != "unknown error code"
    assert ar.ar_strerror(-99) == "unknown error code"


@pytest.mark.parametrize("P", [1, 4, 8, 119, 120, 121, 1 << 20, 3 * 120 + 7])
def test_packed_sizes_match_the_protocol_table(lib, P):
    # LL: 4 B data + 4 B flag per 8 B  ->  2P;  LL128: 120 + 8 per 128  ->  128 ceil(P/120)
    assert ar.ar_ll_bytes(P) == 2 * (-(-P // 4) * 4)
    assert ar.ar_ll128_bytes(P) == 128 * -(-P // 120)
    if P % 4 == 0:
        assert ar.ar_ll_bytes(P) == oracle.ll_bytes(P // 4)
        assert ar.ar_ll128_bytes(P) == oracle.ll128_bytes(P // 4)


E = {"f32": 4, "bf16": 2, "f16": 2}


@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("count", [0, 1, 1000, 1 << 20, 4099])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_plan_matches_closed_forms(lib, n, count, dtype):
    e = E[dtype]
    S = count * e
    t = ar.ar_plan(ar.AR_OP_ONE_SHOT, n, count, dtype)
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_one_shot(n, S))
    assert t.steps == model.steps_one_shot(n)
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == model.hbm_one_shot(n, count, e)
    assert t.launches == (1 if count else 0)
    t = ar.ar_plan(ar.AR_OP_TWO_SHOT, n, count, dtype)
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_two_shot(n, S))
    assert t.steps == model.steps_two_shot(n)
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == model.hbm_two_shot(n, count, e)
    t = ar.ar_plan(ar.AR_OP_RING, n, count, dtype)
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_ring(n, S))
    assert t.steps == model.steps_ring(n) and t.launches == (2 * (n - 1) if count else 0)
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == model.hbm_ring(n, count, e)


@pytest.mark.parametrize("count", [0, 1, 29, 30, 31, 262144])
def test_plan_ll_matches_closed_forms(lib, count):
    assert _rw(ar.ar_plan(ar.AR_OP_LL_PACK, 1, count, "f32")) == model.hbm_ll_pack(count)
    assert _rw(ar.ar_plan(ar.AR_OP_LL_UNPACK, 1, count, "f32")) == model.hbm_ll_unpack(count)
    assert _rw(ar.ar_plan(ar.AR_OP_LL_REDUCE, 8, count, "f32")) == model.hbm_ll_reduce(8, count)
    assert _rw(ar.ar_plan(ar.AR_OP_LL128_PACK, 1, count, "f32")) == model.hbm_ll128_pack(count)
    assert _rw(ar.ar_plan(ar.AR_OP_LL128_UNPACK, 1, count, "f32")) == model.hbm_ll128_unpack(count)
    assert _rw(ar.ar_plan(ar.AR_OP_LL128_REDUCE, 8, count, "f32")) == model.hbm_ll128_reduce(8, count)


def _rw(t):
    return t.hbm_read_bytes, t.hbm_write_bytes


@pytest.mark.parametrize("nb", [1, 8, 16])
def test_plan_batched_pack_scales_with_buffers(lib, nb):
    c = 1000
    for op, f in ((ar.AR_OP_LL_PACK, model.hbm_ll_pack), (ar.AR_OP_LL_UNPACK, model.hbm_ll_unpack),
                  (ar.AR_OP_LL128_PACK, model.hbm_ll128_pack), (ar.AR_OP_LL128_UNPACK, model.hbm_ll128_unpack)):
        rd, wr = f(c)
        assert _rw(ar.ar_plan(op, nb, c, "f32")) == (nb * rd, nb * wr)
    with pytest.raises(ar.ArError):
        ar.ar_plan(ar.AR_OP_LL_PACK, 0, c, "f32")


def test_plan_rejects_bad_arguments(lib):
    bad = [(0, 8), (ar.AR_OP_RING_ROUNDED_FUSED + 1, 8), (ar.AR_OP_ONE_SHOT, 1), (ar.AR_OP_RING, 17),
           (ar.AR_OP_ALLREDUCE_RMSNORM, 1)]
    for op, n in bad:
        with pytest.raises(ar.ArError):
            ar.ar_plan(op, n, 10, "f32")
    with pytest.raises(ar.ArError):
        ar.ar_plan(ar.AR_OP_ONE_SHOT, 8, 10, 7)


# --- argument checks, pointers compared but never dereferenced -------------

BASE = 1 << 40  # fake device addresses, 16-byte aligned, 1 MiB apart


def _bufs(n, stride=1 << 20, off=0):
    return [BASE + off + r * stride for r in range(n)]


def _check(op, n, ins, outs, count, dtype="bf16", max_bytes=1 << 20):
    return ar.ar_check_args(op, n, max_bytes, ins, outs, count, dtype)


OPS = [ar.AR_OP_ONE_SHOT, ar.AR_OP_TWO_SHOT, ar.AR_OP_RING]


@pytest.mark.parametrize("op", OPS)
def test_check_args(lib, op):
    n = 8
    ins, outs = _bufs(n), _bufs(n, off=64 << 20)
    assert _check(op, n, ins, outs, 1000) == ar.AR_OK
    assert _check(op, n, ins, ins, 1000) == ar.AR_OK                     # in place
    assert _check(op, n, [ins[0]] * n, outs, 1000) == ar.AR_OK           # inputs may alias
    assert _check(op, n, ins, outs, 0) == ar.AR_OK                       # empty
    assert _check(op, 1, ins, outs, 10) == ar.AR_ERR_INVALID
    assert _check(op, 17, ins + ins, outs + outs, 10) == ar.AR_ERR_INVALID
    assert _check(op, n, ins, outs, 10, dtype=3) == ar.AR_ERR_INVALID
    assert _check(op, n, None, outs, 10) == ar.AR_ERR_INVALID
    assert _check(op, n, ins[:-1] + [0], outs, 10) == ar.AR_ERR_INVALID
    assert _check(op, n, ins, outs, (1 << 19) + 1) == ar.AR_ERR_TOO_LARGE  # bf16: 2 B each
    assert _check(op, n, ins, outs, 1 << 19) == ar.AR_OK                   # exactly max_bytes
    assert _check(op, n, ins, outs, 1 << 62) == ar.AR_ERR_TOO_LARGE
    assert _check(op, n, [ins[0] + 8] + ins[1:], outs, 10) == ar.AR_ERR_ALIGN
    assert _check(op, n, ins, outs[:3] + [outs[3] + 4] + outs[4:], 10) == ar.AR_ERR_ALIGN
    # overlaps: two outputs, an output with another rank's input, a shifted in-place
    over = outs[:]
    over[2] = outs[1] + 16
    assert _check(op, n, ins, over, 1000) == ar.AR_ERR_INVALID
    cross = outs[:]
    cross[5] = ins[6]
    assert _check(op, n, ins, cross, 1000) == ar.AR_ERR_INVALID
    shifted = [i + 16 for i in ins]
    assert _check(op, n, ins, shifted, 1000) == ar.AR_ERR_INVALID
    assert _check(op, n, ins, shifted, 8) == ar.AR_OK                     # 16 B apart, 16 B long


def test_check_args_ll(lib):
    n = 8
    ins, outs = _bufs(n), _bufs(n, off=64 << 20)
    for op in (ar.AR_OP_LL_REDUCE, ar.AR_OP_LL128_REDUCE):
        assert _check(op, n, ins, outs, 1000, dtype="f32") == ar.AR_OK
        assert _check(op, n, ins, outs, 1000, dtype="bf16") == ar.AR_ERR_INVALID
    # LL lines are twice the payload: 1000 words -> 8000 B, so 4 KiB apart overlaps
    close = [BASE + r * 4096 for r in range(n)]
    assert _check(ar.AR_OP_LL_REDUCE, n, ins, close, 1000, dtype="f32") == ar.AR_ERR_INVALID
    assert _check(ar.AR_OP_LL_REDUCE, n, ins, close, 500, dtype="f32") == ar.AR_OK


def test_check_args_batched_pack(lib):
    n, c = 8, 1000                      # payload 4000 B, LL lines 8000 B, LL128 lines 4352 B
    src = _bufs(n)
    dst = _bufs(n, off=64 << 20)
    for op in (ar.AR_OP_LL_PACK, ar.AR_OP_LL128_PACK, ar.AR_OP_LL_UNPACK, ar.AR_OP_LL128_UNPACK):
        assert _check(op, n, src, dst, c, dtype="f32") == ar.AR_OK
        assert _check(op, 1, src[:1], dst[:1], c, dtype="f32") == ar.AR_OK
        assert _check(op, n, [src[0]] * n, dst, c, dtype="f32") == ar.AR_OK     # sources may alias
        assert _check(op, n, src, dst, c, dtype="bf16") == ar.AR_ERR_INVALID
        assert _check(op, 0, src, dst, c, dtype="f32") == ar.AR_ERR_INVALID
        assert _check(op, n, src, [dst[0]] * n, c, dtype="f32") == ar.AR_ERR_INVALID   # destinations alias
        assert _check(op, n, src, dst[:7] + [src[3]], c, dtype="f32") == ar.AR_ERR_INVALID
        assert _check(op, n, src, dst[:7] + [dst[7] + 8], c, dtype="f32") == ar.AR_ERR_ALIGN
        assert _check(op, n, src, dst, (1 << 18) + 1, dtype="f32") == ar.AR_ERR_TOO_LARGE
    # LL lines are twice the payload: destinations 4 KiB apart overlap at 1000 words
    close = [BASE + (64 << 20) + r * 4096 for r in range(n)]
    assert _check(ar.AR_OP_LL_PACK, n, src, close, c, dtype="f32") == ar.AR_ERR_INVALID
    assert _check(ar.AR_OP_LL_UNPACK, n, src, close, c, dtype="f32") == ar.AR_OK  # unpack writes 4000 B


def test_calls_reject_a_null_handle(lib):
    p = _bufs(8)
    assert ar.ar_one_shot(0, p, p, 10, "bf16") == ar.AR_ERR_INVALID
    assert ar.ar_two_shot(0, p, p, 10, "bf16") == ar.AR_ERR_INVALID
    assert ar.ar_ring(0, p, p, 10, "bf16") == ar.AR_ERR_INVALID
    assert ar.ar_ll_pack(0, p[0], p[1], 10, 1) == ar.AR_ERR_INVALID
    assert ar.ar_ll128_reduce(0, p, p, 10, 1) == ar.AR_ERR_INVALID
    assert ar.ar_destroy(0) == ar.AR_ERR_INVALID
    assert ar.ar_status(0) == ar.AR_ERR_INVALID
    assert ar.ar_set_option(0, ar.AR_OPT_SPIN_NS, 10) == ar.AR_ERR_INVALID
    with pytest.raises(ar.ArError):
        ar.ar_traffic(0)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_a_device_fails_cleanly(lib):
    with pytest.raises(ar.ArError) as e:
        ar.ar_create(8, 1 << 20)
    assert e.value.code == ar.AR_ERR_CUDA
    with pytest.raises(ar.ArError) as e:
        ar.ar_create(1, 1 << 20)
    assert e.value.code == ar.AR_ERR_INVALID


# --- size-based selection ------------------------------------------------------

def test_select_model_matches_the_printed_alpha_beta_table(lib):
    # the fastest of ring / one-shot / two-shot in each printed row of the
    # NCCL chapter's alpha-beta table (n = 8, beta = 450e9, alpha = 1.5e-6)
    path = os.path.join(ROOT, "tests", "golden", "alpha_beta_table.txt")
    rows = [ln.split() for ln in open(path) if ln.startswith("row ")]
    assert len(rows) == 5
    name_of = {ar.AR_OP_ONE_SHOT: "one-shot", ar.AR_OP_TWO_SHOT: "two-shot", ar.AR_OP_RING: "ring"}
    for r in rows:
        S = int(r[1])
        printed = {"ring": float(r[2]), "one-shot": float(r[4]), "two-shot": float(r[5])}
        want = min(printed, key=printed.get)
        got = ar.ar_select(ar.AR_AUTO_MODEL, 8, S, 1.5e-6, 450e9, 0)
        assert name_of[got] == want, (S, name_of[got], printed)
        assert want == r[7]          # the page's own "fastest without NVLS" column


def test_select_model_crossover_and_handoff(lib):
    # S* = 2 alpha beta / ((n-1)(1-2/n)) = 257142.86 B at n = 8 (exercise 2)
    assert ar.ar_select(ar.AR_AUTO_MODEL, 8, 257142, 1.5e-6, 450e9, 0) == ar.AR_OP_ONE_SHOT
    assert ar.ar_select(ar.AR_AUTO_MODEL, 8, 257143, 1.5e-6, 450e9, 0) == ar.AR_OP_TWO_SHOT
    # no crossover at n = 2: one-shot at every size
    for S in (1, 1 << 20, 1 << 30):
        assert ar.ar_select(ar.AR_AUTO_MODEL, 2, S, 1.5e-6, 450e9, 0) == ar.AR_OP_ONE_SHOT
    # above the pre-registered size the ring takes over
    assert ar.ar_select(ar.AR_AUTO_MODEL, 8, 8 << 20, 1.5e-6, 450e9, 8 << 20) == ar.AR_OP_TWO_SHOT
    assert ar.ar_select(ar.AR_AUTO_MODEL, 8, (8 << 20) + 1, 1.5e-6, 450e9, 8 << 20) == ar.AR_OP_RING
    # the emulated policy: one-shot always
    for n in (2, 8, 16):
        assert ar.ar_select(ar.AR_AUTO_EMULATED, n, 1 << 28, 0.0, 1.0, 0) == ar.AR_OP_ONE_SHOT
    assert ar.ar_select(ar.AR_AUTO_MODEL, 1, 10, 1e-6, 1e9, 0) == ar.AR_ERR_INVALID
    assert ar.ar_select(7, 8, 10, 1e-6, 1e9, 0) == ar.AR_ERR_INVALID
    assert ar.ar_select(ar.AR_AUTO_MODEL, 8, 10, 1e-6, 0.0, 0) == ar.AR_ERR_INVALID


@pytest.mark.parametrize("n", [3, 4, 8, 16])
def test_select_model_crossover_formula(lib, n):
    from oracle import model
    a, b = 1.5e-6, 450e9
    s_star = model.one_two_shot_crossover(n, b, a)
    if s_star is None:
        return
    below, above = int(s_star * 0.999), int(s_star * 1.001) + 1
    assert ar.ar_select(ar.AR_AUTO_MODEL, n, below, a, b, 0) == ar.AR_OP_ONE_SHOT
    assert ar.ar_select(ar.AR_AUTO_MODEL, n, above, a, b, 0) in (ar.AR_OP_TWO_SHOT, ar.AR_OP_RING)


@pytest.mark.parametrize("n", [2, 8, 16])
def test_plan_fused_epilogue(lib, n):
    # reads n S of partial sums and S of residual, writes n normalized outputs and the residual
    t = ar.ar_plan(ar.AR_OP_ALLREDUCE_RMSNORM, n, 64 * 8192, "bf16")
    S = 64 * 8192 * 2
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == ((n + 1) * S, (n + 1) * S)
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_one_shot(n, S)) and t.launches == 1


@pytest.mark.parametrize("n", [2, 8, 16])
def test_plan_push_and_copyin(lib, n):
    N = 4099
    S = N * 2
    t = ar.ar_plan(ar.AR_OP_ONE_SHOT_PUSH, n, N, "bf16")
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == (n * S + n * n * S, n * (n - 1) * S + n * S)
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_one_shot(n, S)) and t.launches == 2
    t = ar.ar_plan(ar.AR_OP_ONE_SHOT_COPYIN, n, N, "bf16")
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == (2 * n * S, 2 * n * S)
    ins, outs = _bufs(n), _bufs(n, off=64 << 20)
    for op in (ar.AR_OP_ONE_SHOT_PUSH, ar.AR_OP_ONE_SHOT_COPYIN):
        assert _check(op, n, ins, outs, 1000) == ar.AR_OK
        assert _check(op, n, ins, outs[:1] + [ins[0]] + outs[2:], 1000) == ar.AR_ERR_INVALID  # another rank's input


@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("N", [1, 4099, 1 << 20])
def test_plan_ring_rounded(lib, n, N):
    t = ar.ar_plan(ar.AR_OP_RING_ROUNDED, n, N, "bf16")
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == model.hbm_ring_rounded(n, N, 2)
    assert t.steps == 2 * (n - 1) and t.link_bytes_per_rank == pytest.approx(model.link_bytes_ring(n, 2 * N))


@pytest.mark.parametrize("n", [2, 4, 8, 16])
@pytest.mark.parametrize("N", [0, 1, 4099, 1 << 20])
def test_plan_tree(lib, n, N):
    t = ar.ar_plan(ar.AR_OP_TREE, n, N, "f16")
    levels = {2: 1, 4: 2, 8: 3, 16: 4}[n]
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == model.hbm_tree(n, N, 2)
    assert t.steps == levels and t.launches == (levels if N else 0)
    assert t.link_bytes_per_rank == pytest.approx(levels * 2 * N)


@pytest.mark.parametrize("n", [3, 5, 6, 12, 15])
def test_tree_refuses_other_rank_counts(lib, n):
    with pytest.raises(ar.ArError):
        ar.ar_plan(ar.AR_OP_TREE, n, 100, "bf16")
    ins, outs = _bufs(n), _bufs(n, off=64 << 20)
    assert _check(ar.AR_OP_TREE, n, ins, outs, 1000) == ar.AR_ERR_INVALID
    assert _check(ar.AR_OP_TREE, 8, _bufs(8), _bufs(8, off=64 << 20), 1000) == ar.AR_OK


@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("N", [0, 1, 959, 4099, 1 << 20])
def test_plan_ring_persistent(lib, n, N):
    # per step the n chunks move once as LL128 lines of 30 words; the ranks'
    # own elements are read in n steps and their outputs written in n steps
    t = ar.ar_plan(ar.AR_OP_RING_PERSISTENT, n, N, "bf16")
    C = -(-N // n)
    C = -(-C // 8) * 8
    lines = sum(-(-max(0, min(C, N - c * C)) // 30) for c in range(n))
    want = n * 2 * N + (2 * n - 2) * 128 * lines
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == (want, want)
    assert t.steps == 2 * (n - 1) and t.launches == (1 if N else 0)
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_ring(n, 2 * N))
    ins, outs = _bufs(n), _bufs(n, off=64 << 20)
    assert _check(ar.AR_OP_RING_PERSISTENT, n, ins, outs, 1000) == ar.AR_OK


@pytest.mark.parametrize("n", [2, 3, 8, 16])
def test_plan_ring_cluster(lib, n):
    N = 4099
    t = ar.ar_plan(ar.AR_OP_RING_CLUSTER, n, N, "bf16")
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == (n * 2 * N, n * 2 * N)
    assert t.steps == 2 * (n - 1) and t.launches == 1
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_ring(n, 2 * N))


@pytest.mark.parametrize("n", [2, 4, 8, 16])
def test_plan_tree_fused(lib, n):
    N = 4099
    t = ar.ar_plan(ar.AR_OP_TREE_FUSED, n, N, "bf16")
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == (n * 2 * N, n * 2 * N)
    assert t.steps == n.bit_length() - 1 and t.launches == 1
    with pytest.raises(ar.ArError):
        ar.ar_plan(ar.AR_OP_TREE_FUSED, 6, N, "bf16")


@pytest.mark.parametrize("op", ["AR_OP_RING_FUSED", "AR_OP_RING_ROUNDED_FUSED"])
@pytest.mark.parametrize("n", [2, 3, 8, 16])
def test_plan_ring_fused(lib, op, n):
    N = 4099
    t = ar.ar_plan(getattr(ar, op), n, N, "bf16")
    assert (t.hbm_read_bytes, t.hbm_write_bytes) == (n * 2 * N, n * 2 * N)
    assert t.steps == 2 * (n - 1) and t.launches == 1
    assert t.link_bytes_per_rank == pytest.approx(model.link_bytes_ring(n, 2 * N))
    assert ar.ar_plan(getattr(ar, op), n, 0, "bf16").launches == 0
    ins, outs = _bufs(n), _bufs(n, off=64 << 20)
    assert _check(getattr(ar, op), n, ins, outs, 1000) == ar.AR_OK
    assert _check(getattr(ar, op), n, ins, ins, 1000) == ar.AR_OK   # in place
    outs[1] = outs[0]
    assert _check(getattr(ar, op), n, ins, outs, 1000) == ar.AR_ERR_INVALID


def _header_constants():
    text = open(os.path.join(ROOT, "include", "ar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return {k: int(v) for k, v in re.findall(r"\b(AR_[A-Z0-9_]+)\s*=\s*(-?\d+)", text)}


def test_binding_constants_match_the_header():
    # every enum value of include/ar.h has the same value in the Python binding, and
    # every kernel id its name in ar.KERNELS (what ar_timing reports)
    consts = _header_constants()
    assert len(consts) >= 60
    kernels = {v: k[len("AR_K_"):].lower() for k, v in consts.items() if k.startswith("AR_K_")}
    assert kernels == ar.KERNELS
    for name, value in consts.items():
        if name.startswith("AR_K_"):
            continue
        assert getattr(ar, name) == value, name
    assert ar.DTYPES == {"f32": consts["AR_F32"], "bf16": consts["AR_BF16"], "f16": consts["AR_F16"]}
