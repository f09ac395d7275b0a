"""Parity of the LL / LL128 calls against the CPU oracle (bit-exact: they
move bits and add in rank order), and their bounded flag waits.

Fault tests make a wait run out on purpose the way the protocol allows: a
line whose flag nothing will set (a stale step id, one corrupted flag).  The
consumer re-reads it for a short, bounded time (AR_OPT_SPIN_NS), leaves it
unconsumed and reports AR_ERR_FLAG_TIMEOUT through ar_status; nothing traps
or hangs."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Buf, Handle, ptrs

pytestmark = pytest.mark.gpu

CFG = workloads.CONFIGS[4]


def _pack_all(h, xs, step, kind):
    pack = ar.ar_ll_pack if kind == "ll" else ar.ar_ll128_pack
    nbytes = oracle.ll_bytes if kind == "ll" else oracle.ll128_bytes
    srcs = [Buf(x.nbytes).upload(x) for x in xs]
    lines = [Buf(nbytes(x.size)).fill(0) for x in xs]
    for s, l, x in zip(srcs, lines, xs):
        assert pack(h, s.ptr, l.ptr, x.size, step) == ar.AR_OK
    return srcs, lines


@pytest.mark.parametrize("kind", ["ll", "ll128"])
@pytest.mark.parametrize("count", CFG["counts"] + [3, 29, 31, 61, 4099, 300_007])
def test_pipeline_pack_reduce_unpack(kind, count):
    n = CFG["n"]
    xs = workloads.payload_f32(n, count, seed=workloads.seed_of(4) + count)
    o_pack = oracle.ll_pack if kind == "ll" else oracle.ll128_pack
    o_reduce = oracle.ll_reduce if kind == "ll" else oracle.ll128_reduce
    o_unpack = oracle.ll_unpack if kind == "ll" else oracle.ll128_unpack
    reduce = ar.ar_ll_reduce if kind == "ll" else ar.ar_ll128_reduce
    unpack = ar.ar_ll_unpack if kind == "ll" else ar.ar_ll128_unpack
    with Handle(n, max(16, 4 * count)) as h:               # a handle holds at least 16 B
        for step in (1, 2, 3):                                  # a fresh step id each pass
            srcs, lines = _pack_all(h, xs, step, kind)
            outs = [Buf(l.nbytes).fill(0) for l in lines]
            assert reduce(h, ptrs(lines), ptrs(outs), count, step) == ar.AR_OK
            dsts = [Buf(4 * count).fill(0) for _ in range(n)]
            for o, d in zip(outs, dsts):
                assert unpack(h, o.ptr, d.ptr, count, step) == ar.AR_OK
            assert ar.ar_status(h) == ar.AR_OK
            packed = [o_pack(x, step) for x in xs]
            for l, p in zip(lines, packed):
                np.testing.assert_array_equal(l.download(np.uint8), p)
            want_lines, bad = o_reduce(packed, count, step)
            assert bad == 0
            for o, w in zip(outs, want_lines):
                np.testing.assert_array_equal(o.download(np.uint8), w)
            want = oracle.all_reduce(xs, "f32")[0]
            for d in dsts:
                np.testing.assert_array_equal(d.download(np.uint32), want.view(np.uint32))
            for b in srcs + lines + outs + dsts:
                assert b.guards_intact()


@pytest.mark.parametrize("kind", ["ll", "ll128"])
def test_reduce_in_place(kind):
    n, count, step = 8, 10_001, 7
    xs = workloads.payload_f32(n, count, seed=3)
    with Handle(n, 4 * count) as h:
        _, lines = _pack_all(h, xs, step, kind)
        reduce = ar.ar_ll_reduce if kind == "ll" else ar.ar_ll128_reduce
        assert reduce(h, ptrs(lines), ptrs(lines), count, step) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
        o_pack = oracle.ll_pack if kind == "ll" else oracle.ll128_pack
        o_reduce = oracle.ll_reduce if kind == "ll" else oracle.ll128_reduce
        want, _ = o_reduce([o_pack(x, step) for x in xs], count, step)
        for l, w in zip(lines, want):
            np.testing.assert_array_equal(l.download(np.uint8), w)


def test_step_zero_and_bad_arguments_are_rejected():
    with Handle(8, 4096) as h:
        a, b = Buf(4096), Buf(8192)
        assert ar.ar_ll_pack(h, a.ptr, b.ptr, 16, 0) == ar.AR_ERR_INVALID
        assert ar.ar_ll128_unpack(h, b.ptr, a.ptr, 16, 0) == ar.AR_ERR_INVALID
        assert ar.ar_ll_pack(h, a.ptr + 4, b.ptr, 16, 1) == ar.AR_ERR_ALIGN
        assert ar.ar_ll_pack(h, a.ptr, b.ptr, 1025, 1) == ar.AR_ERR_TOO_LARGE
        assert ar.ar_ll_pack(h, a.ptr, a.ptr + 16, 16, 1) == ar.AR_ERR_INVALID   # overlap


@pytest.mark.parametrize("kind", ["ll", "ll128"])
def test_stale_rank_times_out_and_consumes_nothing(kind):
    n, count, step = 8, 3001, 5
    xs = workloads.payload_f32(n, count, seed=44)
    reduce = ar.ar_ll_reduce if kind == "ll" else ar.ar_ll128_reduce
    with Handle(n, 4 * count, spin_ns=200_000) as h:
        _, lines = _pack_all(h, xs, step, kind)
        # rank 5 still holds the previous step's lines: nothing will ever set its flags
        pack = ar.ar_ll_pack if kind == "ll" else ar.ar_ll128_pack
        src5 = Buf(xs[5].nbytes).upload(xs[5])
        assert pack(h, src5.ptr, lines[5].ptr, count, step - 1) == ar.AR_OK
        outs = [Buf(l.nbytes).fill(0xEE) for l in lines]
        assert reduce(h, ptrs(lines), ptrs(outs), count, step) == ar.AR_OK   # the launch itself is fine
        rc, info = ar.ar_status_info(h)
        assert rc == ar.AR_ERR_FLAG_TIMEOUT and info.code == ar.AR_ERR_FLAG_TIMEOUT
        assert info.rank == 5
        n_lines = count if kind == "ll" else oracle.ll128_lines(count)
        assert info.lines_skipped == n_lines
        for o in outs:
            assert bool((o.body() == 0xEE).all())
        assert ar.ar_status(h) == ar.AR_OK                   # cleared; the context still works
        assert pack(h, src5.ptr, lines[5].ptr, count, step) == ar.AR_OK
        assert reduce(h, ptrs(lines), ptrs(outs), count, step) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK


@pytest.mark.parametrize("kind", ["ll", "ll128"])
def test_one_corrupted_flag_loses_one_line(kind):
    count, step = 901, 9
    x = workloads.payload_f32(1, count, seed=2)[0]
    with Handle(2, 4 * count, spin_ns=100_000) as h:
        _, (lines,) = _pack_all(h, [x], step, kind)
        if kind == "ll":
            bad_line, flag_off, lo, hi = 17, 8 * 17 + 4, 17, 18
        else:
            bad_line, flag_off, lo, hi = 1, 128 * 1 + 120, 30, 60
        lines.body()[flag_off] ^= 1
        dst = Buf(4 * count).upload(np.full(count, -3.0, np.float32))
        unpack = ar.ar_ll_unpack if kind == "ll" else ar.ar_ll128_unpack
        assert unpack(h, lines.ptr, dst.ptr, count, step) == ar.AR_OK
        rc, info = ar.ar_status_info(h)
        assert rc == ar.AR_ERR_FLAG_TIMEOUT and info.line == bad_line and info.lines_skipped == 1
        got = dst.download(np.float32)
        assert np.all(got[lo:hi] == -3.0)
        keep = np.ones(count, bool)
        keep[lo:hi] = False
        np.testing.assert_array_equal(got[keep].view(np.uint32), x[keep].view(np.uint32))


def test_spin_option_bounds():
    with Handle(2, 64) as h:
        assert ar.ar_set_option(h, ar.AR_OPT_SPIN_NS, 0) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_SPIN_NS, 10**10 + 1) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_CTAS_PER_SM, 1025) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_TIMING_PAUSE, 1) == ar.AR_ERR_INVALID   # timing is off
        assert ar.ar_set_option(h, 99, 1) == ar.AR_ERR_INVALID


@pytest.mark.parametrize("kind", ["ll", "ll128"])
@pytest.mark.parametrize("n,count", [(8, 262144), (8, 61), (16, 4099), (2, 1)])
def test_batched_pack_and_unpack_equal_the_oracle(kind, n, count):
    xs = workloads.payload_f32(n, count, seed=n * 31 + count)
    o_pack = oracle.ll_pack if kind == "ll" else oracle.ll128_pack
    nbytes = oracle.ll_bytes(count) if kind == "ll" else oracle.ll128_bytes(count)
    pack_n = ar.ar_ll_pack_n if kind == "ll" else ar.ar_ll128_pack_n
    unpack_n = ar.ar_ll_unpack_n if kind == "ll" else ar.ar_ll128_unpack_n
    reduce = ar.ar_ll_reduce if kind == "ll" else ar.ar_ll128_reduce
    step = 21
    with Handle(n, max(16, 4 * count)) as h:
        srcs = [Buf(x.nbytes).upload(x) for x in xs]
        lines = [Buf(nbytes).fill(0) for _ in range(n)]
        red = [Buf(nbytes).fill(0) for _ in range(n)]
        dsts = [Buf(4 * count).fill(0) for _ in range(n)]
        assert pack_n(h, ptrs(srcs), ptrs(lines), count, step) == ar.AR_OK
        assert ar.ar_traffic(h).launches == 1
        assert reduce(h, ptrs(lines), ptrs(red), count, step) == ar.AR_OK
        assert unpack_n(h, ptrs(red), ptrs(dsts), count, step) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
        for l, x in zip(lines, xs):
            np.testing.assert_array_equal(l.download(np.uint8), o_pack(x, step))
        want = oracle.all_reduce(xs, "f32")[0]
        for d in dsts:
            np.testing.assert_array_equal(d.download(np.uint32), want.view(np.uint32))
        for b in srcs + lines + red + dsts:
            assert b.guards_intact()


def test_batched_unpack_reports_the_rank_of_a_stale_buffer():
    n, count, step = 4, 1000, 3
    xs = workloads.payload_f32(n, count, seed=8)
    with Handle(n, 4 * count, spin_ns=100_000) as h:
        srcs = [Buf(x.nbytes).upload(x) for x in xs]
        lines = [Buf(oracle.ll_bytes(count)).fill(0) for _ in range(n)]
        assert ar.ar_ll_pack_n(h, ptrs(srcs), ptrs(lines), count, step) == ar.AR_OK
        assert ar.ar_ll_pack(h, srcs[2].ptr, lines[2].ptr, count, step + 1) == ar.AR_OK   # rank 2 runs ahead
        dsts = [Buf(4 * count).fill(0x7F) for _ in range(n)]
        assert ar.ar_ll_unpack_n(h, ptrs(lines), ptrs(dsts), count, step) == ar.AR_OK
        rc, info = ar.ar_status_info(h)
        assert rc == ar.AR_ERR_FLAG_TIMEOUT and info.rank == 2 and info.lines_skipped == count
        assert bool((dsts[2].body() == 0x7F).all())
        for r in (0, 1, 3):
            np.testing.assert_array_equal(dsts[r].download(np.uint32), xs[r].view(np.uint32))
