"""Pins for the oracle's LL and LL128 lines.

Handbook chapter "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce",
§协议 table: LL carries 4 B of data and a 4 B flag in every 8 B (so a payload
of P bytes takes 2P); LL128 carries 120 B of data and an 8 B flag in every
128 B (so P bytes take 128 ceil(P/120)).  The receiver knows the data is
there when it sees the flag.  Byte positions inside a line are the reading
stated in the oracle's header; they are decoded here with ``struct``,
independently of the oracle's byte handling.
"""

import struct

import numpy as np
import pytest

import oracle
import workloads

COUNTS = [1, 2, 3, 29, 30, 31, 59, 60, 61, 1000, 4099]


@pytest.mark.parametrize("count", COUNTS)
def test_packed_sizes(count):
    P = 4 * count
    assert oracle.ll_bytes(count) == 2 * P
    assert oracle.ll128_bytes(count) == 128 * -(-P // 120)
    assert oracle.ll128_lines(count) == -(-P // 120)


def _bits_payload(count, seed):
    """Arbitrary 32-bit words, NaN and infinity patterns included."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 32, size=count, dtype=np.uint64).astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("count", COUNTS)
def test_ll_layout_and_roundtrip(count):
    src = _bits_payload(count, count)
    step = 0xA5A50000 + count
    lines = oracle.ll_pack(src, step)
    raw = lines.tobytes()
    for i in range(count):
        data, flag = struct.unpack_from("<II", raw, 8 * i)
        assert data == int(src.view(np.uint32)[i]) and flag == step
    dst, bad = oracle.ll_unpack(lines, count, step)
    assert bad == 0
    np.testing.assert_array_equal(dst.view(np.uint32), src.view(np.uint32))


@pytest.mark.parametrize("count", COUNTS)
def test_ll128_layout_and_roundtrip(count):
    src = _bits_payload(count, 1000 + count)
    step = 0x0123456789ABCDEF
    lines = oracle.ll128_pack(src, step)
    raw = lines.tobytes()
    words = src.view(np.uint32)
    for k in range(oracle.ll128_lines(count)):
        vals = struct.unpack_from("<30IQ", raw, 128 * k)
        for j in range(30):
            idx = 30 * k + j
            assert vals[j] == (int(words[idx]) if idx < count else 0)
        assert vals[30] == step
    dst, bad = oracle.ll128_unpack(lines, count, step)
    assert bad == 0
    np.testing.assert_array_equal(dst.view(np.uint32), words)


def test_unpack_rejects_wrong_step_and_leaves_dst():
    count = 100
    src = workloads.payload_f32(1, count, seed=1)[0]
    marker = np.full(count, 7.0, np.float32)
    dst, bad = oracle.ll_unpack(oracle.ll_pack(src, 5), count, 6, marker.copy())
    assert bad == count and np.all(dst == 7.0)
    dst, bad = oracle.ll128_unpack(oracle.ll128_pack(src, 5), count, 6, marker.copy())
    assert bad == oracle.ll128_lines(count) and np.all(dst == 7.0)


def test_single_corrupted_flag_is_the_only_line_lost():
    count = 90
    src = workloads.payload_f32(1, count, seed=2)[0]
    lines = oracle.ll_pack(src, 9)
    lines[8 * 17 + 4] ^= 1                      # flag of line 17
    dst, bad = oracle.ll_unpack(lines, count, 9, np.full(count, -3.0, np.float32))
    assert bad == 1 and dst[17] == -3.0
    keep = np.arange(count) != 17
    np.testing.assert_array_equal(dst[keep], src[keep])
    l128 = oracle.ll128_pack(src, 9)
    l128[128 * 1 + 127] ^= 0x80                 # flag of line 1 (elements 30..59)
    dst, bad = oracle.ll128_unpack(l128, count, 9, np.full(count, -3.0, np.float32))
    assert bad == 1 and np.all(dst[30:60] == -3.0)
    np.testing.assert_array_equal(dst[:30], src[:30])
    np.testing.assert_array_equal(dst[60:], src[60:])


@pytest.mark.parametrize("n", [2, 8, 16])
@pytest.mark.parametrize("count", [1, 31, 4099])
def test_flag_checked_reduce_is_the_sum(n, count):
    xs = workloads.payload_f32(n, count, seed=n * count)
    step = 3
    want = oracle.all_reduce(xs, "f32")[0]
    out, bad = oracle.ll_reduce([oracle.ll_pack(x, step) for x in xs], count, step)
    assert bad == 0
    for o in out:
        dst, b = oracle.ll_unpack(o, count, step)
        assert b == 0
        np.testing.assert_array_equal(dst, want)
    out, bad = oracle.ll128_reduce([oracle.ll128_pack(x, step) for x in xs], count, step)
    assert bad == 0
    for o in out:
        dst, b = oracle.ll128_unpack(o, count, step)
        assert b == 0
        np.testing.assert_array_equal(dst, want)
        # padding sums to zero and the flag is the step
        raw = o.tobytes()
        last = oracle.ll128_lines(count) - 1
        vals = struct.unpack_from("<30IQ", raw, 128 * last)
        used = count - 30 * last
        assert all(v == 0 for v in vals[used:30]) and vals[30] == step


def test_reduce_with_a_stale_rank_consumes_nothing():
    n, count, step = 8, 200, 12
    xs = workloads.payload_f32(n, count, seed=44)
    packed = [oracle.ll_pack(x, step) for x in xs]
    packed[5] = oracle.ll_pack(xs[5], step - 1)     # rank 5 still holds the last step
    before = [np.full_like(packed[0], 0xEE) for _ in range(n)]
    out, bad = oracle.ll_reduce(packed, count, step, [b.copy() for b in before])
    assert bad == count
    for o, b in zip(out, before):
        np.testing.assert_array_equal(o, b)
    p128 = [oracle.ll128_pack(x, step) for x in xs]
    p128[0] = oracle.ll128_pack(xs[0], step + 1)
    before = [np.full_like(p128[0], 0xEE) for _ in range(n)]
    out, bad = oracle.ll128_reduce(p128, count, step, [b.copy() for b in before])
    assert bad == oracle.ll128_lines(count)
    for o, b in zip(out, before):
        np.testing.assert_array_equal(o, b)
