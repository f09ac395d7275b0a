"""Pins for the oracle's one-shot sum and its reduce-scatter / all-gather.

What fixes the result, none of it the oracle's own code:
- integer-valued inputs make every summation order exact, so the result is
  the integer sum (numpy int64);
- the NCCL example program's check ("多 GPU 与 NCCL", §NCCL 编程): rank g
  holds g + i % 7, so every rank must end with n(n-1)/2 + n (i % 7);
- for n = 2 the method is one binary32 add followed by one rounding to the
  payload type: numpy's float32 add and torch's / numpy's casts;
- the exact sum (math.fsum) within the accumulation error bound;
- all-reduce = reduce-scatter + all-gather ("多 GPU 与 NCCL", §集合通信).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads

DTYPES = ["f32", "bf16", "f16"]


def widen(a, dtype):
    return oracle.to_f32(a, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("N", [1, 7, 1024, 4099])
def test_integer_inputs_sum_exactly(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "int8", seed=n * 100 + N)
    out = oracle.all_reduce(xs, dtype)
    exact = sum(widen(x, dtype).astype(np.int64) for x in xs)
    for o in out:
        np.testing.assert_array_equal(widen(o, dtype).astype(np.int64), exact)
        np.testing.assert_array_equal(o, out[0])


@pytest.mark.parametrize("n", range(2, 17))
def test_nccl_example_fill_pattern(n):
    N = 7 * 37 + 3
    xs = workloads.rank_inputs(n, N, "f32", "fill7", seed=0)
    i = np.arange(N)
    want = np.float32(n * (n - 1) / 2) + np.float32(n) * (i % 7).astype(np.float32)
    out = oracle.all_reduce(xs, "f32")
    assert sum(int(np.count_nonzero(o != want)) for o in out) == 0
    # the same pattern in bf16 stays exact while |sum| <= 256 (n <= 16 gives <= 216)
    xb = [oracle.f32_to_bf16(x) for x in xs]
    ob = oracle.all_reduce(xb, "bf16")
    assert all(np.array_equal(widen(o, "bf16"), want) for o in ob)


def _stratified_bf16(count, rng):
    """bf16 patterns spread over every exponent, both signs, zeros, subnormals."""
    h = rng.integers(0, 1 << 16, size=count).astype(np.uint16)
    f = oracle.bf16_to_f32(h)
    return h[np.isfinite(f)]


def test_brute_force_n2_bf16_all_a():
    rng = np.random.default_rng(5)
    a_all = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    a_all = a_all[np.isfinite(oracle.bf16_to_f32(a_all))]
    b_set = _stratified_bf16(640, rng)[:512]
    a = np.repeat(a_all, b_set.size)
    b = np.tile(b_set, a_all.size)
    got = oracle.all_reduce([a, b], "bf16")
    # one binary32 add (numpy) then one round-to-nearest-even to bf16 (torch);
    # sums beyond the binary32 range overflow to +-Inf on both sides
    with np.errstate(over="ignore"):
        s = oracle.bf16_to_f32(a) + oracle.bf16_to_f32(b)
    ref = torch.from_numpy(s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    gf, rf = oracle.bf16_to_f32(got[0]), oracle.bf16_to_f32(ref)
    same = (got[0] == ref) | (np.isnan(gf) & np.isnan(rf))
    assert same.all()
    np.testing.assert_array_equal(got[1], got[0])


def test_brute_force_n2_f16():
    rng = np.random.default_rng(6)
    a_all = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    a_all = a_all[np.isfinite(a_all.view(np.float16))]
    b_set = rng.choice(a_all, size=256, replace=False)
    a = np.repeat(a_all, b_set.size)
    b = np.tile(b_set, a_all.size)
    got = oracle.all_reduce([a, b], "f16")[0]
    with np.errstate(over="ignore"):
        s = a.view(np.float16).astype(np.float32) + b.view(np.float16).astype(np.float32)
        ref = s.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_n2_f32_is_one_binary32_add():
    rng = np.random.default_rng(8)
    bits = rng.integers(0, 1 << 32, size=(2, 1 << 18), dtype=np.uint64).astype(np.uint32)
    a, b = bits[0].view(np.float32), bits[1].view(np.float32)
    keep = np.isfinite(a) & np.isfinite(b)
    a, b = np.ascontiguousarray(a[keep]), np.ascontiguousarray(b[keep])
    with np.errstate(over="ignore", invalid="ignore"):
        ref = a + b
    got = oracle.all_reduce([a, b], "f32")[0]
    nan = np.isnan(got) & np.isnan(ref)
    assert np.all((got.view(np.uint32) == ref.view(np.uint32)) | nan)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [4, 8, 16])
def test_within_accumulation_bound_of_exact_sum(dtype, n):
    N = 20000
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=99 + n)
    out = widen(oracle.all_reduce(xs, dtype)[0], dtype).astype(np.float64)
    cols = np.stack([widen(x, dtype).astype(np.float64) for x in xs])
    exact = np.array([math.fsum(cols[:, i]) for i in range(N)])
    abs_sum = np.abs(cols).sum(axis=0)
    # n fp32 adds (each <= 2^-24 relative to the running |sum| <= sum|x|), then
    # one rounding to the payload type (half an ulp of the result).
    ulp_bits = {"f32": 24, "bf16": 8, "f16": 11}[dtype]
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(out), 2.0**-126))) - ulp_bits)
    if dtype == "f16":
        half_ulp = np.maximum(half_ulp, 2.0**-25)
    bound = half_ulp + n * 2.0**-24 * abs_sum
    assert np.all(np.abs(out - exact) <= bound * (1 + 1e-12))


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_nonzero_rank_is_copied_exactly(dtype):
    n, N, k = 8, 999, 5
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=3)
    zero = np.zeros_like(xs[0])
    ys = [xs[k] if r == k else zero for r in range(n)]
    out = oracle.all_reduce(ys, dtype)
    # +0 + x = x exactly for every x except -0 (which gives +0)
    want = xs[k].copy()
    w = widen(want, dtype)
    want[(w == 0)] = 0
    for o in out:
        np.testing.assert_array_equal(o, want)


@pytest.mark.parametrize("dtype", DTYPES)
def test_x_and_minus_x_give_plus_zero(dtype):
    N = 512
    x = workloads.rank_inputs(1, N, dtype, "normal", seed=4)[0]
    sign = np.uint32(0x80000000) if dtype == "f32" else np.uint16(0x8000)
    neg = (x.view(np.uint32 if dtype == "f32" else np.uint16) ^ sign).view(x.dtype)
    out = oracle.all_reduce([x, neg], dtype)[0]
    assert np.all(out.view(np.uint32 if dtype == "f32" else np.uint16) == 0)


@pytest.mark.parametrize("dtype", DTYPES)
def test_all_negative_zero_gives_plus_zero(dtype):
    # the accumulator starts at +0 (custom all-reduce notes, §4: acc = {})
    negz = np.full(64, 0x80000000 if dtype == "f32" else 0x8000,
                   np.uint32 if dtype == "f32" else np.uint16)
    x = negz.view(np.float32) if dtype == "f32" else negz
    out = oracle.all_reduce([x.copy() for _ in range(4)], dtype)[0]
    assert np.all(out.view(np.uint32 if dtype == "f32" else np.uint16) == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rank_permutation_changes_bits_only_within_tolerance(dtype):
    n, N = 8, 4096
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=12)
    a = widen(oracle.all_reduce(xs, dtype)[0], dtype)
    b = widen(oracle.all_reduce(xs[::-1], dtype)[0], dtype)
    abs_sum = sum(np.abs(widen(x, dtype)) for x in xs)
    ulp = {"bf16": 2.0**-7, "f16": 2.0**-10}[dtype]
    tol = np.maximum(ulp * np.abs(a), 2.0**-8 * abs_sum)
    assert np.all(np.abs(a - b) <= tol)


def test_chunk_size_rounds_to_whole_vectors():
    assert oracle.chunk_elems(2, 1024, "f32") == 512
    assert oracle.chunk_elems(8, 10, "bf16") == 8      # ceil(10/8)=2 -> one 8-element vector
    assert oracle.chunk_elems(8, 64, "bf16") == 8
    assert oracle.chunk_elems(8, 65, "bf16") == 16
    assert oracle.chunk_elems(3, 12, "f32") == 4
    assert oracle.chunk_elems(16, 0, "f16") == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n,N", [(2, 1024), (8, 10), (8, 65), (8, 4096 + 5), (16, 3), (16, 1000), (5, 77)])
def test_reduce_scatter_then_all_gather_is_all_reduce(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=N + n)
    want = oracle.all_reduce(xs, dtype)
    sentinel = 0x7FC00001 if dtype == "f32" else 0x7E01
    fill = np.full(N, sentinel, np.uint32 if dtype == "f32" else np.uint16)
    outs = [fill.view(xs[0].dtype).copy() for _ in range(n)]
    oracle.reduce_scatter(xs, dtype, outs)
    C = oracle.chunk_elems(n, N, dtype)
    for r in range(n):   # reduce-scatter writes chunk r of rank r and nothing else
        lo, hi = min(r * C, N), min((r + 1) * C, N)
        np.testing.assert_array_equal(outs[r][lo:hi], want[r][lo:hi])
        rest = np.concatenate([outs[r][:lo], outs[r][hi:]]).view(fill.dtype)
        assert np.all(rest == sentinel)
    oracle.all_gather(outs, dtype)
    for r in range(n):
        np.testing.assert_array_equal(outs[r], want[r])
