"""Pins for the oracle's ring all-reduce ("多 GPU 与 NCCL", §ring all-reduce).

- integer-valued inputs: every order is exact, so the ring must give the
  integer sum, for every n and for ragged lengths;
- a hand-worked n = 3 case whose values expose the summation order (below);
- the literal step simulation equals the per-element order statement;
- n = 2: the ring is one add of the two ranks (commutative), i.e. one-shot;
- reordered sums stay within the 1-bf16-ulp / 2^-8 tolerance of one-shot.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads

DTYPES = ["f32", "bf16", "f16"]


def test_hand_worked_rotation_n3():
    # fp32, n = 3, N = 12 -> C = 4: chunk 0 = elements 0..3, chunk 1 = 4..7,
    # chunk 2 = 8..11.  Rank 0 holds 1e8, rank 1 holds 1, rank 2 holds -1e8.
    # fp32 spacing at 1e8 is 8, so adding 1 to +-1e8 is lost.
    #   chunk 0 starts at rank 0: (1e8 + 1) + (-1e8)  = 1e8 - 1e8 = 0
    #   chunk 1 starts at rank 1: (1 + (-1e8)) + 1e8  = -1e8 + 1e8 = 0
    #   chunk 2 starts at rank 2: (-1e8 + 1e8) + 1    = 1
    # whereas the rank-order one-shot sum is (0 + 1e8 + 1) - 1e8 = 0 everywhere.
    xs = [np.full(12, v, np.float32) for v in (1e8, 1.0, -1e8)]
    want = np.array([0, 0, 0, 0, 0, 0, 0, 0, 1, 1, 1, 1], np.float32)
    out = oracle.ring(xs, "f32")
    for o in out:
        np.testing.assert_array_equal(o, want)
    np.testing.assert_array_equal(oracle.all_reduce(xs, "f32")[0], np.zeros(12, np.float32))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("N", [1, 9, 1000, 4096 + 3])
def test_ring_integer_inputs_exact(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "int8", seed=7 * n + N)
    want = oracle.all_reduce(xs, dtype)
    out = oracle.ring(xs, dtype)
    for r in range(n):
        np.testing.assert_array_equal(out[r], want[r])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [3, 8, 16])
def test_ring_simulation_equals_order_statement(dtype, n):
    N = 3001
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=n)
    out = oracle.ring(xs, dtype)
    C = oracle.chunk_elems(n, N, dtype)
    chunk = (np.arange(N) // C).astype(np.int32)
    want = oracle.ring_order_sum(xs, chunk, dtype)
    for o in out:
        np.testing.assert_array_equal(o, want)


@pytest.mark.parametrize("dtype", DTYPES)
def test_ring_n2_equals_one_shot(dtype):
    xs = workloads.rank_inputs(2, 5000, dtype, "normal", seed=21)
    a = oracle.ring(xs, dtype)
    b = oracle.all_reduce(xs, dtype)
    for r in range(2):
        np.testing.assert_array_equal(a[r], b[r])


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("n", [8, 16])
def test_ring_within_tolerance_of_one_shot(dtype, n):
    N = 8192 + 17
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=31 + n)
    g = oracle.to_f32(oracle.ring(xs, dtype)[0], dtype).astype(np.float64)
    o = oracle.to_f32(oracle.all_reduce(xs, dtype)[0], dtype).astype(np.float64)
    abs_sum = sum(np.abs(oracle.to_f32(x, dtype)).astype(np.float64) for x in xs)
    if dtype == "f32":
        tol = 1e-6 * np.maximum(np.abs(o), abs_sum)
    else:
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o), 2.0**-126))) - (7 if dtype == "bf16" else 10))
        tol = np.maximum(ulp, 2.0**-8 * abs_sum)
    assert np.all(np.abs(g - o) <= tol)


def test_ring_negative_zero_reading():
    # the first hop adds two raw values, so an all-(-0) chunk stays -0 in the
    # ring, while one-shot starts from +0
    x = np.full(8, -0.0, np.float32)
    out = oracle.ring([x.copy() for _ in range(3)], "f32")
    assert np.all(out[0].view(np.uint32) == 0x80000000)
    assert np.all(oracle.all_reduce([x.copy() for _ in range(3)], "f32")[0].view(np.uint32) == 0)


# --- the ring with partials rounded at every hop --------------------------

def test_rounded_ring_hand_worked_bf16():
    # n = 3 bf16, N = 24 -> C = 8: chunk 0 = elements 0..7, 1 = 8..15, 2 = 16..23.
    # Rank 0 holds 256, ranks 1 and 2 hold 1; bf16 spacing at 256 is 2.
    #   chunk 0 (order 0,1,2): RN(RN(256 + 1) + 1) = RN(256 + 1) = 256   (257 ties to even)
    #   chunk 1 (order 1,2,0): RN(RN(1 + 1) + 256) = 258
    #   chunk 2 (order 2,0,1): RN(RN(1 + 256) + 1) = 256
    # while fp32 partials give 258 everywhere.
    b = lambda v: oracle.f32_to_bf16(np.full(24, v, np.float32))
    xs = [b(256.0), b(1.0), b(1.0)]
    want = np.array([256.0] * 8 + [258.0] * 8 + [256.0] * 8, np.float32)
    for o in oracle.ring_rounded(xs, "bf16"):
        np.testing.assert_array_equal(oracle.bf16_to_f32(o), want)
    for o in oracle.ring(xs, "bf16"):
        np.testing.assert_array_equal(oracle.bf16_to_f32(o), np.full(24, 258.0, np.float32))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("n", [2, 5, 8])
def test_rounded_ring_per_element_with_library_arithmetic(dtype, n):
    # chunk c: p = x_c; p = round(p + x_{c+j}) for j = 1..n-1, with numpy's
    # float32 add and torch's / numpy's rounding to the payload type
    N = 999
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=60 + n)
    C = oracle.chunk_elems(n, N, dtype)
    f = [oracle.to_f32(x, dtype) for x in xs]

    def rnd(v):
        if dtype == "bf16":
            return torch.from_numpy(v).to(torch.bfloat16).float().numpy()
        return v.astype(np.float16).astype(np.float32)

    want = np.empty(N, np.float32)
    for c in range(n):
        lo, hi = min(c * C, N), min((c + 1) * C, N)
        p = f[c][lo:hi].copy()
        for j in range(1, n):
            p = rnd(p + f[(c + j) % n][lo:hi])
        want[lo:hi] = p
    for o in oracle.ring_rounded(xs, dtype):
        np.testing.assert_array_equal(oracle.to_f32(o, dtype), want)


@pytest.mark.parametrize("n", [3, 8])
def test_rounded_ring_equals_ring_for_f32_and_for_exact_integers(n):
    xs = workloads.rank_inputs(n, 4099, "f32", "normal", seed=n)
    for a, b in zip(oracle.ring_rounded(xs, "f32"), oracle.ring(xs, "f32")):
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
    xi = workloads.rank_inputs(n, 4099, "bf16", "int8", seed=n)
    exact = sum(oracle.to_f32(x, "bf16").astype(np.int64) for x in xi)
    for o in oracle.ring_rounded(xi, "bf16"):
        np.testing.assert_array_equal(oracle.to_f32(o, "bf16").astype(np.int64), exact)
