"""Pins for the oracle's pairwise tree (the PCIe-IPC blog, §3.1: ranks pair
up, each reads its own and its peer's data, adds, writes both; log2 n
levels).

- integer-valued inputs: every order is exact, so the tree gives the sum;
- a hand-worked bf16 case where the per-level rounding shows;
- per element, the same pairing computed with numpy's float32 add and
  torch's / numpy's rounding;
- n = 2 is one add: one-shot's result (inputs without -0).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [2, 4, 8, 16])
def test_tree_integer_inputs_exact(dtype, n):
    xs = workloads.rank_inputs(n, 1001, dtype, "int8", seed=n)
    exact = sum(oracle.to_f32(x, dtype).astype(np.int64) for x in xs)
    for o in oracle.tree(xs, dtype):
        np.testing.assert_array_equal(oracle.to_f32(o, dtype).astype(np.int64), exact)


def test_tree_hand_worked_bf16():
    # n = 4, ranks hold 256, 1, 1, 0 (bf16 spacing at 256 is 2):
    #   level 0: RN(256 + 1) = 256 (257 ties to even) on ranks 0,1; RN(1 + 0) = 1 on ranks 2,3
    #   level 1: RN(256 + 1) = 256 everywhere   -- one-shot gives RN(258) = 258
    b = lambda v: oracle.f32_to_bf16(np.full(16, v, np.float32))
    xs = [b(256.0), b(1.0), b(1.0), b(0.0)]
    for o in oracle.tree(xs, "bf16"):
        np.testing.assert_array_equal(oracle.bf16_to_f32(o), np.full(16, 256.0, np.float32))
    np.testing.assert_array_equal(oracle.bf16_to_f32(oracle.all_reduce(xs, "bf16")[0]),
                                  np.full(16, 258.0, np.float32))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("n", [4, 8, 16])
def test_tree_per_element_with_library_arithmetic(dtype, n):
    xs = workloads.rank_inputs(n, 777, dtype, "normal_over_n", seed=90 + n)
    v = [oracle.to_f32(x, dtype) for x in xs]

    def rnd(a):
        if dtype == "bf16":
            return torch.from_numpy(a).to(torch.bfloat16).float().numpy()
        return a.astype(np.float16).astype(np.float32)

    d = 1
    while d < n:
        v = [rnd(v[r] + v[r ^ d]) for r in range(n)]
        d *= 2
    for o in oracle.tree(xs, dtype):
        np.testing.assert_array_equal(oracle.to_f32(o, dtype), v[0])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_n2_is_one_shot_and_other_n_are_refused(dtype):
    xs = workloads.rank_inputs(2, 5000, dtype, "normal", seed=3)
    np.testing.assert_array_equal(oracle.tree(xs, dtype)[1], oracle.all_reduce(xs, dtype)[1])
    with pytest.raises(ValueError):
        oracle.tree(workloads.rank_inputs(3, 10, dtype, "normal", seed=1), dtype)
