"""Pins for the oracle's all-reduce + residual add + RMSNorm.

- residual_out is the all-reduce (pinned elsewhere) plus the residual with
  one binary32 add (numpy) and one rounding to the payload (torch/numpy);
- constant rows have a closed form: r / sqrt(r^2 + eps) * w;
- with unit weight the output of every row has mean square 1 (to within
  the payload's rounding), and scaling a row's inputs by a power of two
  leaves it unchanged (eps = 0);
- the output is proportional to r * w within a row (signs and ratios).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads


def _round(x32, dtype):
    if dtype == "f32":
        return x32.astype(np.float32)
    if dtype == "bf16":
        return torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return x32.astype(np.float32).astype(np.float16).view(np.uint16)


def _layout(x32, dtype):
    return _round(np.asarray(x32, np.float32), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_residual_out_is_allreduce_plus_residual(dtype):
    n, T, H = 8, 3, 4096
    xs = workloads.rank_inputs(n, T * H, dtype, "normal", seed=1)
    res = workloads.rank_inputs(1, T * H, dtype, "normal", seed=2)[0]
    w = workloads.rank_inputs(1, H, dtype, "uniform", seed=3)[0]
    _, r = oracle.allreduce_rmsnorm(xs, res, w, 1e-6, T, H, dtype)
    a = oracle.to_f32(oracle.all_reduce(xs, dtype)[0], dtype)
    want = _round(a + oracle.to_f32(res, dtype), dtype)          # numpy binary32 add, library rounding
    np.testing.assert_array_equal(r, want)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_constant_rows_closed_form(dtype):
    n, H = 4, 1024
    vals = np.array([0.5, -2.0, 3.0], np.float32)            # per-row constant of the all-reduce
    T = vals.size
    xs = [_layout(np.repeat(vals / n, H), dtype) for _ in range(n)]    # exact: n copies sum to vals
    res = _layout(np.zeros(T * H), dtype)
    w = _layout(np.linspace(0.5, 1.5, H), dtype)
    eps = 1e-5
    y, r = oracle.allreduce_rmsnorm(xs, res, w, eps, T, H, dtype)
    wf = oracle.to_f32(w, dtype).astype(np.float64)
    for t, c in enumerate(vals.astype(np.float64)):
        want = c / np.sqrt(c * c + eps) * wf
        got = oracle.to_f32(y[t * H:(t + 1) * H], dtype).astype(np.float64)
        ulp = {"bf16": 2.0**-7, "f16": 2.0**-10, "f32": 2.0**-22}[dtype] * np.abs(want)
        assert np.all(np.abs(got - want) <= ulp)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unit_weight_rows_have_unit_mean_square_and_are_scale_free(dtype):
    n, T, H = 8, 4, 8192
    xs = workloads.rank_inputs(n, T * H, dtype, "normal", seed=5)
    res = workloads.rank_inputs(1, T * H, dtype, "normal", seed=6)[0]
    one = _layout(np.ones(H), dtype)
    y, _ = oracle.allreduce_rmsnorm(xs, res, one, 0.0, T, H, dtype)
    yf = oracle.to_f32(y, dtype).astype(np.float64).reshape(T, H)
    tol = {"bf16": 2.0**-7, "f32": 1e-6}[dtype]
    assert np.all(np.abs((yf**2).mean(axis=1) - 1.0) <= 2 * tol)
    # multiply every input and the residual by 4 (exact): the same output
    x4 = [_layout(oracle.to_f32(x, dtype) * 4, dtype) for x in xs]
    r4 = _layout(oracle.to_f32(res, dtype) * 4, dtype)
    y4, _ = oracle.allreduce_rmsnorm(x4, r4, one, 0.0, T, H, dtype)
    np.testing.assert_array_equal(y4, y)


def test_output_is_proportional_to_r_times_w():
    n, T, H, dtype = 2, 2, 2048, "f32"
    xs = workloads.rank_inputs(n, T * H, dtype, "normal", seed=8)
    res = workloads.rank_inputs(1, T * H, dtype, "normal", seed=9)[0]
    w = workloads.rank_inputs(1, H, dtype, "uniform", seed=10)[0]
    y, r = oracle.allreduce_rmsnorm(xs, res, w, 1e-6, T, H, dtype)
    for t in range(T):
        rw = r[t * H:(t + 1) * H].astype(np.float64) * w.astype(np.float64)
        ratio = y[t * H:(t + 1) * H].astype(np.float64) / rw
        assert np.allclose(ratio, ratio[0], rtol=1e-6)
        assert ratio[0] > 0
