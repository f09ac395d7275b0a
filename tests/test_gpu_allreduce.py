"""Parity of ar_one_shot / ar_two_shot / ar_ring against the CPU oracle,
through the C-ABI, on seeded inputs.

Bar: one-shot and two-shot keep the oracle's rank order, so they must be
bit-exact to oracle.all_reduce; the ring must be bit-exact to oracle.ring
(its own order) and within 1 payload ulp, or 2^-8 of sum|x| (1e-6 relative
for fp32), of the one-shot result.  Every buffer carries canary bands that
must be untouched afterwards.
"""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Buf, Handle, bits, empty_ranks, payload_np_dtype, ptrs, upload_ranks

pytestmark = pytest.mark.gpu

CALLS = {"one_shot": ar.ar_one_shot, "two_shot": ar.ar_two_shot, "ring": ar.ar_ring}
E = {"f32": 4, "bf16": 2, "f16": 2}


def run(algo, xs, dtype, in_place=False, stream=None, h=None, max_bytes=None):
    n, N = len(xs), xs[0].size
    ins = upload_ranks(xs)
    outs = ins if in_place else empty_ranks(n, xs[0].nbytes)
    mb = max_bytes or max(16, N * E[dtype])

    def call(handle):
        rc = CALLS[algo](handle, ptrs(ins), ptrs(outs), N, dtype, stream)
        assert rc == ar.AR_OK, ar.ar_strerror(rc)
        assert ar.ar_status(handle) == ar.AR_OK

    if h is None:
        with Handle(n, mb) as handle:
            call(handle)
    else:
        call(h)
    torch.cuda.synchronize()
    for b in ins + outs:
        assert b.guards_intact()
    return [o.download(payload_np_dtype(dtype)) for o in outs]


def tolerance_ok(g, o, xs, dtype):
    gf = oracle.to_f32(g, dtype).astype(np.float64)
    of = oracle.to_f32(o, dtype).astype(np.float64)
    abs_sum = sum(np.abs(oracle.to_f32(x, dtype)).astype(np.float64) for x in xs)
    if dtype == "f32":
        tol = 1e-6 * np.maximum(np.abs(of), abs_sum)
    else:
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(of), 2.0**-126))) - (7 if dtype == "bf16" else 10))
        tol = np.maximum(ulp, 2.0**-8 * abs_sum)
    return bool(np.all(np.abs(gf - of) <= tol))


# sizes: several tiles of 256 threads x 16 B and ragged tails of every length
SIZES = [1, 3, 7, 8, 9, 15, 17, 100, 1000, 4096, 8191, 65536 + 5, 300_001]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("N", SIZES)
def test_one_and_two_shot_bit_exact(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=n * 7919 + N)
    want = oracle.all_reduce(xs, dtype)
    for algo in ("one_shot", "two_shot"):
        got = run(algo, xs, dtype)
        for r in range(n):
            np.testing.assert_array_equal(bits(got[r]), bits(want[r]), err_msg=f"{algo} rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("N", [1, 9, 1000, 4099, 65536 + 3, 300_001])
def test_ring_matches_its_order_and_tolerance(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=n * 104729 + N)
    want = oracle.ring(xs, dtype)
    got = run("ring", xs, dtype)
    for r in range(n):
        np.testing.assert_array_equal(bits(got[r]), bits(want[r]), err_msg=f"rank {r}")
    assert tolerance_ok(got[0], oracle.all_reduce(xs, dtype)[0], xs, dtype)


@pytest.mark.parametrize("algo", ["one_shot", "two_shot", "ring"])
@pytest.mark.parametrize("n", [2, 8, 16])
def test_in_place(algo, n):
    dtype, N = "bf16", 50_001
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=5 + n)
    want = (oracle.ring if algo == "ring" else oracle.all_reduce)(xs, dtype)
    got = run(algo, xs, dtype, in_place=True)
    for r in range(n):
        np.testing.assert_array_equal(bits(got[r]), bits(want[r]))


def test_config1_n2_f32_integers_exact():
    cfg = workloads.CONFIGS[1]
    xs = workloads.rank_inputs(cfg["n"], cfg["counts"][0], "f32", cfg["dist"], workloads.seed_of(1))
    exact = (xs[0].astype(np.int64) + xs[1].astype(np.int64)).astype(np.float32)
    for algo in cfg["algos"]:
        got = run(algo, xs, "f32")
        for g in got:
            np.testing.assert_array_equal(g, exact)


@pytest.mark.parametrize("N", workloads.CONFIGS[2]["counts"])
def test_config2_decode_sizes(N):
    cfg = workloads.CONFIGS[2]
    xs = workloads.rank_inputs(cfg["n"], N, "bf16", cfg["dist"], workloads.seed_of(2) + N)
    want = oracle.all_reduce(xs, "bf16")
    for algo in cfg["algos"]:
        got = run(algo, xs, "bf16")
        for r in range(cfg["n"]):
            np.testing.assert_array_equal(got[r], want[r])


@pytest.mark.parametrize("n", range(2, 17))
def test_every_rank_count(n):
    N = 4096 + 7
    xs = workloads.rank_inputs(n, N, "bf16", "int8", seed=n)
    exact = sum(oracle.to_f32(x, "bf16").astype(np.int64) for x in xs)
    for algo in ("one_shot", "two_shot", "ring"):
        got = run(algo, xs, "bf16")
        for g in got:
            np.testing.assert_array_equal(oracle.to_f32(g, "bf16").astype(np.int64), exact)


def test_nccl_fill_pattern_zero_mismatches():
    # the NCCL example's check: rank g holds g + i % 7, expect n(n-1)/2 + n (i % 7)
    n, N = 8, (1 << 20) + 3
    xs = workloads.rank_inputs(n, N, "f32", "fill7", seed=0)
    i = np.arange(N)
    want = np.float32(n * (n - 1) / 2) + np.float32(n) * (i % 7).astype(np.float32)
    for algo in ("one_shot", "two_shot", "ring"):
        got = run(algo, xs, "f32", in_place=True)
        assert sum(int(np.count_nonzero(g != want)) for g in got) == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_signed_zero_readings(dtype):
    neg = np.full(64, 0x80000000 if dtype == "f32" else 0x8000, np.uint32 if dtype == "f32" else np.uint16)
    x = neg.view(np.float32) if dtype == "f32" else neg
    xs = [x.copy() for _ in range(3)]
    for algo in ("one_shot", "two_shot"):
        assert np.all(bits(run(algo, xs, dtype)[1]) == 0)         # accumulator starts at +0
    assert np.all(bits(run("ring", xs, dtype)[1]) == bits(oracle.ring(xs, dtype)[1]))


def test_inf_and_nan_propagate():
    n, N = 4, 4096
    xs = workloads.rank_inputs(n, N, "f32", "normal", seed=77)
    xs[1][::7] = np.inf
    xs[2][::11] = -np.inf
    xs[3][::13] = np.nan
    want = oracle.all_reduce(xs, "f32")[0]
    for algo in ("one_shot", "two_shot", "ring"):
        g = run(algo, xs, "f32")[0]
        assert np.array_equal(np.isnan(g), np.isnan(want))
        keep = ~np.isnan(want)
        if algo == "ring":
            assert np.array_equal(np.isinf(g[keep]), np.isinf(want[keep]))
        else:
            np.testing.assert_array_equal(bits(g[keep]), bits(want[keep]))


def test_empty_count_is_a_no_op():
    with Handle(8, 1 << 16) as h:
        outs = empty_ranks(8, 64, byte=0x33)
        for call in CALLS.values():
            assert call(h, ptrs(outs), ptrs(outs), 0, "bf16") == ar.AR_OK
            assert ar.ar_traffic(h).launches == 0
        torch.cuda.synchronize()
        assert all(bool((o.body() == 0x33).all()) for o in outs)


def test_max_bytes_boundary_and_errors():
    n, N = 4, 1 << 16
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=9)
    want = oracle.all_reduce(xs, "bf16")
    with Handle(n, N * 2) as h:                      # exactly one buffer's worth
        for algo in CALLS:
            got = run(algo, xs, "bf16", h=h)
            if algo != "ring":
                np.testing.assert_array_equal(got[2], want[2])
        ins = upload_ranks(xs)
        outs = empty_ranks(n, xs[0].nbytes, byte=0x11)
        assert ar.ar_one_shot(h, ptrs(ins), ptrs(outs), N + 1, "bf16") == ar.AR_ERR_TOO_LARGE
        bad = ptrs(outs)
        bad[1] += 2
        assert ar.ar_two_shot(h, ptrs(ins), bad, N - 8, "bf16") == ar.AR_ERR_ALIGN
        assert ar.ar_ring(h, ptrs(ins), ptrs(outs), 10, 5) == ar.AR_ERR_INVALID
        torch.cuda.synchronize()
        assert all(bool((o.body() == 0x11).all()) for o in outs)   # nothing launched


def test_traffic_reports_the_last_call():
    n, N = 8, 12345
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=1)
    with Handle(n, N * 2) as h:
        for algo, op in (("one_shot", ar.AR_OP_ONE_SHOT), ("two_shot", ar.AR_OP_TWO_SHOT), ("ring", ar.AR_OP_RING)):
            run(algo, xs, "bf16", h=h)
            t = ar.ar_traffic(h).as_dict()
            p = ar.ar_plan(op, n, N, "bf16").as_dict()
            assert t == p and t["op"] == op


def test_non_default_stream():
    n, N = 8, 200_000
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=3)
    want = oracle.all_reduce(xs, "bf16")
    s = torch.cuda.Stream()
    got = run("one_shot", xs, "bf16", stream=s)
    np.testing.assert_array_equal(got[7], want[7])
    got = run("ring", xs, "bf16", stream=s)
    np.testing.assert_array_equal(got[0], oracle.ring(xs, "bf16")[0])


def test_cuda_graph_capture_and_replay():
    n, N = 8, 65536
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=4)
    ys = workloads.rank_inputs(n, N, "bf16", "normal", seed=5)
    ins = upload_ranks(xs)
    outs = empty_ranks(n, xs[0].nbytes)
    with Handle(n, N * 2) as h:
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rc1 = ar.ar_one_shot(h, ptrs(ins), ptrs(outs), N, "bf16", s)
            rc2 = ar.ar_ring(h, ptrs(ins), ptrs(outs), N, "bf16", s)
            rc3 = ar.ar_two_shot(h, ptrs(ins), ptrs(outs), N, "bf16", s)
        assert rc1 == rc2 == rc3 == ar.AR_OK
        for src in (xs, ys):             # same addresses, new contents, replay
            for b, a in zip(ins, src):
                b.upload(a)
            g.replay()
            torch.cuda.synchronize()
            want = oracle.all_reduce(src, "bf16")
            for r in range(n):
                np.testing.assert_array_equal(outs[r].download(np.uint16), want[r])
        assert ar.ar_status(h) == ar.AR_OK


def test_handle_is_reusable_across_sizes_and_types():
    with Handle(8, 1 << 20) as h:
        for dtype, N in (("bf16", 77), ("f32", 1 << 18), ("f16", 5000), ("bf16", 1 << 19)):
            xs = workloads.rank_inputs(8, N, dtype, "normal", seed=N)
            for algo in CALLS:
                got = run(algo, xs, dtype, h=h)
                want = (oracle.ring if algo == "ring" else oracle.all_reduce)(xs, dtype)
                np.testing.assert_array_equal(bits(got[3]), bits(want[3]))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("N", [1, 7, 9, 2047, 2048, 4096 + 8, 300_001, 1 << 21])
def test_one_shot_bulk_copy_variant_bit_exact(dtype, n, N):
    # AR_OPT_ONE_SHOT_IMPL = 2: rank tiles staged in shared memory by bulk copies,
    # tiles of 4 KiB per rank (several tiles, a partial last tile, a ragged tail)
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=n * 13 + N)
    want = oracle.all_reduce(xs, dtype)
    with Handle(n, max(16, N * E[dtype]), one_shot_impl=2) as h:
        for in_place in (False, True):
            got = run("one_shot", xs, dtype, h=h, in_place=in_place)
            for r in range(n):
                np.testing.assert_array_equal(bits(got[r]), bits(want[r]), err_msg=f"rank {r} in_place={in_place}")


@pytest.mark.parametrize("ctas", [1, 3, 16, 64])
@pytest.mark.parametrize("impl", [1, 2])
def test_grid_size_option_changes_nothing_but_speed(ctas, impl):
    n, N = 8, 1 << 20
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=ctas)
    with Handle(n, 2 * N, ctas_per_sm=ctas, one_shot_impl=impl) as h:
        for algo in CALLS:
            got = run(algo, xs, "bf16", h=h)
            want = (oracle.ring if algo == "ring" else oracle.all_reduce)(xs, "bf16")
            np.testing.assert_array_equal(got[5], want[5])


@pytest.mark.parametrize("pdl", [0, 1])
def test_programmatic_launch_on_and_off_give_the_same_bits(pdl):
    # back-to-back calls that depend on each other through memory: in place,
    # so each call reads what the previous one wrote
    n, N = 8, (1 << 18) + 5
    xs = workloads.rank_inputs(n, N, "f32", "int8", seed=pdl)
    ins = upload_ranks(xs)
    with Handle(n, 4 * N, pdl=pdl) as h:
        for call in (ar.ar_one_shot, ar.ar_two_shot, ar.ar_ring, ar.ar_one_shot):
            assert call(h, ptrs(ins), ptrs(ins), N, "f32") == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    # integer inputs, |sum| <= 64 n^4 < 2^24: every pass is exact, and each
    # pass after the first sums n equal copies
    s = sum(x.astype(np.int64) for x in xs)
    want = (s * n**3).astype(np.float32)
    for b in ins:
        np.testing.assert_array_equal(b.download(np.float32), want)


@pytest.mark.parametrize("policy", [0, 1])
@pytest.mark.parametrize("N", [4096, 200_000, 5_000_000])
def test_auto_runs_the_selected_call(policy, N):
    n, dtype = 8, "bf16"
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=N + policy)
    with Handle(n, 2 * N, auto_policy=policy, auto_handoff=4 << 20) as h:
        got = run("one_shot", xs, dtype, h=h)  # warm the handle, then the auto call below
        ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
        assert ar.ar_auto(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
        chosen = ar.ar_traffic(h).op
    torch.cuda.synchronize()
    want_op = ar.ar_select(policy, n, 2 * N, 1.5e-6, 450e9, 4 << 20)
    assert chosen == want_op
    want = (oracle.ring if chosen == ar.AR_OP_RING else oracle.all_reduce)(xs, dtype)
    for r in range(n):
        np.testing.assert_array_equal(outs[r].download(np.uint16), want[r])


def test_launch_timing_records():
    n, N = 8, 1 << 20
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=12)
    ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
    with Handle(n, 2 * N, timing=64) as h:
        assert ar.ar_one_shot(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
        assert ar.ar_ring(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
        assert ar.ar_set_option(h, ar.AR_OPT_TIMING_PAUSE, 1) == ar.AR_OK
        assert ar.ar_two_shot(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK     # not recorded
        assert ar.ar_set_option(h, ar.AR_OPT_TIMING_PAUSE, 0) == ar.AR_OK
        recs = ar.ar_timing(h)
        assert ar.ar_timing(h) == []                                               # read clears
        assert ar.ar_status(h) == ar.AR_OK
    names = [r[0] for r in recs]
    assert names == ["one_shot", "ring_rs_step", "ring_ag_step"]
    assert [r[4] for r in recs] == [1, n - 1, n - 1]
    assert all(r[2] > 0 for r in recs)
    plan_ring = ar.ar_plan(ar.AR_OP_RING, n, N, "bf16")
    assert recs[0][3] == 2 * n * N * 2
    assert recs[1][3] + recs[2][3] == plan_ring.hbm_read_bytes + plan_ring.hbm_write_bytes


# --- the ring with per-hop rounding, and the pairwise tree -------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n,N", [(2, 9), (3, 1000), (8, 4099), (8, 300_001), (16, 65536 + 3)])
def test_ring_rounded_matches_its_oracle(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=n * 3 + N)
    want = oracle.ring_rounded(xs, dtype)
    ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
    with Handle(n, max(16, N * E[dtype])) as h:
        assert ar.ar_ring_rounded(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
        assert ar.ar_traffic(h).op == ar.AR_OP_RING_ROUNDED
    torch.cuda.synchronize()
    for r in range(n):
        np.testing.assert_array_equal(bits(outs[r].download(payload_np_dtype(dtype))), bits(want[r]))
    for b in ins + outs:
        assert b.guards_intact()
    if dtype == "f32":
        np.testing.assert_array_equal(bits(outs[0].download(np.float32)), bits(oracle.ring(xs, "f32")[0]))


def test_ring_rounded_in_place_hand_worked():
    # bf16, n = 3, 8 elements per chunk: rank 0 holds 256, ranks 1 and 2 hold 1
    b = lambda v: oracle.f32_to_bf16(np.full(24, v, np.float32))
    ins = upload_ranks([b(256.0), b(1.0), b(1.0)])
    with Handle(3, 48) as h:
        assert ar.ar_ring_rounded(h, ptrs(ins), ptrs(ins), 24, "bf16") == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    want = np.array([256.0] * 8 + [258.0] * 8 + [256.0] * 8, np.float32)
    for x in ins:
        np.testing.assert_array_equal(oracle.bf16_to_f32(x.download(np.uint16)), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n,N", [(2, 9), (4, 1000), (8, 4099), (8, 300_001), (16, 65536 + 3), (16, 7)])
def test_tree_matches_its_oracle(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=5 * n + N)
    want = oracle.tree(xs, dtype)
    ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
    with Handle(n, max(16, N * E[dtype])) as h:
        assert ar.ar_tree(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
        t = ar.ar_traffic(h)
        assert t.op == ar.AR_OP_TREE and t.launches == n.bit_length() - 1
    torch.cuda.synchronize()
    for r in range(n):
        np.testing.assert_array_equal(bits(outs[r].download(payload_np_dtype(dtype))), bits(want[r]))
    for b in ins + outs:
        assert b.guards_intact()


def test_tree_in_place_hand_worked_and_refusals():
    # bf16, n = 4: ranks hold 256, 1, 1, 0 -> 256 on every rank (one-shot gives 258)
    b = lambda v: oracle.f32_to_bf16(np.full(40, v, np.float32))
    ins = upload_ranks([b(256.0), b(1.0), b(1.0), b(0.0)])
    with Handle(4, 80) as h:
        assert ar.ar_tree(h, ptrs(ins), ptrs(ins), 40, "bf16") == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    for x in ins:
        np.testing.assert_array_equal(oracle.bf16_to_f32(x.download(np.uint16)), np.full(40, 256.0, np.float32))
    with Handle(3, 64) as h:
        ins3, outs3 = empty_ranks(3, 64), empty_ranks(3, 64)
        assert ar.ar_tree(h, ptrs(ins3), ptrs(outs3), 16, "bf16") == ar.AR_ERR_INVALID
        assert ar.ar_tree(h, ptrs(ins3), ptrs(outs3), 0, "bf16") == ar.AR_ERR_INVALID


@pytest.mark.parametrize("call,oracle_fn", [
    ("ar_one_shot_push", "all_reduce"), ("ar_one_shot_copyin", "all_reduce"), ("ar_ring_rounded", "ring_rounded"),
    ("ar_tree", "tree"), ("ar_tree_fused", "tree"), ("ar_ring_persistent", "ring"), ("ar_ring_cluster", "ring"),
    ("ar_ring_fused", "ring"), ("ar_ring_rounded_fused", "ring_rounded")])
def test_cuda_graph_capture_of_the_other_calls(call, oracle_fn):
    # captured once, replayed on new contents of the same buffers
    n, N = 8, 65536 + 3
    xs = workloads.rank_inputs(n, N, "bf16", "normal_over_n", seed=14)
    ys = workloads.rank_inputs(n, N, "bf16", "normal_over_n", seed=15)
    ins = upload_ranks(xs)
    outs = empty_ranks(n, xs[0].nbytes)
    with Handle(n, N * 2, push_staging=1, registered=1, persistent=1) as h:
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rc = getattr(ar, call)(h, ptrs(ins), ptrs(outs), N, "bf16", s)
        assert rc == ar.AR_OK
        for src in (xs, ys):
            for b, a in zip(ins, src):
                b.upload(a)
            g.replay()
            torch.cuda.synchronize()
            want = getattr(oracle, oracle_fn)(src, "bf16")
            for r in (0, 5):
                np.testing.assert_array_equal(outs[r].download(np.uint16), want[r])
        assert ar.ar_status(h) == ar.AR_OK


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n,N", [(2, 9), (4, 1000), (8, 4099), (8, 300_001), (16, 65536 + 3), (16, 7)])
def test_tree_fused_matches_the_tree(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=9 * n + N)
    want = oracle.tree(xs, dtype)
    ins = upload_ranks(xs)
    a, b = empty_ranks(n, xs[0].nbytes), empty_ranks(n, xs[0].nbytes)
    with Handle(n, max(16, N * E[dtype])) as h:
        assert ar.ar_tree_fused(h, ptrs(ins), ptrs(a), N, dtype) == ar.AR_OK
        t = ar.ar_traffic(h)
        assert t.op == ar.AR_OP_TREE_FUSED and t.launches == 1
        assert ar.ar_tree(h, ptrs(ins), ptrs(b), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    for r in range(n):
        got = a[r].download(payload_np_dtype(dtype))
        np.testing.assert_array_equal(bits(got), bits(want[r]))
        np.testing.assert_array_equal(bits(got), bits(b[r].download(payload_np_dtype(dtype))))
    for buf in ins + a + b:
        assert buf.guards_intact()


def test_tree_fused_in_place_and_refusal():
    b = lambda v: oracle.f32_to_bf16(np.full(40, v, np.float32))
    ins = upload_ranks([b(256.0), b(1.0), b(1.0), b(0.0)])
    with Handle(4, 80) as h:
        assert ar.ar_tree_fused(h, ptrs(ins), ptrs(ins), 40, "bf16") == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    for x in ins:
        np.testing.assert_array_equal(oracle.bf16_to_f32(x.download(np.uint16)), np.full(40, 256.0, np.float32))
    with Handle(6, 64) as h:
        i6, o6 = empty_ranks(6, 64), empty_ranks(6, 64)
        assert ar.ar_tree_fused(h, ptrs(i6), ptrs(o6), 16, "bf16") == ar.AR_ERR_INVALID


# --- the ring's steps done in registers in one pass -----------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n,N", [(2, 9), (3, 1000), (5, 4099), (8, 4099), (8, 300_001), (13, 50_001),
                                 (16, 65536 + 3), (16, 7)])
def test_ring_fused_matches_the_ring(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=11 * n + N)
    ins = upload_ranks(xs)
    a, b = empty_ranks(n, xs[0].nbytes), empty_ranks(n, xs[0].nbytes)
    ra, rb = empty_ranks(n, xs[0].nbytes), empty_ranks(n, xs[0].nbytes)
    with Handle(n, max(16, N * E[dtype])) as h:
        assert ar.ar_ring_fused(h, ptrs(ins), ptrs(a), N, dtype) == ar.AR_OK
        t = ar.ar_traffic(h)
        assert t.op == ar.AR_OP_RING_FUSED and t.launches == 1 and t.steps == 2 * (n - 1)
        assert ar.ar_ring(h, ptrs(ins), ptrs(b), N, dtype) == ar.AR_OK
        assert ar.ar_ring_rounded_fused(h, ptrs(ins), ptrs(ra), N, dtype) == ar.AR_OK
        assert ar.ar_traffic(h).op == ar.AR_OP_RING_ROUNDED_FUSED
        assert ar.ar_ring_rounded(h, ptrs(ins), ptrs(rb), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    want, want_r = oracle.ring(xs, dtype), oracle.ring_rounded(xs, dtype)
    for r in range(n):
        got = a[r].download(payload_np_dtype(dtype))
        np.testing.assert_array_equal(bits(got), bits(want[r]))
        np.testing.assert_array_equal(bits(got), bits(b[r].download(payload_np_dtype(dtype))))
        got_r = ra[r].download(payload_np_dtype(dtype))
        np.testing.assert_array_equal(bits(got_r), bits(want_r[r]))
        np.testing.assert_array_equal(bits(got_r), bits(rb[r].download(payload_np_dtype(dtype))))
    for buf in ins + a + b + ra + rb:
        assert buf.guards_intact()


def test_ring_fused_in_place_hand_worked():
    # bf16, n = 3, 8 elements per chunk: rank 0 holds 256, ranks 1 and 2 hold 1.
    # Chunk 0 adds 256 + 1 + 1 = 258 in fp32 (exact in bf16); the hop-rounded
    # form rounds 257 to 256 first and ends at 256.  Chunk 1 starts at rank 1:
    # 1 + 1 + 256 = 258 both ways.  Chunk 2 starts at rank 2: 1 + 256 = 257,
    # which the hop-rounded form rounds to 256 before adding the last 1.
    b = lambda v: oracle.f32_to_bf16(np.full(24, v, np.float32))
    x = [b(256.0), b(1.0), b(1.0)]
    ins, ins_r = upload_ranks(x), upload_ranks(x)
    with Handle(3, 48) as h:
        assert ar.ar_ring_fused(h, ptrs(ins), ptrs(ins), 24, "bf16") == ar.AR_OK
        assert ar.ar_ring_rounded_fused(h, ptrs(ins_r), ptrs(ins_r), 24, "bf16") == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    for y in ins:
        np.testing.assert_array_equal(oracle.bf16_to_f32(y.download(np.uint16)), np.full(24, 258.0, np.float32))
    want_r = np.array([256.0] * 8 + [258.0] * 8 + [256.0] * 8, np.float32)
    for y in ins_r:
        np.testing.assert_array_equal(oracle.bf16_to_f32(y.download(np.uint16)), want_r)
