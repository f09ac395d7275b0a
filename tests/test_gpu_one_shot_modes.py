"""ar_one_shot_push and ar_one_shot_copyin (custom all-reduce notes, §实现:
one-shot push beside one-shot pull; §5 写回: copy-in to a registered buffer
outside graph capture).  Both do one-shot's arithmetic (fp32 sum in rank
order from +0, one rounding), so both are compared bit for bit with the
oracle's all-reduce and with ar_one_shot; canary bands must stay intact."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Handle, bits, empty_ranks, payload_np_dtype, ptrs, upload_ranks

pytestmark = pytest.mark.gpu

E = {"f32": 4, "bf16": 2, "f16": 2}
CALLS = {"push": (ar.ar_one_shot_push, "push_staging", ar.AR_OP_ONE_SHOT_PUSH, 2),
         "copyin": (ar.ar_one_shot_copyin, "registered", ar.AR_OP_ONE_SHOT_COPYIN, 2)}


@pytest.mark.parametrize("mode", ["push", "copyin"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n,N", [(2, 1), (2, 9), (3, 1000), (8, 4099), (8, 300_001), (16, 65536 + 3)])
def test_mode_matches_one_shot_bit_for_bit(mode, dtype, n, N):
    call, opt, op, launches = CALLS[mode]
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=17 * n + N)
    want = oracle.all_reduce(xs, dtype)
    ins, outs, ref = upload_ranks(xs), empty_ranks(n, xs[0].nbytes), empty_ranks(n, xs[0].nbytes)
    with Handle(n, max(16, N * E[dtype]), **{opt: 1}) as h:
        assert call(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        t = ar.ar_traffic(h)
        assert t.op == op and t.launches == launches
        assert ar.ar_one_shot(h, ptrs(ins), ptrs(ref), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    for r in range(n):
        got = outs[r].download(payload_np_dtype(dtype))
        np.testing.assert_array_equal(bits(got), bits(want[r]))
        np.testing.assert_array_equal(bits(got), bits(ref[r].download(payload_np_dtype(dtype))))
    for b in ins + outs + ref:
        assert b.guards_intact()


@pytest.mark.parametrize("mode", ["push", "copyin"])
def test_mode_in_place(mode):
    call, opt, _, _ = CALLS[mode]
    n, N = 8, 100_003
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=4)
    want = oracle.all_reduce(xs, "bf16")
    ins = upload_ranks(xs)
    with Handle(n, N * 2, **{opt: 1}) as h:
        assert call(h, ptrs(ins), ptrs(ins), N, "bf16") == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    for r in range(n):
        np.testing.assert_array_equal(ins[r].download(np.uint16), want[r])


@pytest.mark.parametrize("mode", ["push", "copyin"])
def test_mode_needs_its_buffers(mode):
    call, opt, _, _ = CALLS[mode]
    option = getattr(ar, "AR_OPT_" + opt.upper())
    n, N = 4, 1000
    ins, outs = empty_ranks(n, N * 4), empty_ranks(n, N * 4)
    with Handle(n, N * 4) as h:
        assert call(h, ptrs(ins), ptrs(outs), N, "f32") == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, option, 2) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, option, 1) == ar.AR_OK
        assert call(h, ptrs(ins), ptrs(outs), N, "f32") == ar.AR_OK
        assert call(h, ptrs(ins), ptrs(outs), N + 1, "f32") == ar.AR_ERR_TOO_LARGE
        assert ar.ar_set_option(h, option, 0) == ar.AR_OK
        assert call(h, ptrs(ins), ptrs(outs), N, "f32") == ar.AR_ERR_INVALID
        assert ar.ar_status(h) == ar.AR_OK


def test_push_timing_records_both_phases():
    n, N = 8, 65536
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=8)
    ins, outs = upload_ranks(xs), empty_ranks(n, N * 2)
    with Handle(n, N * 2, push_staging=1, timing=8) as h:
        assert ar.ar_one_shot_push(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
        recs = ar.ar_timing(h)
    assert [r[0] for r in recs] == ["push", "push_reduce"]
    t = ar.ar_plan(ar.AR_OP_ONE_SHOT_PUSH, n, N, "bf16")
    assert recs[0][3] + recs[1][3] == t.hbm_read_bytes + t.hbm_write_bytes


def test_copyin_timing_records_copy_and_one_shot():
    n, N = 8, 65536
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=9)
    ins, outs = upload_ranks(xs), empty_ranks(n, N * 2)
    with Handle(n, N * 2, registered=1, timing=8) as h:
        assert ar.ar_one_shot_copyin(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
        recs = ar.ar_timing(h)
    assert [r[0] for r in recs] == ["copyin", "one_shot"]
    t = ar.ar_plan(ar.AR_OP_ONE_SHOT_COPYIN, n, N, "bf16")
    assert recs[0][3] + recs[1][3] == t.hbm_read_bytes + t.hbm_write_bytes


@pytest.mark.parametrize("mode,n,N", [("push", 8, (1 << 20) + 5), ("push", 3, (12 << 20) + 7),
                                      ("copyin", 8, (8 << 20) + 3), ("copyin", 16, (4 << 20) + 1)])
def test_pieces_whole_buffers_launches_and_records(mode, n, N):
    # staged bytes (push: n (n-1) S; copy-in: n S) over half of L2: the call runs in pieces, each
    # staged and reduced in turn; every element of every rank against the oracle, the launches
    # the piece rule gives, and per-launch timing records whose bytes add up to the plan's
    dtype = "bf16"
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=17 + N % 7)
    want = oracle.all_reduce(xs, dtype)
    ins, outs = upload_ranks(xs), empty_ranks(n, N * 2)
    half = torch.cuda.get_device_properties(0).L2_cache_size // 2
    staged = n * (n - 1) * N * 2 if mode == "push" else n * N * 2
    P = min(64, max(1, (staged + half // 2) // half))
    PL = min(N, -(-(-(-N // P)) // 256) * 256)
    pieces = -(-N // PL)
    assert pieces > 1
    opts = {"push_staging": 1} if mode == "push" else {"registered": 1}
    with Handle(n, N * 2, timing=64, **opts) as h:
        call = ar.ar_one_shot_push if mode == "push" else ar.ar_one_shot_copyin
        assert call(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
        assert ar.ar_traffic(h).launches == 2 * pieces
        recs = ar.ar_timing(h)
        t = ar.ar_plan(ar.AR_OP_ONE_SHOT_PUSH if mode == "push" else ar.AR_OP_ONE_SHOT_COPYIN, n, N, dtype)
        assert len(recs) == 2 * pieces
        assert sum(r[3] for r in recs) == t.hbm_read_bytes + t.hbm_write_bytes
    for r in range(n):
        np.testing.assert_array_equal(outs[r].download(np.uint16), want[r])



@pytest.mark.parametrize("mode,n,N", [("push", 8, (2 << 20) + 5), ("copyin", 8, (8 << 20) + 3),
                                      ("copyin", 3, (24 << 20) + 1)])
def test_pieces_on_two_streams_whole_buffers(mode, n, N):
    # staged bytes over half of L2 and no timing records: the pieces run on two streams (twice as
    # many, alternating between the caller's stream and the handle's); every element of every
    # rank against the oracle, and the launches the rule gives
    dtype = "bf16"
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=29 + N % 11)
    want = oracle.all_reduce(xs, dtype)
    ins, outs = upload_ranks(xs), empty_ranks(n, N * 2)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    half = l2 // 2
    staged = n * (n - 1) * N * 2 if mode == "push" else n * N * 2
    assert staged * 2 >= l2
    P = min(64, max(1, (staged + half // 2) // half))
    PL = N if P == 1 else min(N, -(-(-(-N // P)) // 256) * 256)
    PL = min(N, -(-(-(-PL // 2)) // 256) * 256)
    opts = {"push_staging": 1} if mode == "push" else {"registered": 1}
    with Handle(n, N * 2, **opts) as h:
        call = ar.ar_one_shot_push if mode == "push" else ar.ar_one_shot_copyin
        for _ in range(2):   # twice: the handle's second stream is reused
            for o in outs:
                o.fill(0x5A)
            assert call(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
            assert ar.ar_status(h) == ar.AR_OK
            assert ar.ar_traffic(h).launches == 2 * -(-N // PL)
            for r in range(n):
                np.testing.assert_array_equal(outs[r].download(np.uint16), want[r])
