"""The three forms of ar_two_shot (AR_OPT_TWO_SHOT_IMPL): two launches; one
launch whose phases are separated per tile by a CTA barrier (the default);
one launch whose tiles are handed between CTAs by ready flags.

Handbook "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §算法
(two-shot: a reduce-scatter, a synchronization, an all-gather); every form
keeps one-shot's rank order, so each must equal oracle.all_reduce bit for
bit, on every rank, with the buffers' guard bands intact.  The flag form
keeps a call counter in the handle: repeated calls, in-place calls and graph
replays must each see their own flags.  Its bounded wait is made to run out
by a 1 ns limit; the call must then report AR_ERR_WAIT_TIMEOUT or succeed,
every output element must be either the right sum or untouched, and the next
call must succeed.
"""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Handle, bits, empty_ranks, payload_np_dtype, ptrs, upload_ranks

pytestmark = pytest.mark.gpu

E = {"f32": 4, "bf16": 2, "f16": 2}
TWO_LAUNCHES, ONE_LAUNCH, TILE_FLAGS = 1, 2, 3
FORMS = [TWO_LAUNCHES, ONE_LAUNCH, TILE_FLAGS]
SIZES = [1, 7, 8, 9, 100, 1000, 4096, 8191, 65536 + 5, 300_001, (1 << 21) + 3]


def run(xs, dtype, impl, in_place=False, h=None):
    n, N = len(xs), xs[0].size
    ins = upload_ranks(xs)
    outs = ins if in_place else empty_ranks(n, xs[0].nbytes)

    def call(handle):
        assert ar.ar_set_option(handle, ar.AR_OPT_TWO_SHOT_IMPL, impl) == ar.AR_OK
        rc = ar.ar_two_shot(handle, ptrs(ins), ptrs(outs), N, dtype)
        assert rc == ar.AR_OK, ar.ar_strerror(rc)
        assert ar.ar_status(handle) == ar.AR_OK
        assert ar.ar_traffic(handle).launches == (2 if impl == TWO_LAUNCHES else 1)

    if h is None:
        with Handle(n, max(16, N * E[dtype])) as handle:
            call(handle)
    else:
        call(h)
    torch.cuda.synchronize()
    for b in ins + outs:
        assert b.guards_intact()
    return [o.download(payload_np_dtype(dtype)) for o in outs]


@pytest.mark.parametrize("impl", FORMS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("N", SIZES)
def test_every_form_bit_exact(impl, dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal", seed=31 * n + N)
    want = oracle.all_reduce(xs, dtype)
    got = run(xs, dtype, impl)
    for r in range(n):
        np.testing.assert_array_equal(bits(got[r]), bits(want[r]), err_msg=f"impl {impl} rank {r}")


@pytest.mark.parametrize("impl", FORMS)
@pytest.mark.parametrize("n", [2, 8, 16])
def test_in_place(impl, n):
    N = 400_003
    xs = workloads.rank_inputs(n, N, "bf16", "normal_over_n", seed=50 + n)
    want = oracle.all_reduce(xs, "bf16")
    got = run(xs, "bf16", impl, in_place=True)
    for r in range(n):
        np.testing.assert_array_equal(got[r], want[r])


@pytest.mark.parametrize("impl", [ONE_LAUNCH, TILE_FLAGS])
@pytest.mark.parametrize("mib", [8, 16])
def test_one_launch_at_the_prefill_gate_sizes(impl, mib):
    # n = 8 bf16 at 8 and 16 MiB per rank (the prefill workload's sizes where the
    # HBM target is set), whole buffers against the oracle
    n, N = 8, mib * (1 << 20) // 2
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=1003 + mib)
    want = oracle.all_reduce(xs, "bf16")
    got = run(xs, "bf16", impl)
    for r in range(n):
        np.testing.assert_array_equal(got[r], want[r], err_msg=f"rank {r}")


@pytest.mark.parametrize("impl", [ONE_LAUNCH, TILE_FLAGS])
def test_repeated_calls_each_see_their_own_flags(impl):
    # the flags of one call must never release a tile of the next: five calls in a row on
    # one handle, new inputs each time, outputs reset to a sentinel in between
    n, N = 8, 1 << 20
    with Handle(n, N * 2, two_shot_impl=impl) as h:
        ins = upload_ranks(workloads.rank_inputs(n, N, "bf16", "normal", seed=0))
        outs = empty_ranks(n, N * 2)
        for k in range(5):
            xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=700 + k)
            for b, a in zip(ins, xs):
                b.upload(a)
            for o in outs:
                o.fill(0x5A)
            assert ar.ar_two_shot(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
            assert ar.ar_status(h) == ar.AR_OK
            want = oracle.all_reduce(xs, "bf16")
            for r in range(n):
                np.testing.assert_array_equal(outs[r].download(np.uint16), want[r], err_msg=f"call {k} rank {r}")


@pytest.mark.parametrize("impl", [ONE_LAUNCH, TILE_FLAGS])
def test_one_launch_in_a_cuda_graph(impl):
    # each replay is a new call: the call counter lives in device memory, so replays advance it
    n, N = 8, 300_001
    with Handle(n, N * 2, two_shot_impl=impl) as h:
        xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=11)
        ins = upload_ranks(xs)
        outs = empty_ranks(n, N * 2)
        s = torch.cuda.Stream()
        assert ar.ar_two_shot(h, ptrs(ins), ptrs(outs), N, "bf16", s) == ar.AR_OK   # outside capture first
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rc = ar.ar_two_shot(h, ptrs(ins), ptrs(outs), N, "bf16", s)
        assert rc == ar.AR_OK
        for k in range(3):
            src = workloads.rank_inputs(n, N, "bf16", "normal", seed=900 + k)
            for b, a in zip(ins, src):
                b.upload(a)
            for o in outs:
                o.fill(0x5A)
            g.replay()
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK
            want = oracle.all_reduce(src, "bf16")
            for r in range(n):
                np.testing.assert_array_equal(outs[r].download(np.uint16), want[r], err_msg=f"replay {k} rank {r}")


def test_a_wait_that_runs_out_is_reported_and_leaves_tiles_untouched():
    # a 1 ns limit makes the gathering CTAs' waits run out whenever a tile is not ready at
    # their first look; whatever happens, no GPU fault: the status is OK or AR_ERR_WAIT_TIMEOUT,
    # each output element is the right sum or the sentinel (reduced chunks themselves are always
    # written), and a call with the default limit afterwards is exact
    n, N = 8, 4 << 20
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=12)
    want = oracle.all_reduce(xs, "bf16")
    C = oracle.chunk_elems(n, N, "bf16")
    with Handle(n, N * 2, two_shot_impl=TILE_FLAGS, spin_ns=1) as h:
        ins = upload_ranks(xs)
        outs = empty_ranks(n, N * 2, byte=0x5A)
        assert ar.ar_two_shot(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
        st = ar.ar_status(h)
        assert st in (ar.AR_OK, ar.AR_ERR_WAIT_TIMEOUT)
        untouched = 0
        for r in range(n):
            got = outs[r].download(np.uint16)
            right = got == want[r]
            sentinel = got == 0x5A5A
            assert np.all(right | sentinel)
            own = slice(r * C, min((r + 1) * C, N))
            assert np.all(right[own]), "a rank's own reduced chunk is always written"
            untouched += int(np.count_nonzero(~right))
        if st == ar.AR_OK:
            assert untouched == 0
        for b in ins + outs:
            assert b.guards_intact()
        assert ar.ar_set_option(h, ar.AR_OPT_SPIN_NS, 1_000_000) == ar.AR_OK
        outs2 = empty_ranks(n, N * 2)
        assert ar.ar_two_shot(h, ptrs(ins), ptrs(outs2), N, "bf16") == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
        for r in range(n):
            np.testing.assert_array_equal(outs2[r].download(np.uint16), want[r])


def test_forms_report_their_launches_and_timing_records():
    n, N = 8, 1 << 20
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed=13)
    ins = upload_ranks(xs)
    outs = empty_ranks(n, N * 2)
    with Handle(n, N * 2, timing=8) as h:
        for impl, kernels in ((TWO_LAUNCHES, ["reduce_scatter", "all_gather"]), (ONE_LAUNCH, ["two_shot"]),
                              (TILE_FLAGS, ["two_shot"])):
            assert ar.ar_set_option(h, ar.AR_OPT_TWO_SHOT_IMPL, impl) == ar.AR_OK
            assert ar.ar_two_shot(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
            recs = ar.ar_timing(h)
            assert [r[0] for r in recs[-len(kernels):]] == kernels
            assert sum(r[3] for r in recs[-len(kernels):]) == (2 * n + 1) * N * 2
        assert ar.ar_set_option(h, ar.AR_OPT_TWO_SHOT_IMPL, 4) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_TWO_SHOT_IMPL, -1) == ar.AR_ERR_INVALID
