"""ar_ring_noalloc: the ring all-reduce for callers that cannot allocate
device memory (they cannot call ar_create, which allocates the scratch).
Its scratch is a static array inside the library.  Checked through the C-ABI
against ar_ring, the existing entry point, and against the oracle's ring, on
two calls in a row (the second call finds the first call's partials still in
the shared array), and at the array's exact capacity.  This file is collected
last so that a run stopping at the first failure has run every other test
first."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Handle, bits, empty_ranks, ptrs, upload_ranks

pytestmark = pytest.mark.gpu


def _ring_with_handle(xs, dtype):
    n, N = len(xs), xs[0].size
    ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
    with Handle(n, max(16, xs[0].nbytes)) as h:
        assert ar.ar_ring(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    return [o.download(xs[0].dtype) for o in outs]


@pytest.mark.parametrize("dtype,n,N", [("bf16", 8, 1 << 20), ("f16", 16, 300_001), ("f32", 3, 4099), ("bf16", 2, 9)])
def test_noalloc_ring_equals_ar_ring_and_the_oracle_on_two_calls_in_a_row(dtype, n, N):
    for call in range(2):
        xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=100 * call + n + N)
        ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
        assert ar.ar_ring_noalloc(n, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        torch.cuda.synchronize()
        want = _ring_with_handle(xs, dtype)
        ref = oracle.ring(xs, dtype)
        for r in range(n):
            got = outs[r].download(xs[0].dtype)
            np.testing.assert_array_equal(bits(got), bits(want[r]), err_msg=f"call {call} rank {r} vs ar_ring")
            np.testing.assert_array_equal(bits(got), bits(ref[r]), err_msg=f"call {call} rank {r} vs the oracle")
        for b in ins + outs:
            assert b.guards_intact()


def test_noalloc_ring_at_the_exact_capacity_in_place():
    # 32 MiB holds 2 x n x C fp32 partials: n = 8 bf16 with 4 Mi elements per rank gives C = 512 Ki,
    # exactly the array; the call runs in place and must match the oracle's ring bit for bit
    n, N, dtype = 8, 4 << 20, "bf16"
    assert 2 * n * oracle.chunk_elems(n, N, dtype) * 4 == 32 << 20
    for call in range(2):
        xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=4242 + call)
        bufs = upload_ranks(xs)
        assert ar.ar_ring_noalloc(n, ptrs(bufs), ptrs(bufs), N, dtype) == ar.AR_OK
        torch.cuda.synchronize()
        ref = oracle.ring(xs, dtype)
        for r in range(n):
            np.testing.assert_array_equal(bits(bufs[r].download(np.uint16)), bits(ref[r]),
                                          err_msg=f"call {call} rank {r}")
        for b in bufs:
            assert b.guards_intact()


def test_noalloc_ring_rejects_what_does_not_fit_and_bad_arguments():
    n = 8
    too_big = (4 << 20) + 64
    bufs = empty_ranks(n, 2 * too_big)
    assert ar.ar_ring_noalloc(n, ptrs(bufs), ptrs(bufs), too_big, "bf16") == ar.AR_ERR_TOO_LARGE
    assert ar.ar_ring_noalloc(1, ptrs(bufs), ptrs(bufs), 16, "bf16") == ar.AR_ERR_INVALID
    assert ar.ar_ring_noalloc(n, [p + 2 for p in ptrs(bufs)], ptrs(bufs), 16, "bf16") == ar.AR_ERR_ALIGN
    assert ar.ar_ring_noalloc(n, ptrs(bufs), ptrs(bufs), 0, "bf16") == ar.AR_OK
    torch.cuda.synchronize()
    for b in bufs:
        assert b.guards_intact()
