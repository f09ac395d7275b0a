"""Both launch forms of the streaming calls, at the size where one gives way
to the other.

A call too small to give every SM a full 256-thread CTA runs one 16-byte
vector per thread in narrower CTAs (a separately compiled small form of the
kernel); a larger call runs full CTAs, some with several vectors per thread.
Where the switch happens depends on the device's SM count, so the sizes are
computed from it here: the largest count that still takes the small form, the
next one, and one with a ragged tail just past it.  Each is compared with the
oracle bit for bit on every rank, with the buffers' guard bands intact."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Buf, Handle, bits, empty_ranks, payload_np_dtype, ptrs, upload_ranks

pytestmark = pytest.mark.gpu

E = {"f32": 4, "bf16": 2, "f16": 2}
THREADS = 256


def _sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def _unroll(n: int) -> int:
    # vectors per thread of the full-size one-shot, reduce-scatter and one-pass ring kernels
    return 4 if n <= 4 else 2 if n <= 8 else 1


def _counts(call: str, n: int, dtype: str) -> list[int]:
    """Counts just below, at and past the switch from the small form to full CTAs."""
    sm, ve = _sm_count(), 16 // E[dtype]
    if call in ("one_shot", "tree_fused"):
        u = _unroll(n) if call == "one_shot" else 1
        nvec = (sm - 1) * THREADS * u            # the most vectors that leave an SM without a full CTA
        return [nvec * ve + ve - 1, (nvec + 1) * ve, (nvec + 1) * ve + ve - 1]
    # two-shot and the one-pass ring: n rows (chunks) of C = ceil(N/n), rounded to a vector
    rows_max = -(-sm // n) - 1                   # full CTAs per row that still leave SMs idle
    cvec = rows_max * THREADS * _unroll(n)
    return [n * cvec * ve, n * cvec * ve + 1, n * (cvec + 1) * ve + 3]


CALLS = {
    "one_shot": (ar.ar_one_shot, oracle.all_reduce),
    "two_shot": (ar.ar_two_shot, oracle.all_reduce),
    "ring_fused": (ar.ar_ring_fused, oracle.ring),
    "tree_fused": (ar.ar_tree_fused, oracle.tree),
}


@pytest.mark.parametrize("call", list(CALLS))
@pytest.mark.parametrize("n,dtype", [(8, "bf16"), (4, "f32"), (16, "f16")])
@pytest.mark.parametrize("which", [0, 1, 2])
def test_small_and_full_forms_at_the_switch(call, n, dtype, which):
    N = _counts(call, n, dtype)[which]
    fn, ref = CALLS[call]
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=31 * n + which)
    ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
    with Handle(n, N * E[dtype]) as h:
        assert fn(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    want = ref(xs, dtype)
    for r in range(n):
        np.testing.assert_array_equal(bits(outs[r].download(payload_np_dtype(dtype))), bits(want[r]),
                                      err_msg=f"{call} n={n} N={N} rank {r}")
    for b in ins + outs:
        assert b.guards_intact()


@pytest.mark.parametrize("kind", ["ll", "ll128"])
@pytest.mark.parametrize("which", [0, 1, 2])
def test_ll_reduce_forms_at_the_switch(kind, which):
    # the flag-checked reduce: one thread per 16 bytes of lines (two LL lines, or one 8-lane slot of
    # an LL128 line), narrowed when it holds a full CTA of work but full CTAs would leave SMs idle
    n, sm = 8, _sm_count()
    work = (sm - 1) * THREADS                    # threads of work that still take the narrow form
    if kind == "ll":
        counts = [2 * work - 1, 2 * work + 1, 2 * work + 7]
    else:
        lines = work // 8
        counts = [30 * lines - 7, 30 * lines + 1, 30 * lines + 29]
    count = counts[which]
    xs = workloads.payload_f32(n, count, seed=workloads.seed_of(4) + 7 * which)
    o_pack = oracle.ll_pack if kind == "ll" else oracle.ll128_pack
    o_reduce = oracle.ll_reduce if kind == "ll" else oracle.ll128_reduce
    reduce = ar.ar_ll_reduce if kind == "ll" else ar.ar_ll128_reduce
    step = 5
    packed = [o_pack(x, step) for x in xs]
    lines_in = [Buf(p.nbytes).upload(p) for p in packed]
    lines_out = [Buf(p.nbytes).fill(0) for p in packed]
    with Handle(n, 4 * count) as h:
        assert reduce(h, ptrs(lines_in), ptrs(lines_out), count, step) == ar.AR_OK
        assert ar.ar_status(h) == ar.AR_OK
    want, bad = o_reduce(packed, count, step)
    assert bad == 0
    for o, w in zip(lines_out, want):
        np.testing.assert_array_equal(o.download(np.uint8), w)
    for b in lines_in + lines_out:
        assert b.guards_intact()


@pytest.mark.parametrize("cap", [1, 2])
@pytest.mark.parametrize("call", list(CALLS))
def test_small_forms_under_a_cta_cap(call, cap):
    # AR_OPT_CTAS_PER_SM bounds every launch, the narrowed small forms included: with one or two
    # CTAs per SM allowed the small calls still cover every element, bit for bit
    n, dtype = 8, "bf16"
    for N in (7, 4099, _counts(call, n, dtype)[0]):
        xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=53 * cap + N)
        ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
        fn, ref = CALLS[call]
        with Handle(n, max(16, N * E[dtype]), ctas_per_sm=cap) as h:
            assert fn(h, ptrs(ins), ptrs(outs), N, dtype) == ar.AR_OK
            assert ar.ar_status(h) == ar.AR_OK
        torch.cuda.synchronize()
        want = ref(xs, dtype)
        for r in (0, n - 1):
            np.testing.assert_array_equal(bits(outs[r].download(np.uint16)), bits(want[r]),
                                          err_msg=f"{call} cap={cap} N={N}")
        for b in ins + outs:
            assert b.guards_intact()
