"""ar_ring_persistent: the whole ring in one cooperative launch, hops carried
as LL128 lines with per-step flags ("集合通信：NCCL 的算法、协议与推理框架的
定制 all-reduce", §协议; "多 GPU 与 NCCL", §ring all-reduce).

Its sums are ar_ring's (fp32 partials, chunk c summed from rank c), so every
output is compared bit for bit with the oracle's ring.  Cases span one and
many 32-line batches per warp, several CTAs per rank, ragged chunks and empty
chunks; repeated calls on one handle check that no line of an earlier call is
taken for the current one.  The failure cases emulate a rank that never joins
(AR_OPT_ABSENT_RANK): its neighbours' bounded waits run out, the status says
so, and the next call on the same handle succeeds."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Buf, Handle, bits, empty_ranks, payload_np_dtype, ptrs, upload_ranks

pytestmark = pytest.mark.gpu

E = {"f32": 4, "bf16": 2, "f16": 2}


def _run(xs, dtype, h, in_place=False):
    n, N = len(xs), xs[0].size
    ins = upload_ranks(xs)
    outs = ins if in_place else empty_ranks(n, xs[0].nbytes)
    rc = ar.ar_ring_persistent(h, ptrs(ins), ptrs(outs), N, dtype)
    assert rc == ar.AR_OK, ar.ar_strerror(rc)
    torch.cuda.synchronize()
    assert ar.ar_status(h) == ar.AR_OK
    for b in ins + outs:
        assert b.guards_intact()
    return [o.download(payload_np_dtype(dtype)) for o in outs]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n,N", [(2, 1), (2, 9), (3, 1000), (8, 4099), (8, 7680 * 8 + 3), (5, 300_001),
                                 (16, 65536 + 3), (16, 17), (8, 2_000_003)])
def test_persistent_ring_matches_the_ring_oracle(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=11 * n + N)
    want = oracle.ring(xs, dtype)
    with Handle(n, max(16, N * E[dtype]), persistent=1) as h:
        got = _run(xs, dtype, h)
        t = ar.ar_traffic(h)
        assert t.op == ar.AR_OP_RING_PERSISTENT and t.launches == 1
    for r in range(n):
        np.testing.assert_array_equal(bits(got[r]), bits(want[r]))


@pytest.mark.parametrize("ctas_per_sm", [1, 2])
def test_persistent_ring_few_ctas_many_batches(ctas_per_sm):
    # few CTAs per rank: every warp loops over many batches and the inbox
    # slots are reused step after step, so the acknowledgements are waited on
    n, N, dtype = 8, 3_000_017, "bf16"
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=ctas_per_sm)
    want = oracle.ring(xs, dtype)
    with Handle(n, N * 2, persistent=1, ctas_per_sm=ctas_per_sm) as h:
        got = _run(xs, dtype, h)
    for r in range(n):
        np.testing.assert_array_equal(got[r], want[r])


def test_persistent_ring_in_place_and_repeated_calls():
    # one handle, several calls of different sizes: each call's flags are new,
    # so a line left by an earlier call is never consumed
    n = 8
    with Handle(n, 2 * 400_000, persistent=1) as h:
        for i, N in enumerate([400_000, 1000, 400_000, 123_457, 8]):
            xs = workloads.rank_inputs(n, N, "bf16", "normal_over_n", seed=100 + i)
            got = _run(xs, "bf16", h, in_place=(i % 2 == 1))
            want = oracle.ring(xs, "bf16")
            for r in range(n):
                np.testing.assert_array_equal(got[r], want[r])


def test_persistent_ring_equals_ar_ring_at_a_large_size():
    n, N, dtype = 8, 8 * 1024 * 1024 + 5, "bf16"
    gen = torch.Generator(device="cuda")
    ins = []
    for r in range(n):
        gen.manual_seed(7000 + r)
        b = Buf(N * 2)
        b.body().view(torch.bfloat16).copy_(torch.randn(N, generator=gen, device="cuda").to(torch.bfloat16) / n)
        ins.append(b)
    a, p = empty_ranks(n, N * 2), empty_ranks(n, N * 2)
    with Handle(n, N * 2, persistent=1) as h:
        assert ar.ar_ring(h, ptrs(ins), ptrs(a), N, dtype) == ar.AR_OK
        assert ar.ar_ring_persistent(h, ptrs(ins), ptrs(p), N, dtype) == ar.AR_OK
        torch.cuda.synchronize()
        assert ar.ar_status(h) == ar.AR_OK
    for r in range(n):
        assert torch.equal(a[r].body(), p[r].body())


def _persist_pieces(n, N, dtype):
    """Pieces of a persistent ring call: the two inbox slots of a step (128-byte lines of 30
    words, all ranks' chunks) over half of this device's L2, rounded, at most 64."""
    half = torch.cuda.get_device_properties(0).L2_cache_size // 2
    C = oracle.chunk_elems(n, N, dtype)
    lines = sum(-(-max(0, min(C, N - c * C)) // 30) for c in range(n))
    return min(64, max(1, (2 * 128 * lines + half // 2) // half))


@pytest.mark.parametrize("n,N,dtype,ctas_per_sm,in_place", [
    (8, 16 * 1024 * 1024 + 5, "bf16", 0, False), (8, 32 * 1024 * 1024 + 3, "bf16", 0, False),
    (4, 12_000_007, "f32", 0, False), (16, 24_000_001, "f16", 0, False),
    (8, 16 * 1024 * 1024 + 5, "bf16", 1, False), (8, 16 * 1024 * 1024 + 5, "bf16", 0, True)])
def test_persistent_ring_in_pieces_equals_ar_ring(n, N, dtype, ctas_per_sm, in_place):
    # calls whose inbox traffic exceeds L2 run their CTAs' slices in pieces (every piece through
    # all 2(n-1) steps, the flags numbering the messages across pieces): every element of every
    # rank equal to ar_ring's, on two calls of one handle; one CTA per SM gives every warp many
    # batches per piece (the slot acknowledgements are waited on), and in place each piece's
    # outputs overwrite inputs that only that piece reads
    assert _persist_pieces(n, N, dtype) >= 2
    e = E[dtype]
    iv = torch.int16 if e == 2 else torch.int32
    ins = workloads.rank_inputs_device(n, N, dtype, "normal_over_n", workloads.seed_of(9) + n)
    keep = [t.clone() for t in ins]
    a = [torch.empty_like(t) for t in ins]
    opts = {"persistent": 1, **({"ctas_per_sm": ctas_per_sm} if ctas_per_sm else {})}
    with Handle(n, N * e, **opts) as h:
        ptr = lambda ts: [t.data_ptr() for t in ts]
        assert ar.ar_ring(h, ptr(ins), ptr(a), N, dtype) == ar.AR_OK
        for k in range(2):
            for t, x in zip(ins, keep):
                t.copy_(x)
            p = ins if in_place else [torch.zeros_like(t) for t in ins]
            assert ar.ar_ring_persistent(h, ptr(ins), ptr(p), N, dtype) == ar.AR_OK
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK
            for r in range(n):
                assert torch.equal(a[r].view(iv), p[r].view(iv)), (k, r)


def test_persistent_ring_in_pieces_in_a_cuda_graph_against_the_oracle():
    # captured once and replayed on new inputs: every replay has its own call number, so no line
    # of an earlier replay or piece is taken; every element against the oracle's ring
    n, N, dtype = 8, 12 * 1024 * 1024 + 77, "bf16"
    assert _persist_pieces(n, N, dtype) >= 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal_over_n", workloads.seed_of(9) + 100)
    outs = [torch.empty_like(t) for t in ins]
    with Handle(n, N * 2, persistent=1) as h:
        s = torch.cuda.Stream()
        assert ar.ar_ring_persistent(h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs],
                                     N, dtype) == ar.AR_OK
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rc = ar.ar_ring_persistent(h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], N, dtype, s)
        assert rc == ar.AR_OK
        for k in range(2):
            src = workloads.rank_inputs_device(n, N, dtype, "normal_over_n", workloads.seed_of(9) + 101 + k)
            for t, x in zip(ins, src):
                t.copy_(x)
            for o in outs:
                o.fill_(0x5A5A)
            g.replay()
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK
            want = oracle.ring([t.cpu().numpy().view(np.uint16) for t in ins], dtype)[0]
            for r in range(n):
                bad = np.flatnonzero(outs[r].cpu().numpy().view(np.uint16) != want)
                assert bad.size == 0, (k, r, bad[:5])


def test_persistent_ring_needs_its_buffers_and_rejects_bad_options():
    with Handle(4, 4096) as h:
        ins, outs = empty_ranks(4, 4096), empty_ranks(4, 4096)
        assert ar.ar_ring_persistent(h, ptrs(ins), ptrs(outs), 100, "f32") == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_PERSISTENT, 2) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_ABSENT_RANK, 4) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_ABSENT_RANK, -2) == ar.AR_ERR_INVALID
        assert ar.ar_set_option(h, ar.AR_OPT_PERSISTENT, 1) == ar.AR_OK
        assert ar.ar_ring_persistent(h, ptrs(ins), ptrs(outs), 100, "f32") == ar.AR_OK
        assert ar.ar_set_option(h, ar.AR_OPT_PERSISTENT, 0) == ar.AR_OK
        assert ar.ar_ring_persistent(h, ptrs(ins), ptrs(outs), 100, "f32") == ar.AR_ERR_INVALID
        assert ar.ar_status(h) == ar.AR_OK


def test_persistent_ring_timing_record():
    n, N = 4, 100_000
    xs = workloads.rank_inputs(n, N, "f32", "normal", seed=5)
    with Handle(n, N * 4, persistent=1, timing=16) as h:
        _run(xs, "f32", h)
        recs = ar.ar_timing(h)
    assert [r[0] for r in recs] == ["ring_persistent"]
    assert recs[0][3] == ar.ar_plan(ar.AR_OP_RING_PERSISTENT, n, N, "f32").hbm_read_bytes * 2


@pytest.mark.parametrize("absent", [0, 3])
def test_persistent_ring_absent_rank_times_out_and_the_handle_stays_usable(absent):
    # rank `absent` never joins: its successor waits for lines that never come
    # and its predecessor for acknowledgements that never come; both waits
    # are bounded
    n, N = 4, 200_000
    xs = workloads.rank_inputs(n, N, "f32", "normal", seed=9)
    ins, outs = upload_ranks(xs), empty_ranks(n, N * 4)
    with Handle(n, N * 4, persistent=1, spin_ns=200_000, absent_rank=absent) as h:
        assert ar.ar_ring_persistent(h, ptrs(ins), ptrs(outs), N, "f32") == ar.AR_OK
        torch.cuda.synchronize()
        rc, info = ar.ar_status_info(h)
        assert rc in (ar.AR_ERR_FLAG_TIMEOUT, ar.AR_ERR_WAIT_TIMEOUT)
        assert info.code == rc
        assert ar.ar_status(h) == ar.AR_OK   # read once, then cleared
        # the same handle, every rank present again: a clean call
        assert ar.ar_set_option(h, ar.AR_OPT_ABSENT_RANK, -1) == ar.AR_OK
        got = _run(xs, "f32", h)
    want = oracle.ring(xs, "f32")
    for r in range(n):
        np.testing.assert_array_equal(got[r], want[r])


# --- the same ring over a thread-block cluster (ar_ring_cluster) -------------

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n,N", [(2, 1), (2, 9), (3, 1000), (5, 300_001), (8, 4099), (8, 7680 * 8 + 3),
                                 (16, 65536 + 3), (16, 17), (8, 2_000_003)])
def test_cluster_ring_matches_the_ring_oracle(dtype, n, N):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=13 * n + N)
    want = oracle.ring(xs, dtype)
    ins, outs = upload_ranks(xs), empty_ranks(n, xs[0].nbytes)
    with Handle(n, max(16, N * E[dtype])) as h:
        rc = ar.ar_ring_cluster(h, ptrs(ins), ptrs(outs), N, dtype)
        assert rc == ar.AR_OK, ar.ar_strerror(rc)
        torch.cuda.synchronize()
        assert ar.ar_status(h) == ar.AR_OK
        t = ar.ar_traffic(h)
        assert t.op == ar.AR_OP_RING_CLUSTER and t.launches == 1
    for b in ins + outs:
        assert b.guards_intact()
    for r in range(n):
        np.testing.assert_array_equal(bits(outs[r].download(payload_np_dtype(dtype))), bits(want[r]))


def test_cluster_ring_in_place_repeated_and_equal_to_the_step_ring():
    n = 8
    with Handle(n, 2 * 3_000_017) as h:
        for i, N in enumerate([3_000_017, 1000, 400_000, 8]):
            xs = workloads.rank_inputs(n, N, "bf16", "normal_over_n", seed=200 + i)
            ins = upload_ranks(xs)
            outs = ins if i % 2 else empty_ranks(n, xs[0].nbytes)
            assert ar.ar_ring_cluster(h, ptrs(ins), ptrs(outs), N, "bf16") == ar.AR_OK
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK
            want = oracle.ring(xs, "bf16")
            for r in range(n):
                np.testing.assert_array_equal(outs[r].download(np.uint16), want[r])


@pytest.mark.parametrize("absent", [0, 5])
def test_cluster_ring_absent_rank_times_out_and_the_handle_stays_usable(absent):
    n, N = 8, 200_000
    xs = workloads.rank_inputs(n, N, "f32", "normal", seed=19)
    ins, outs = upload_ranks(xs), empty_ranks(n, N * 4)
    with Handle(n, N * 4, spin_ns=200_000, absent_rank=absent) as h:
        assert ar.ar_ring_cluster(h, ptrs(ins), ptrs(outs), N, "f32") == ar.AR_OK
        torch.cuda.synchronize()
        rc, info = ar.ar_status_info(h)
        assert rc in (ar.AR_ERR_FLAG_TIMEOUT, ar.AR_ERR_WAIT_TIMEOUT)
        assert ar.ar_status(h) == ar.AR_OK
        assert ar.ar_set_option(h, ar.AR_OPT_ABSENT_RANK, -1) == ar.AR_OK
        assert ar.ar_ring_cluster(h, ptrs(ins), ptrs(outs), N, "f32") == ar.AR_OK
        torch.cuda.synchronize()
        assert ar.ar_status(h) == ar.AR_OK
    want = oracle.ring(xs, "f32")
    for r in range(n):
        np.testing.assert_array_equal(outs[r].download(np.float32), want[r])


def test_cluster_ring_timing_record_and_plan():
    n, N = 4, 100_000
    xs = workloads.rank_inputs(n, N, "f32", "normal", seed=21)
    ins, outs = upload_ranks(xs), empty_ranks(n, N * 4)
    with Handle(n, N * 4, timing=16) as h:
        assert ar.ar_ring_cluster(h, ptrs(ins), ptrs(outs), N, "f32") == ar.AR_OK
        recs = ar.ar_timing(h)
    assert [r[0] for r in recs] == ["ring_cluster"]
    t = ar.ar_plan(ar.AR_OP_RING_CLUSTER, n, N, "f32")
    assert recs[0][3] == t.hbm_read_bytes + t.hbm_write_bytes == 2 * n * N * 4


@pytest.mark.parametrize("n,N,dtype", [(2, 16 << 20, "bf16"), (8, 32 << 20, "bf16"), (8, 8 << 20, "f32"),
                                       (4, 16 << 20, "f16"), (16, 4 << 20, "bf16")])
def test_cluster_ring_large_slices(n, N, dtype):
    # sizes where one wave of clusters would give a warp many batches per step: the slices
    # are capped so that a step's batches fit the inbox, the calls run in several waves, and
    # every inbox slot is reused many times (fp32 lines in every hop for f32, payload-type
    # all-gather hops for 16-bit data)
    ins = workloads.rank_inputs_device(n, N, dtype, "normal_over_n", 4321 + n)
    a = [torch.empty_like(t) for t in ins]
    c = [torch.empty_like(t) for t in ins]
    h = ar.ar_create(n, E[dtype] * N)
    try:
        assert ar.ar_ring(h, [t.data_ptr() for t in ins], [t.data_ptr() for t in a], N, dtype) == ar.AR_OK
        assert ar.ar_ring_cluster(h, [t.data_ptr() for t in ins], [t.data_ptr() for t in c], N, dtype) == ar.AR_OK
        torch.cuda.synchronize()
        assert ar.ar_status(h) == ar.AR_OK
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK
    for r in range(n):
        assert torch.equal(a[r], c[r])
