"""Full-size parity: the prefill workload (n = 8 bf16, 8..64 MiB per rank)
in the launch configuration the bench times, and the n = 16 sweep's largest
sizes.  The oracle computes sampled outputs one by one; properties that hold
at any size (every rank identical, two-shot == one-shot bit for bit) cover
the rest of each buffer."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads

pytestmark = pytest.mark.gpu

MiB = 1 << 20


def _sample_idx(N, C, rng, k=100_000):
    edges = []
    for c in range(0, N, max(C, 1)):          # chunk boundaries and the ragged end
        edges += [c - 1, c, c + 1]
    idx = np.concatenate([rng.integers(0, N, size=k), np.arange(min(N, 4096)),
                          np.arange(max(0, N - 4096), N), np.array(edges)])
    return np.unique(idx[(idx >= 0) & (idx < N)])


def _cols(ts, idx, dtype):
    ti = torch.from_numpy(idx).to(ts[0].device)
    np_t = np.float32 if dtype == "f32" else np.uint16
    return [t[ti].cpu().numpy().view(np_t) for t in ts]


def _ring_pieces(n, N, dtype, rounded):
    """Pieces of a ring call: a step's partials (fp32, or the payload when rounded per hop) over
    half of this device's L2, rounded, at most 64; each chunk cut into that many pieces of whole
    256-element blocks; twice as many (half the length) when the partials reach a tenth of L2
    and the call runs on two streams."""
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    half = l2 // 2
    pe = {"f32": 4, "bf16": 2, "f16": 2}[dtype] if rounded else 4
    P = min(64, max(1, (N * pe + half // 2) // half))
    C = oracle.chunk_elems(n, N, dtype)
    PL = C if P == 1 else min(C, -(-(-(-C // P)) // 256) * 256)
    if N * pe * 10 >= l2:
        PL = min(C, -(-(-(-PL // 2)) // 256) * 256)
    return -(-C // PL)


def _run(call, h, ins, outs, N, dtype):
    rc = call(h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], N, dtype)
    assert rc == ar.AR_OK, ar.ar_strerror(rc)


@pytest.mark.parametrize("S", [8 * MiB, 64 * MiB])
def test_prefill_one_and_two_shot(S):
    n, dtype = 8, "bf16"
    N = S // 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal", workloads.seed_of(3) + S)
    o1 = [torch.empty_like(t) for t in ins]
    o2 = [torch.empty_like(t) for t in ins]
    with_h = ar.ar_create(n, S)
    try:
        _run(ar.ar_one_shot, with_h, ins, o1, N, dtype)
        _run(ar.ar_two_shot, with_h, ins, o2, N, dtype)
        assert ar.ar_status(with_h) == ar.AR_OK
    finally:
        assert ar.ar_destroy(with_h) == ar.AR_OK
    for r in range(1, n):
        assert torch.equal(o1[r], o1[0]) and torch.equal(o2[r], o2[0])
    assert torch.equal(o1[0], o2[0])
    idx = _sample_idx(N, oracle.chunk_elems(n, N, dtype), np.random.default_rng(S))
    want = oracle.all_reduce(_cols(ins, idx, dtype), dtype)[0]
    np.testing.assert_array_equal(_cols([o1[0]], idx, dtype)[0], want)


@pytest.mark.parametrize("dtype,S", [("bf16", 256 * MiB), ("f16", 64 * MiB)])
def test_n16_sweep_largest(dtype, S):
    n = 16
    N = S // 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal_over_n", workloads.seed_of(5) + S)
    out_r = [torch.empty_like(t) for t in ins]
    out_1 = [torch.empty_like(t) for t in ins]
    h = ar.ar_create(n, S)
    try:
        _run(ar.ar_ring, h, ins, out_r, N, dtype)
        _run(ar.ar_one_shot, h, ins, out_1, N, dtype)
        assert ar.ar_status(h) == ar.AR_OK
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK
    for r in range(1, n):
        assert torch.equal(out_r[r], out_r[0]) and torch.equal(out_1[r], out_1[0])
    C = oracle.chunk_elems(n, N, dtype)
    idx = _sample_idx(N, C, np.random.default_rng(S + 1))
    cols = _cols(ins, idx, dtype)
    want_ring = oracle.ring_order_sum(cols, (idx // C).astype(np.int32), dtype)
    np.testing.assert_array_equal(_cols([out_r[5]], idx, dtype)[0], want_ring)
    want_one = oracle.all_reduce(cols, dtype)[0]
    np.testing.assert_array_equal(_cols([out_1[9]], idx, dtype)[0], want_one)
    del ins, out_r, out_1
    torch.cuda.empty_cache()


def test_ll_largest_payload_in_the_bench_configuration():
    n, count = 8, (1 * MiB) // 4
    xs = workloads.rank_inputs_device(n, count, "f32", "uniform", workloads.seed_of(4))
    h = ar.ar_create(n, 4 * count)
    try:
        for kind in ("ll", "ll128"):
            nb = ar.ar_ll_bytes(4 * count) if kind == "ll" else ar.ar_ll128_bytes(4 * count)
            pack = ar.ar_ll_pack if kind == "ll" else ar.ar_ll128_pack
            reduce = ar.ar_ll_reduce if kind == "ll" else ar.ar_ll128_reduce
            unpack = ar.ar_ll_unpack if kind == "ll" else ar.ar_ll128_unpack
            lines = [torch.zeros(nb, dtype=torch.uint8, device="cuda") for _ in range(n)]
            outs = [torch.zeros(nb, dtype=torch.uint8, device="cuda") for _ in range(n)]
            dst = [torch.zeros(count, dtype=torch.float32, device="cuda") for _ in range(n)]
            for step in (11, 12):
                for x, l in zip(xs, lines):
                    assert pack(h, x.data_ptr(), l.data_ptr(), count, step) == ar.AR_OK
                assert reduce(h, [l.data_ptr() for l in lines], [o.data_ptr() for o in outs], count, step) == 0
                for o, d in zip(outs, dst):
                    assert unpack(h, o.data_ptr(), d.data_ptr(), count, step) == ar.AR_OK
                assert ar.ar_status(h) == ar.AR_OK
                want = oracle.all_reduce([x.cpu().numpy() for x in xs], "f32")[0]
                for d in dst:
                    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint32), want.view(np.uint32))
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK


def test_other_calls_at_the_prefill_size():
    # n = 8 bf16, 64 MiB per rank, in the configuration the bench's variants
    # leg times: push and copy-in == one-shot and the persistent ring == the
    # step ring, all bit for bit over whole buffers; the hop-rounded ring and
    # the tree against the oracle over whole buffers
    n, dtype, S = 8, "bf16", 64 * MiB
    N = S // 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal_over_n", workloads.seed_of(3) + 77)
    outs = {k: [torch.empty_like(t) for t in ins] for k in
            ("one_shot", "push", "copyin", "ring", "persistent", "rounded", "tree")}
    h = ar.ar_create(n, S)
    try:
        for opt in (ar.AR_OPT_PUSH_STAGING, ar.AR_OPT_REGISTERED, ar.AR_OPT_PERSISTENT):
            assert ar.ar_set_option(h, opt, 1) == ar.AR_OK
        for key, call in (("one_shot", ar.ar_one_shot), ("push", ar.ar_one_shot_push),
                          ("copyin", ar.ar_one_shot_copyin), ("ring", ar.ar_ring),
                          ("persistent", ar.ar_ring_persistent), ("rounded", ar.ar_ring_rounded),
                          ("tree", ar.ar_tree)):
            _run(call, h, ins, outs[key], N, dtype)
        torch.cuda.synchronize()
        assert ar.ar_status(h) == ar.AR_OK
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK
    for r in range(n):
        assert torch.equal(outs["push"][r], outs["one_shot"][r])
        assert torch.equal(outs["copyin"][r], outs["one_shot"][r])
        assert torch.equal(outs["persistent"][r], outs["ring"][r])
    host = [t.cpu().numpy().view(np.uint16) for t in ins]
    want_rounded = oracle.ring_rounded(host, dtype)
    want_tree = oracle.tree(host, dtype)
    for r in (0, 3, 7):
        np.testing.assert_array_equal(outs["rounded"][r].cpu().numpy().view(np.uint16), want_rounded[r])
        np.testing.assert_array_equal(outs["tree"][r].cpu().numpy().view(np.uint16), want_tree[r])


def test_fused_rings_at_the_prefill_size():
    # n = 8 bf16, 64 MiB per rank: the one-pass rings against the oracle's
    # ring orders over whole buffers, and equal to the step-by-step rings
    n, dtype, S = 8, "bf16", 64 * MiB
    N = S // 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal_over_n", workloads.seed_of(3) + 78)
    outs = {k: [torch.empty_like(t) for t in ins] for k in ("fused", "ring", "rounded_fused", "rounded")}
    h = ar.ar_create(n, S)
    try:
        for key, call in (("fused", ar.ar_ring_fused), ("ring", ar.ar_ring),
                          ("rounded_fused", ar.ar_ring_rounded_fused), ("rounded", ar.ar_ring_rounded)):
            _run(call, h, ins, outs[key], N, dtype)
        torch.cuda.synchronize()
        assert ar.ar_status(h) == ar.AR_OK
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK
    for r in range(n):
        assert torch.equal(outs["fused"][r], outs["ring"][r])
        assert torch.equal(outs["rounded_fused"][r], outs["rounded"][r])
    host = [t.cpu().numpy().view(np.uint16) for t in ins]
    want, want_rounded = oracle.ring(host, dtype), oracle.ring_rounded(host, dtype)
    for r in (0, 4, 7):
        np.testing.assert_array_equal(outs["fused"][r].cpu().numpy().view(np.uint16), want[r])
        np.testing.assert_array_equal(outs["rounded_fused"][r].cpu().numpy().view(np.uint16), want_rounded[r])


def test_prefill_64mib_whole_buffers_against_the_oracle():
    # the bench's own size, n = 8 bf16 at 64 MiB per rank, every element of every rank's output
    # against the oracle: one-shot and two-shot (the default, one launch) against the rank-order
    # sum, the step ring and the cluster ring against the ring's order
    n, dtype, S = 8, "bf16", 64 * MiB
    N = S // 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal", workloads.seed_of(3) + 7)
    xs = [t.cpu().numpy().view(np.uint16) for t in ins]
    want_sum = oracle.all_reduce(xs, dtype)[0]
    want_ring = oracle.ring(xs, dtype)[0]
    outs = [torch.empty_like(t) for t in ins]
    h = ar.ar_create(n, S)
    try:
        for call, want in ((ar.ar_one_shot, want_sum), (ar.ar_two_shot, want_sum), (ar.ar_ring, want_ring),
                           (ar.ar_ring_cluster, want_ring)):
            for o in outs:
                o.fill_(0x5A5A)
            _run(call, h, ins, outs, N, dtype)
            assert ar.ar_status(h) == ar.AR_OK
            for r in range(n):
                got = outs[r].cpu().numpy().view(np.uint16)
                bad = np.flatnonzero(got != want)
                assert bad.size == 0, (call.__name__, r, bad[:5])
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK


@pytest.mark.parametrize("dtype,n,N,call,ref", [
    ("f32", 4, (16 << 20) + 3, "ar_ring", "ring"),
    ("f16", 3, (32 << 20) + 5, "ar_ring", "ring"),
    ("bf16", 4, (40 << 20) + 1, "ar_ring_rounded", "ring_rounded"),
])
def test_ring_steps_in_the_l2_order_whole_buffers(dtype, n, N, call, ref):
    # sizes whose step data (fp32 partials, or the payload when rounded per hop) exceeds half of
    # L2, so the steps take their tiles in the reversed, rotated order, keep their partials in
    # L2 with write-back stores and streaming last-use loads, and (f16 here) run in pieces:
    # every element of every rank against the oracle, with ragged chunk ends, and the launches
    # the documented piece rule gives
    ins = workloads.rank_inputs_device(n, N, dtype, "normal", workloads.seed_of(5) + n)
    np_t = np.float32 if dtype == "f32" else np.uint16
    xs = [t.cpu().numpy().view(np_t) for t in ins]
    want = getattr(oracle, ref)(xs, dtype)[0]
    outs = [torch.empty_like(t) for t in ins]
    h = ar.ar_create(n, N * ins[0].element_size())
    try:
        for rep in range(2):   # the second call finds the first call's partials in the scratch
            for o in outs:
                o.fill_(0x5A5A if dtype != "f32" else 7.0)
            _run(getattr(ar, call), h, ins, outs, N, dtype)
            assert ar.ar_status(h) == ar.AR_OK
            assert ar.ar_traffic(h).launches == 2 * (n - 1) * _ring_pieces(n, N, dtype, call == "ar_ring_rounded")
            for r in range(n):
                got = outs[r].cpu().numpy().view(np_t)
                bad = np.flatnonzero(got.view(np.uint32 if dtype == "f32" else np.uint16)
                                     != want.view(np.uint32 if dtype == "f32" else np.uint16))
                assert bad.size == 0, (call, rep, r, bad[:5])
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK


@pytest.mark.parametrize("n,N,dtype", [(8, 8 << 20, "bf16"), (4, (10 << 20) + 3, "f32"), (16, (8 << 20) + 5, "f16")])
def test_tree_in_pieces_whole_buffers(n, N, dtype):
    # a level's output (n S) over half of L2: the tree runs piece by piece through its levels, on
    # two streams; every element of every rank against the oracle's tree, and the launches the
    # piece rule gives
    e = 4 if dtype == "f32" else 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal", workloads.seed_of(5) + 100 + n)
    np_t = np.float32 if dtype == "f32" else np.uint16
    bits_t = np.uint32 if dtype == "f32" else np.uint16
    xs = [t.cpu().numpy().view(np_t) for t in ins]
    want = oracle.tree(xs, dtype)[0].view(bits_t)
    outs = [torch.empty_like(t) for t in ins]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    half = l2 // 2
    P = min(64, max(1, (n * N * e + half // 2) // half))
    PL = N if P == 1 else min(N, -(-(-(-N // P)) // 256) * 256)
    if n * N * e * 2 >= l2:   # two streams: twice the pieces
        PL = min(N, -(-(-(-PL // 2)) // 256) * 256)
    h = ar.ar_create(n, N * e)
    try:
        _run(ar.ar_tree, h, ins, outs, N, dtype)
        assert ar.ar_status(h) == ar.AR_OK
        assert ar.ar_traffic(h).launches == (n.bit_length() - 1) * -(-N // PL)
        for r in range(n):
            bad = np.flatnonzero(outs[r].cpu().numpy().view(bits_t) != want)
            assert bad.size == 0, (r, bad[:5])
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK


def test_ring_on_two_streams_in_a_cuda_graph():
    # a ring call whose partials reach a tenth of L2 forks its odd pieces onto the handle's
    # stream and joins them back: captured into a CUDA graph and replayed on new inputs, every
    # element of every rank against the oracle each time
    n, dtype = 8, "bf16"
    N = (torch.cuda.get_device_properties(0).L2_cache_size // 4) // 4 + 4096   # 4 N bytes > L2 / 4
    assert _ring_pieces(n, N, dtype, False) >= 2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal", workloads.seed_of(5) + 300)
    outs = [torch.empty_like(t) for t in ins]
    h = ar.ar_create(n, N * 2)
    try:
        s = torch.cuda.Stream()
        _run(ar.ar_ring, h, ins, outs, N, dtype)   # outside capture first
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rc = ar.ar_ring(h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], N, dtype, s)
        assert rc == ar.AR_OK
        for k in range(2):
            src = workloads.rank_inputs_device(n, N, dtype, "normal", workloads.seed_of(5) + 301 + k)
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
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK


def test_ring_takes_one_stream_while_timing_records():
    # with AR_OPT_TIMING recording, the same call runs its pieces on the caller's stream alone
    # (one-stream piece count), each record timing its own launches; the sums are unchanged
    n, dtype = 8, "bf16"
    N = 16 << 20   # 32 MiB per rank: 4 N bytes = 64 MiB, above a tenth of L2
    ins = workloads.rank_inputs_device(n, N, dtype, "normal", workloads.seed_of(5) + 400)
    want = oracle.ring([t.cpu().numpy().view(np.uint16) for t in ins], dtype)[0]
    outs = [torch.empty_like(t) for t in ins]
    half = torch.cuda.get_device_properties(0).L2_cache_size // 2
    P = min(64, max(1, (N * 4 + half // 2) // half))
    C = oracle.chunk_elems(n, N, dtype)
    PL = C if P == 1 else min(C, -(-(-(-C // P)) // 256) * 256)
    one_stream = -(-C // PL)
    h = ar.ar_create(n, N * 2)
    try:
        _run(ar.ar_ring, h, ins, outs, N, dtype)
        assert ar.ar_traffic(h).launches == 2 * (n - 1) * _ring_pieces(n, N, dtype, False)
        assert ar.ar_set_option(h, ar.AR_OPT_TIMING, 256) == ar.AR_OK
        for o in outs:
            o.fill_(0x5A5A)
        _run(ar.ar_ring, h, ins, outs, N, dtype)
        assert ar.ar_status(h) == ar.AR_OK
        assert ar.ar_traffic(h).launches == 2 * (n - 1) * one_stream
        recs = ar.ar_timing(h)
        assert sum(r[4] for r in recs) == 2 * (n - 1) * one_stream
        for r in range(n):
            assert not np.flatnonzero(outs[r].cpu().numpy().view(np.uint16) != want).size
    finally:
        assert ar.ar_destroy(h) == ar.AR_OK
