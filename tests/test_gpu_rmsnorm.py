"""ar_allreduce_rmsnorm against the oracle: the all-reduce and the residual
add bit for bit (residual_out), the normalized output within one payload ulp
for bf16 / fp16 and 1e-6 relative for fp32 (the kernel sums the squares in
its own order), every rank's output identical, canary bands untouched."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Buf, Handle, bits, empty_ranks, payload_np_dtype, ptrs, upload_ranks

pytestmark = pytest.mark.gpu

E = {"f32": 4, "bf16": 2, "f16": 2}
ULP_BITS = {"f32": 23, "bf16": 7, "f16": 10}


def _within_one_ulp(got, want, dtype):
    g = oracle.to_f32(got, dtype).astype(np.float64)
    w = oracle.to_f32(want, dtype).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(w), 2.0**-126))) - ULP_BITS[dtype])
    if dtype == "f16":
        ulp = np.maximum(ulp, 2.0**-24)
    if dtype == "f32":
        # the fp32 sum of H squares, 1/sqrt and two products: ~1e-6 relative
        # (the bound used for every reordered fp32 result)
        ulp = np.maximum(ulp, 1e-6 * np.abs(w))
    return np.abs(g - w) <= ulp * (1 + 1e-9)


def _run(n, T, H, dtype, seed, in_place=False, res_in_place=False, eps=1e-6, h=None):
    xs = workloads.rank_inputs(n, T * H, dtype, "normal", seed)
    res = workloads.rank_inputs(1, T * H, dtype, "normal", seed + 1)[0]
    w = workloads.rank_inputs(1, H, dtype, "uniform", seed + 2)[0]
    ins = upload_ranks(xs)
    outs = ins if in_place else empty_ranks(n, xs[0].nbytes)
    rb = Buf(res.nbytes).upload(res)
    wb = Buf(w.nbytes).upload(w)
    ro = rb if res_in_place else Buf(res.nbytes).fill(0x3C)

    def call(handle):
        rc = ar.ar_allreduce_rmsnorm(handle, ptrs(ins), rb.ptr, wb.ptr, eps, ptrs(outs), ro.ptr, T, H, dtype)
        assert rc == ar.AR_OK, ar.ar_strerror(rc)
        assert ar.ar_status(handle) == ar.AR_OK

    if h is None:
        with Handle(n, max(16, T * H * E[dtype])) as hh:
            call(hh)
            traffic = ar.ar_traffic(hh).as_dict()
    else:
        call(h)
        traffic = ar.ar_traffic(h).as_dict()
    torch.cuda.synchronize()
    for b in ins + outs + [rb, wb, ro]:
        assert b.guards_intact()
    want_y, want_r = oracle.allreduce_rmsnorm(xs, res, w, eps, T, H, dtype)
    got_r = ro.download(payload_np_dtype(dtype))
    got_y = [o.download(payload_np_dtype(dtype)) for o in outs]
    return got_y, got_r, want_y, want_r, traffic


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("n,T,H", [(8, 1, 8192), (8, 64, 4096), (2, 7, 512), (16, 3, 8200), (4, 5, 16), (8, 2, 65536),
                                   (8, 9, 4096), (8, 10, 4096), (8, 48, 6144)])
def test_fused_epilogue_matches_the_unfused_chain(dtype, n, T, H):
    if H % (16 // E[dtype]):
        pytest.skip("hidden must be whole 16-byte vectors")
    got_y, got_r, want_y, want_r, traffic = _run(n, T, H, dtype, seed=n * 100 + T + H)
    np.testing.assert_array_equal(bits(got_r), bits(want_r))
    ok = _within_one_ulp(got_y[0], want_y, dtype)
    assert ok.all(), f"{(~ok).sum()} elements beyond one ulp"
    if dtype != "f32":   # rounding to 8 / 11 bits hides the fp32-level differences
        assert np.mean(bits(got_y[0]) == bits(want_y)) > 0.95
    for y in got_y[1:]:
        np.testing.assert_array_equal(bits(y), bits(got_y[0]))
    S = T * H * E[dtype]
    assert traffic["op"] == ar.AR_OP_ALLREDUCE_RMSNORM
    assert traffic["hbm_read_bytes"] == (n + 1) * S + H * E[dtype]
    assert traffic["hbm_write_bytes"] == (n + 1) * S


def test_fused_epilogue_in_place():
    got_y, got_r, want_y, want_r, _ = _run(8, 4, 4096, "bf16", seed=3, in_place=True, res_in_place=True)
    np.testing.assert_array_equal(got_r, want_r)
    assert _within_one_ulp(got_y[5], want_y, "bf16").all()


def test_fused_epilogue_argument_errors():
    n, T, H = 4, 2, 1024
    with Handle(n, T * H * 2) as h:
        ins, outs = empty_ranks(n, T * H * 2), empty_ranks(n, T * H * 2)
        res, w, ro = Buf(T * H * 2), Buf(H * 2), Buf(T * H * 2)
        call = lambda **k: ar.ar_allreduce_rmsnorm(
            h, k.get("ins", ptrs(ins)), k.get("res", res.ptr), k.get("w", w.ptr), k.get("eps", 1e-6),
            k.get("outs", ptrs(outs)), k.get("ro", ro.ptr), k.get("T", T), k.get("H", H), "bf16")
        assert call(H=1020) == ar.AR_ERR_INVALID                   # not whole 16-byte vectors
        assert call(H=0) == ar.AR_ERR_INVALID
        assert call(eps=-1.0) == ar.AR_ERR_INVALID
        assert call(T=T + 1) == ar.AR_ERR_TOO_LARGE                # beyond max_bytes
        assert call(ro=ptrs(outs)[1]) == ar.AR_ERR_INVALID         # residual_out is an output of a rank
        assert call(w=ptrs(outs)[0]) == ar.AR_ERR_INVALID          # weight overlaps an output
        assert call(res=res.ptr + 8) == ar.AR_ERR_ALIGN
        assert call(T=0) == ar.AR_OK
        assert ar.ar_traffic(h).launches == 0


@pytest.mark.parametrize("mode", ["stream", "graph"])
@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("T,H", [(1, 4096), (8, 8192), (48, 6144), (64, 8192)])
def test_chained_calls_each_read_the_previous_results(mode, pdl, T, H):
    # call k + 1 takes call k's normalized outputs as its rank inputs and call k's residual
    # output as its residual, back to back on one stream (or replayed from a CUDA graph).
    # With programmatic launch a call may start before the one before it has ended (small
    # grids let the next launch in at once); it must still read that call's results.  Every
    # output starts as a sentinel, and each call is checked against the oracle run on the
    # values its predecessor actually left.
    n, K, dtype = 8, 4, "bf16"
    xs = workloads.rank_inputs(n, T * H, dtype, "normal", seed=T + H + pdl)
    res = workloads.rank_inputs(1, T * H, dtype, "normal", seed=T + H + 1)[0]
    w = workloads.rank_inputs(1, H, dtype, "uniform", seed=T + H + 2)[0]
    S = T * H * 2
    ins, rb, wb = upload_ranks(xs), Buf(S).upload(res), Buf(2 * H).upload(w)
    outs = [empty_ranks(n, S, byte=0x3C) for _ in range(K)]
    ros = [Buf(S).fill(0x3C) for _ in range(K)]
    with Handle(n, S, pdl=pdl) as h:
        s = torch.cuda.Stream()

        def chain():
            for k in range(K):
                src, r_in = (ins, rb) if k == 0 else (outs[k - 1], ros[k - 1])
                rc = ar.ar_allreduce_rmsnorm(h, ptrs(src), r_in.ptr, wb.ptr, 1e-6, ptrs(outs[k]), ros[k].ptr, T, H,
                                             dtype, s)
                assert rc == ar.AR_OK

        if mode == "stream":
            chain()
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                chain()
            g.replay()
        torch.cuda.synchronize()
        assert ar.ar_status(h) == ar.AR_OK
    prev_in, prev_res = xs, res
    for k in range(K):
        want_y, want_r = oracle.allreduce_rmsnorm(prev_in, prev_res, w, 1e-6, T, H, dtype)
        got_r = ros[k].download(np.uint16)
        got_y = [o.download(np.uint16) for o in outs[k]]
        np.testing.assert_array_equal(got_r, want_r, err_msg=f"call {k}: residual")
        assert _within_one_ulp(got_y[0], want_y, dtype).all(), f"call {k}: normalized output"
        for y in got_y[1:]:
            np.testing.assert_array_equal(y, got_y[0])
        prev_in, prev_res = got_y, got_r


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fused_epilogue_largest_hidden(dtype):
    # the largest row the call accepts (327680 elements: its slice over a cluster of 8 CTAs
    # is 160 KiB of fp32), and the next whole vector past it refused
    H = 327680
    got_y, got_r, want_y, want_r, _ = _run(2, 1, H, dtype, seed=77)
    np.testing.assert_array_equal(bits(got_r), bits(want_r))
    assert _within_one_ulp(got_y[0], want_y, dtype).all()
    H2 = H + 16 // E[dtype]
    with Handle(2, H2 * E[dtype]) as h:
        ins, outs = empty_ranks(2, H2 * E[dtype]), empty_ranks(2, H2 * E[dtype])
        res, w, ro = Buf(H2 * E[dtype]), Buf(H2 * E[dtype]), Buf(H2 * E[dtype])
        assert ar.ar_allreduce_rmsnorm(h, ptrs(ins), res.ptr, w.ptr, 1e-6, ptrs(outs), ro.ptr, 1, H2,
                                       dtype) == ar.AR_ERR_INVALID
