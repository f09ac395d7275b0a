"""Seeded random parity sweep: every all-reduce call on random rank counts,
lengths (ragged tails, tiny and multi-tile) and payload types, bit for bit
against the oracle's definition of that call (one-shot's rank-order sum for
one-shot, two-shot, push and copy-in; the ring's order for the rings; the
hop-rounded ring and the tree against their own oracles)."""

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
import workloads
from gpu_util import Handle, bits, empty_ranks, payload_np_dtype, ptrs, upload_ranks

pytestmark = pytest.mark.gpu

E = {"f32": 4, "bf16": 2, "f16": 2}
CALLS = {
    "one_shot": (ar.ar_one_shot, oracle.all_reduce),
    "two_shot": (ar.ar_two_shot, oracle.all_reduce),
    "ring": (ar.ar_ring, oracle.ring),
    "push": (ar.ar_one_shot_push, oracle.all_reduce),
    "copyin": (ar.ar_one_shot_copyin, oracle.all_reduce),
    "ring_rounded": (ar.ar_ring_rounded, oracle.ring_rounded),
    "tree": (ar.ar_tree, oracle.tree),
    "tree_fused": (ar.ar_tree_fused, oracle.tree),
    "ring_persistent": (ar.ar_ring_persistent, oracle.ring),
    "ring_cluster": (ar.ar_ring_cluster, oracle.ring),
    "ring_fused": (ar.ar_ring_fused, oracle.ring),
    "ring_rounded_fused": (ar.ar_ring_rounded_fused, oracle.ring_rounded),
}


def _cases(k=24, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(k):
        n = int(rng.integers(2, 17))
        N = int(rng.choice([rng.integers(1, 64), rng.integers(64, 5000), rng.integers(5000, 250_000)]))
        dtype = ["f32", "bf16", "f16"][int(rng.integers(0, 3))]
        out.append((i, n, N, dtype))
    return out


@pytest.mark.parametrize("i,n,N,dtype", _cases())
def test_every_call_on_a_random_case(i, n, N, dtype):
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=777 + i)
    ins = upload_ranks(xs)
    with Handle(n, max(16, N * E[dtype]), push_staging=1, registered=1, persistent=1) as h:
        for name, (call, ref) in CALLS.items():
            if name in ("tree", "tree_fused") and n & (n - 1):
                assert call(h, ptrs(ins), ptrs(empty_ranks(n, xs[0].nbytes)), N, dtype) == ar.AR_ERR_INVALID
                continue
            outs = empty_ranks(n, xs[0].nbytes)
            rc = call(h, ptrs(ins), ptrs(outs), N, dtype)
            assert rc == ar.AR_OK, (name, ar.ar_strerror(rc))
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK, name
            want = ref(xs, dtype)
            for r in sorted({0, n // 2, n - 1}):
                got = outs[r].download(payload_np_dtype(dtype))
                np.testing.assert_array_equal(bits(got), bits(want[r]), err_msg=f"{name} rank {r}")
            for b in outs:
                assert b.guards_intact(), name
        for b in ins:
            assert b.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_every_call_with_signed_zeros_infinities_and_nans(dtype):
    # special values at scattered positions: every finite or infinite output
    # matches the oracle of that call bit for bit, every NaN output is NaN
    # there too (NaN payloads are not compared: IEEE leaves them open)
    n, N = 8, 20_011
    xs = workloads.rank_inputs(n, N, dtype, "normal_over_n", seed=4242)
    f = [oracle.to_f32(x, dtype).copy() for x in xs]
    f[0][::5] = -0.0
    f[1][::5] = -0.0          # all ranks -0 at some positions: the rings keep -0, one-shot gives +0
    for r in range(2, n):
        f[r][::5] = -0.0
    f[3][1::17] = np.inf
    f[5][2::19] = -np.inf
    f[6][3::23] = np.nan
    if dtype == "bf16":
        xs = [oracle.f32_to_bf16(a) for a in f]
    elif dtype == "f16":
        xs = [oracle.f32_to_f16(a) for a in f]
    else:
        xs = [a.astype(np.float32) for a in f]
    ins = upload_ranks(xs)
    with Handle(n, N * E[dtype], push_staging=1, registered=1, persistent=1) as h:
        for name, (call, ref) in CALLS.items():
            outs = empty_ranks(n, xs[0].nbytes)
            rc = call(h, ptrs(ins), ptrs(outs), N, dtype)
            assert rc == ar.AR_OK, (name, ar.ar_strerror(rc))
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK, name
            want = ref(xs, dtype)
            for r in (0, 7):
                got = outs[r].download(payload_np_dtype(dtype))
                gf, wf = oracle.to_f32(got, dtype), oracle.to_f32(want[r], dtype)
                assert np.array_equal(np.isnan(gf), np.isnan(wf)), name
                keep = ~np.isnan(wf)
                np.testing.assert_array_equal(bits(got)[keep], bits(want[r])[keep], err_msg=f"{name} rank {r}")


def test_every_call_with_count_zero_is_a_no_op():
    # count 0: AR_OK, no launch, no byte of any buffer touched, for every all-reduce call
    n = 8
    with Handle(n, 1 << 12, push_staging=1, registered=1, persistent=1) as h:
        ins, outs = empty_ranks(n, 64, byte=0x11), empty_ranks(n, 64, byte=0x33)
        for name, (call, _) in CALLS.items():
            assert call(h, ptrs(ins), ptrs(outs), 0, "bf16") == ar.AR_OK, name
            t = ar.ar_traffic(h)
            assert t.launches == 0 and t.hbm_read_bytes == 0 and t.hbm_write_bytes == 0, name
        assert ar.ar_status(h) == ar.AR_OK
    torch.cuda.synchronize()
    assert all(bool((b.body() == 0x11).all()) for b in ins)
    assert all(bool((b.body() == 0x33).all()) for b in outs)
    for b in ins + outs:
        assert b.guards_intact()
