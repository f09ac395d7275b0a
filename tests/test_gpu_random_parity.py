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
