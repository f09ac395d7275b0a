"""n = 2 brute force on the GPU: every bf16 (and fp16) encoding as rank 0's
value against a stratified set of rank 1 values, through every all-reduce
call, bit for bit against the oracle.

The custom all-reduce notes (SGLang JIT kernel, §4) fix the arithmetic: one
binary32 sum in rank order, one round-to-nearest-even to the payload type.
With n = 2 that is one add and one rounding, so these inputs drive the
device's conversions through every exponent, both signs, signed zeros,
subnormal inputs and results, exact ties, overflow of a finite sum to
infinity, infinities and NaNs.  NaNs are compared by class (any NaN equals
any NaN); every other result must match bit for bit.  A second test checks
hand-worked results (ties, overflow, fp16 subnormal sums) against values
written down here, independent of the oracle, and a third every pair of
16-bit encodings (a 2^28 sample by default, all 2^32 with AR_EXHAUSTIVE=1).
"""

import os

import numpy as np
import pytest
import torch

import all_reduce_reduction_rank_gb300 as ar
import oracle
from gpu_util import Handle, bits

pytestmark = pytest.mark.gpu

# every call, with the oracle that defines its bits
CALLS = {
    "one_shot": (ar.ar_one_shot, oracle.all_reduce),
    "two_shot": (ar.ar_two_shot, oracle.all_reduce),
    "push": (ar.ar_one_shot_push, oracle.all_reduce),
    "copyin": (ar.ar_one_shot_copyin, oracle.all_reduce),
    "ring": (ar.ar_ring, oracle.ring),
    "ring_fused": (ar.ar_ring_fused, oracle.ring),
    "ring_persistent": (ar.ar_ring_persistent, oracle.ring),
    "ring_cluster": (ar.ar_ring_cluster, oracle.ring),
    "ring_rounded": (ar.ar_ring_rounded, oracle.ring_rounded),
    "ring_rounded_fused": (ar.ar_ring_rounded_fused, oracle.ring_rounded),
    "tree": (ar.ar_tree, oracle.tree),
    "tree_fused": (ar.ar_tree_fused, oracle.tree),
}

EXP_BITS = {"bf16": 8, "f16": 5}
MAN_BITS = {"bf16": 7, "f16": 10}


def stratified(dtype: str, per_class: int, seed: int) -> np.ndarray:
    """Rank 1's values: for every sign and every exponent field (zero and
    subnormals, every normal binade, infinity and NaN) `per_class` mantissas
    (the smallest in even binades and the largest in odd ones, the rest
    random), plus +-0, +-inf, a quiet NaN, the smallest and largest subnormal
    and the largest finite value of each sign."""
    eb, mb = EXP_BITS[dtype], MAN_BITS[dtype]
    rng = np.random.default_rng(seed)
    out = []
    for sign in (0, 1):
        for e in range(1 << eb):
            # the first mantissa alternates between the smallest and the largest by binade
            mans = [0 if e % 2 == 0 else (1 << mb) - 1]
            mans += [int(m) for m in rng.integers(1, (1 << mb) - 1, size=per_class - 1)]
            for m in mans:
                out.append((sign << (eb + mb)) | (e << mb) | m)
    top = ((1 << eb) - 1) << mb
    specials = [0, 1 << (eb + mb), top, top | (1 << (eb + mb)), top | (1 << (mb - 1)), 1, (1 << mb) - 1,
                top - 1, (1 << (eb + mb)) | (top - 1)]
    return np.array(sorted(set(out) | set(specials)), dtype=np.uint16)


def all_pairs(dtype: str, per_class: int, seed: int):
    a_all = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    b_set = stratified(dtype, per_class, seed)
    return np.repeat(a_all, b_set.size), np.tile(b_set, a_all.size), b_set.size


def same_or_both_nan(got: np.ndarray, want: np.ndarray, dtype: str) -> np.ndarray:
    gf, wf = oracle.to_f32(got, dtype), oracle.to_f32(want, dtype)
    return (got == want) | (np.isnan(gf) & np.isnan(wf))


@pytest.mark.parametrize("dtype,per_class", [("bf16", 2), ("f16", 4)])
def test_every_encoding_against_a_stratified_set(dtype, per_class):
    a, b, nb = all_pairs(dtype, per_class, seed=20261203)
    assert nb >= (512 if dtype == "bf16" else 256)
    N = a.size
    xs = [a, b]
    dev = torch.device("cuda")
    ins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    wants = {}
    with Handle(2, N * 2, push_staging=1, registered=1, persistent=1) as h:
        for name, (call, ref) in CALLS.items():
            key = ref.__name__
            if key not in wants:
                wants[key] = ref(xs, dtype)
            want = wants[key]
            for o in outs:
                o.fill_(0x5A5A)
            rc = call(h, ins, outs, N, dtype)
            assert rc == ar.AR_OK, (name, ar.ar_strerror(rc))
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK, name
            for r in range(2):
                got = outs[r].cpu().numpy().view(np.uint16)
                ok = same_or_both_nan(got, want[r], dtype)
                if not ok.all():
                    i = int(np.flatnonzero(~ok)[0])
                    raise AssertionError(f"{name} rank {r}: {int((~ok).sum())} mismatches; first a=0x{a[i]:04x} "
                                         f"b=0x{b[i]:04x} got=0x{got[i]:04x} want=0x{want[r][i]:04x}")


# Every pair of 16-bit encodings (2^32 sums per payload type) through ar_one_shot,
# whose conversions (common to every kernel) are the ones under test.  By default
# 4096 values of a, spread over the encodings by an odd multiplier (a bijection
# of the 16-bit codes), against every b: 2^28 pairs per type.  AR_EXHAUSTIVE=1
# runs all 65536 values of a.
EXHAUSTIVE = os.environ.get("AR_EXHAUSTIVE") == "1"
A_PER_CALL = 4096   # 2^28 elements of 2 bytes per rank and call


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_every_pair_of_encodings(dtype):
    codes = np.arange(1 << 16, dtype=np.uint32)
    a_all = codes if EXHAUSTIVE else (codes[:A_PER_CALL] * 40503) % (1 << 16)
    b_all = codes.astype(np.uint16)
    N = A_PER_CALL << 16
    dev = torch.device("cuda")
    d_in = [torch.empty(N, dtype=torch.int16, device=dev) for _ in range(2)]
    d_out = [torch.empty(N, dtype=torch.int16, device=dev) for _ in range(2)]
    checked = 0
    with Handle(2, N * 2) as h:
        for lo in range(0, a_all.size, A_PER_CALL):
            a = np.repeat(a_all[lo:lo + A_PER_CALL].astype(np.uint16), b_all.size)
            b = np.tile(b_all, A_PER_CALL)
            for t, x in zip(d_in, (a, b)):
                t.copy_(torch.from_numpy(x.view(np.int16)))
            rc = ar.ar_one_shot(h, d_in, d_out, N, dtype)
            assert rc == ar.AR_OK, ar.ar_strerror(rc)
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK
            want = oracle.all_reduce([a, b], dtype)
            for r in range(2):
                got = d_out[r].cpu().numpy().view(np.uint16)
                bad = np.flatnonzero(got != want[r])
                if bad.size:   # NaNs compare by class
                    nan = np.isnan(oracle.to_f32(got[bad], dtype)) & np.isnan(oracle.to_f32(want[r][bad], dtype))
                    bad = bad[~nan]
                if bad.size:
                    i = int(bad[0])
                    raise AssertionError(f"rank {r}: {bad.size} mismatches; first a=0x{a[i]:04x} b=0x{b[i]:04x} "
                                         f"got=0x{got[i]:04x} want=0x{want[r][i]:04x}")
            checked += N
    assert checked == a_all.size << 16


# (a, b, expected) as bit patterns, worked by hand from IEEE-754:
# bf16 has 8 significand bits, fp16 11; the binary32 sum of two such values
# is exact unless it overflows (to an infinity), so the result is that sum
# rounded once to nearest, ties to even.
HAND = {
    "bf16": [
        (0x3F80, 0x3B80, 0x3F80),   # 1 + 2^-8: a tie between 1 and 1 + 2^-7 -> even (1)
        (0x3F81, 0x3B80, 0x3F82),   # (1 + 2^-7) + 2^-8: a tie -> even (1 + 2^-6)
        (0x4780, 0x4380, 0x4780),   # 2^16 + 2^8: a tie at a higher exponent -> 2^16
        (0x0080, 0x0001, 0x0081),   # smallest normal + smallest subnormal: exact
        (0x0001, 0x0001, 0x0002),   # two smallest subnormals: exact
        (0x8001, 0x0001, 0x0000),   # x + -x = +0
        (0x8000, 0x8000, 0x8000),   # -0 + -0 = -0 in binary32 (from a +0 start: +0; set per call below)
        (0xBF80, 0xBB80, 0xBF80),   # -1 - 2^-8: a tie -> even (-1)
        (0x3F83, 0x3B80, 0x3F84),   # (1 + 3 2^-7) + 2^-8: a tie that rounds up to the even neighbour
        (0x7F78, 0x7F78, 0x7F80),   # 3.29e38 + 3.29e38 overflows binary32 -> +inf
        (0x7F00, 0x7F00, 0x7F80),   # 2^127 + 2^127 = 2^128 overflows binary32 -> +inf
        (0xFF00, 0xFF00, 0xFF80),   # the same, negative -> -inf
        (0x7F7F, 0x7B00, 0x7F80),   # largest finite + half its ulp (2^119): finite in binary32, a tie whose
                                    # even neighbour is 2^128, past the bf16 range -> +inf
        (0xFF7F, 0xFB00, 0xFF80),   # the same, negative -> -inf
        (0x7F7F, 0x7A80, 0x7F7F),   # largest finite + a quarter of its ulp -> the largest finite
        (0x7F7F, 0x0001, 0x7F7F),   # the largest finite stays
        (0x7F80, 0xFF80, None),     # inf + -inf = NaN
    ],
    "f16": [
        (0x3C00, 0x1000, 0x3C00),   # 1 + 2^-11: a tie -> even (1)
        (0x3C01, 0x1000, 0x3C02),   # (1 + 2^-10) + 2^-11: a tie -> even
        (0x78E2, 0x78E2, 0x7C00),   # 40000 + 40000 = 80000 > 65504 -> +inf
        (0x7800, 0x7800, 0x7C00),   # 32768 + 32768 = 65536: above 65520 -> +inf
        (0x7BFF, 0x3C00, 0x7BFF),   # 65504 + 1 -> 65504
        (0x0001, 0x0001, 0x0002),   # 2^-24 + 2^-24 = 2^-23, a subnormal result
        (0x0200, 0x0200, 0x0400),   # two halves of the smallest normal make it
        (0x0401, 0x8400, 0x0001),   # normal - normal = the smallest subnormal
        (0x03FF, 0x0001, 0x0400),   # largest subnormal + smallest subnormal = smallest normal
        (0x8003, 0x0001, 0x8002),   # a negative subnormal result
        (0x7C00, 0xFC00, None),     # inf + -inf = NaN
    ],
}


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_hand_worked_results(dtype):
    cases = HAND[dtype]
    a = np.array([c[0] for c in cases], dtype=np.uint16)
    b = np.array([c[1] for c in cases], dtype=np.uint16)
    # repeat the cases past one 16-byte vector so both the vector path and the tail see them
    reps = 37
    a, b = np.tile(a, reps), np.tile(b, reps)
    N = a.size
    dev = torch.device("cuda")
    ins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in (a, b)]
    outs = [torch.empty_like(t) for t in ins]
    with Handle(2, N * 2, push_staging=1, registered=1, persistent=1) as h:
        for name, (call, ref) in CALLS.items():
            rc = call(h, ins, outs, N, dtype)
            assert rc == ar.AR_OK, (name, ar.ar_strerror(rc))
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK
            # the sums that start from +0 (one-shot's definition) turn -0 + -0 into +0
            zero_start = ref is oracle.all_reduce
            for r in range(2):
                got = outs[r].cpu().numpy().view(np.uint16)
                for k, (x, y, want) in enumerate(cases):
                    g = got[k::len(cases)]
                    if want is None:
                        assert np.isnan(oracle.to_f32(g, dtype)).all(), (name, hex(x), hex(y))
                        continue
                    if x == 0x8000 and y == 0x8000 and zero_start:
                        want = 0x0000
                    assert (g == want).all(), (name, r, hex(x), hex(y), hex(int(g[0])), hex(want))


def test_f32_n2_random_bit_patterns():
    # fp32: the sum is one binary32 add; random bit patterns cover every exponent and the specials
    rng = np.random.default_rng(17)
    N = (1 << 20) + 3
    xs = [rng.integers(0, 1 << 32, size=N, dtype=np.uint64).astype(np.uint32).view(np.float32) for _ in range(2)]
    dev = torch.device("cuda")
    ins = [torch.from_numpy(x.copy()).to(dev) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    with Handle(2, N * 4, push_staging=1, registered=1, persistent=1) as h:
        for name, (call, ref) in CALLS.items():
            want = ref(xs, "f32")
            rc = call(h, ins, outs, N, "f32")
            assert rc == ar.AR_OK, (name, ar.ar_strerror(rc))
            torch.cuda.synchronize()
            assert ar.ar_status(h) == ar.AR_OK
            for r in range(2):
                got = outs[r].cpu().numpy()
                ok = (bits(got) == bits(want[r])) | (np.isnan(got) & np.isnan(want[r]))
                assert ok.all(), (name, r, int((~ok).sum()))
