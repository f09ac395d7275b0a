"""Pins for the oracle's payload conversions.

The oracle writes bf16 and fp16 rounding from the IEEE-754 definitions; here
they are checked against independent library routines: torch's CPU bfloat16
cast and numpy's float16 cast (both round to nearest, ties to even).
"""

import numpy as np
import pytest
import torch

import oracle


def _torch_bf16_bits(f: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f32_cases(rng, count):
    """Random bit patterns over the whole binary32 range, plus every tie and
    boundary that the rounding rules single out."""
    rand = rng.integers(0, 1 << 32, size=count, dtype=np.uint64).astype(np.uint32)
    hi = rng.integers(0, 1 << 16, size=count // 4, dtype=np.uint64).astype(np.uint32) << 16
    ties = hi | 0x8000                      # exactly half a bf16 ulp
    near = np.concatenate([hi | 0x7FFF, hi | 0x8001, hi | 0x0001, hi | 0xFFFF])
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0xFF7FFFFF,
                        0x00000001, 0x807FFFFF, 0x00800000, 0x7F7F8000, 0x7F7F7FFF,
                        0x3F808000, 0x3F818000, 0x3F800000], dtype=np.uint32)
    return np.concatenate([rand, ties, near, special])


def _same_bits_or_both_nan(a_bits, b_bits, a_f, b_f):
    nan = np.isnan(a_f) & np.isnan(b_f)
    return np.all((a_bits == b_bits) | nan)


def test_bf16_widening_exhaustive():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert _same_bits_or_both_nan(ours.view(np.uint32), ref.view(np.uint32), ours, ref)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    bits = _f32_cases(rng, 1 << 20)
    f = bits.view(np.float32)
    ours = oracle.f32_to_bf16(f)
    ref = _torch_bf16_bits(f)
    ours_f = oracle.bf16_to_f32(ours)
    ref_f = oracle.bf16_to_f32(ref)
    assert _same_bits_or_both_nan(ours, ref, ours_f, ref_f)


def test_bf16_ties_go_to_even():
    # 1 + 2^-8 is halfway between bf16 1.0 and 1.0078125: ties to the even 1.0.
    x = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -(1.0 + 2.0**-8)], np.float32)
    got = oracle.bf16_to_f32(oracle.f32_to_bf16(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0 + 4 * 2.0**-8, -1.0], np.float32))


def test_f16_widening_exhaustive():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    assert _same_bits_or_both_nan(ours.view(np.uint32), ref.view(np.uint32), ours, ref)


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(11)
    rand = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # magnitudes around the binary16 range: subnormals, the normal range, overflow
    mags = rng.uniform(-30, 17, size=1 << 19)
    around = (np.exp2(mags) * rng.choice([-1, 1], size=mags.size)).astype(np.float32).view(np.uint32)
    # exact halfway points between neighbouring binary16 values
    h = rng.integers(0, 0x7C00, size=1 << 16).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32).view(np.uint32)
    special = np.array([0x477FE000, 0x477FF000, 0x477FEFFF, 0x47800000, 0x33800000,
                        0x33000000, 0x33000001, 0x387FC000, 0x38800000, 0x7FC00000], np.uint32)
    bits = np.concatenate([rand, around, mid, special])
    f = bits.view(np.float32)
    ours = oracle.f32_to_f16(f)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    assert _same_bits_or_both_nan(ours, ref, oracle.f16_to_f32(ours), oracle.f16_to_f32(ref))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_roundtrip_of_every_finite_payload(dtype):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle.to_f32(h, dtype)
    keep = np.isfinite(f)
    back = oracle.f32_to_bf16(f) if dtype == "bf16" else oracle.f32_to_f16(f)
    np.testing.assert_array_equal(back[keep], h[keep])
