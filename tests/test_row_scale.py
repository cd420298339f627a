"""The per-row scale division of the dynamic-FP8 kernels, checked on the host.

The latent gather with dynamic FP8 turns a row's largest magnitude `amax`
into its scale RN(amax / 448) as q0 = RN(amax * y), r = amax - 448 q0 (one
fused multiply-add, exact), sc = RN(q0 + r y) (one fused multiply-add),
with y = RN(1/448): Markstein's refinement of the quotient by a correctly
rounded reciprocal.  The kernel uses it while amax lies in [2^-100, 2^100]
and the IEEE divide elsewhere.  Scaling amax by a power of two scales q0, r
and the result exactly in that range, so the claim holds for every amax
there if it holds for every significand: this test runs all 2^23 fp32
significands of [1, 2) and compares with the correctly rounded quotient.

Exactness of the emulation: products of two fp32 numbers and differences of
nearby ones are exact in fp64; the last rounding, RN32(q0 + r y), is decided
by comparing the exact fp64 distances to the fp32 neighbours of q0 (|r y| is
below one ulp of q0).  The reference RN32(a / 448) is the fp64 quotient
rounded to fp32: a / 7 has a binary expansion of period 3 unless 7 divides
the significand, so it never lies within 2^-53 of an fp32 midpoint and the
double rounding cannot err.
"""
import numpy as np


def _rn32_of_sum(q0, d):
    """RN32(q0 + d) for fp32 q0 and an fp64 d with |d| at most one ulp of q0,
    exactly, ties to even."""
    lo = np.nextafter(q0, np.float32(-np.inf))
    hi = np.nextafter(q0, np.float32(np.inf))
    cands = np.stack([lo, q0, hi])                       # fp32 neighbours
    dist = np.abs((q0.astype(np.float64) - cands.astype(np.float64)) + d)  # exact in fp64
    best = dist.min(axis=0)
    tie = (dist == best).sum(axis=0) > 1
    pick = np.argmin(dist, axis=0)
    out = cands[pick, np.arange(q0.size)]
    if tie.any():  # ties to the even significand
        even = (cands.view(np.uint32) & 1) == 0
        ok = (dist == best) & even
        out[tie] = cands[np.argmax(ok[:, tie], axis=0), np.nonzero(tie)[0]]
    return out


def _refined_scale(a):
    y = np.float32(1.0) / np.float32(448.0)
    q0 = (a * y).astype(np.float32)                      # fp32 multiply, RN
    r64 = a.astype(np.float64) - 448.0 * q0.astype(np.float64)  # exact
    r = r64.astype(np.float32)
    assert np.array_equal(r.astype(np.float64), r64), "remainder not representable"
    return _rn32_of_sum(q0, r.astype(np.float64) * np.float64(y))  # r y exact in fp64


def test_every_significand():
    a = (np.arange(1 << 23, dtype=np.uint32) | np.uint32(127 << 23)).view(np.float32)
    ref = (a.astype(np.float64) / 448.0).astype(np.float32)
    got = _refined_scale(a)
    bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
    assert bad.size == 0, (bad[:5], a[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_range_ends_and_powers_of_two():
    """The same formula at the ends of the refined range and at powers of two
    (where the ulp below q0 is half the ulp above)."""
    a = np.array([2.0 ** -100, 2.0 ** 100, 448.0, 896.0, 1.0, 2.0 ** -100 * 1.75,
                  2.0 ** 99 * 1.999], np.float32)
    ref = (a.astype(np.float64) / 448.0).astype(np.float32)
    assert np.array_equal(_refined_scale(a).view(np.uint32), ref.view(np.uint32))


def test_emulation_catches_a_plain_multiply():
    """The check is strong enough to see the error the refinement removes:
    RN(a * RN(1/448)) alone is wrong for some significands."""
    a = (np.arange(1 << 16, dtype=np.uint32) * 128 | np.uint32(127 << 23)).view(np.float32)
    ref = (a.astype(np.float64) / 448.0).astype(np.float32)
    plain = (a * (np.float32(1.0) / np.float32(448.0))).astype(np.float32)
    assert (plain.view(np.uint32) != ref.view(np.uint32)).any()
