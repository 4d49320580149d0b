"""The activation quantiser kernel's arithmetic shortcut, emulated in numpy, decides every
E2M1 code as the oracle's encoder does on the correctly rounded quotient (no GPU).

The kernel replaces q = RN(x / den) by q' = RN(x * RN(1/den)) and divides exactly only
when den is not a normal power of two (whose reciprocal is exact) and q' lies within 8
ulps of a number whose low 21 mantissa bits are zero (every E2M1 decision point is one);
it then reads the code off the fp32 bits.  This test restates those steps in
numpy float32 and compares with the oracle's nearest-even encoder over values planted
near every decision point and grid value, for block scales of every E4M3 shape and
tensor scales from tiny to large."""
import numpy as np

import oracle


def _code_from_bits(q: np.ndarray) -> np.ndarray:
    a = np.abs(q).astype(np.float32)
    ua = a.view(np.uint32).astype(np.uint64)
    with np.errstate(over="ignore", invalid="ignore"):
        lo = (np.float32(a.astype(np.float64) * 2 + 2.0 ** 23).view(np.uint32) & 3).astype(np.uint64)
    hi = np.minimum(7, ((ua + 0x1FFFFF + ((ua >> 22) & 1)) >> 22) - 252)
    return np.where(a < 1, lo, hi).astype(np.uint8) | (np.signbit(q).astype(np.uint8) << 3)


def _near_decision(q: np.ndarray) -> np.ndarray:
    u = q.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 8) & 0x1FFFFF) <= 16


def test_reciprocal_shortcut_matches_division():
    rng = np.random.default_rng(7)
    e4m3 = oracle.e4m3fn_value(np.arange(1, 0x7F)).astype(np.float32)
    points = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1, 1.5, 2, 3, 4, 6, 7, 100])
    flagged = 0
    for it, a in enumerate([1.0, 0.5, 0.37, 3e-3, 1e-6, 1e3, 2.0 ** -20, 1e-40, 0.1] * 6):
        a = np.float32(a)
        den = np.float32(np.float32(rng.choice(e4m3)) * a)
        n = 8000
        near = rng.choice(points, n) * float(den) * (1 + rng.integers(-300, 301, n) * 2.0 ** -10)
        x = np.concatenate([near * rng.choice([-1, 1], n), rng.uniform(-7, 7, n) * float(den), [0.0, -0.0]])
        x = (x.astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)  # bf16 values
        with np.errstate(all="ignore"):
            q_div = (x / den).astype(np.float32) if den > 0 else (x * np.float32(0)).astype(np.float32)
            rcp = np.float32(np.float32(1) / den) if den > 0 else np.float32(0)
            q_fast = (x * rcp).astype(np.float32)
        exact = (np.float32(den).view(np.uint32) & 0x7FFFFF) == 0
        redo = (~exact) & _near_decision(q_fast)
        q = np.where(redo, q_div, q_fast).astype(np.float32)
        flagged += int(redo.sum())
        got = _code_from_bits(q)
        want = oracle.e2m1_encode(q_div)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (float(a), float(den), x[bad[:3]], got[bad[:3]], want[bad[:3]])
    assert flagged > 1000  # the exact division path was exercised too
