"""CPU check of the fixed-point form of the stochastic-rounding decision.

The oracle rounds up iff r * 2^-16 < p, r the element's 16 random bits and
p = (a - lo) / (hi - lo) the position of a between its grid neighbours
(ufp4_oracle.c, ref_round_sr).  The kernels take the same decision in fixed
point: with t = a scaled so that the neighbours are consecutive integers,
T = ceil(t * 2^16) holds the lower neighbour's index in its top bits and
ceil(p * 2^16) in its low 16, and the decision is r < T mod 2^16 (one
rounding-up conversion per code); the E1M2 kernels take it as the carry of
an addition, the index (T + 0xFFFF - r) >> 16.  This test restates those
rules, checks that the two E1M2 forms agree, and compares them with the
oracle's float decision for random magnitudes, grid points, the clamp, and
for every r next to each threshold (including fractions above 1 - 2^-16,
whose rounding-up conversion carries into the index).
"""
import math

import numpy as np
import pytest


F32 = np.float32


def fixed_point_code(grid, a, r):
    """Magnitude index chosen by the kernels' fixed-point rule (a >= 0)."""
    a = F32(a)
    if grid == 1:   # E1M2: neighbours 0.5 apart
        t = min(F32(a * F32(2.0 ** 17)), F32(7 << 16))
        T = int(math.ceil(float(t)))
        compare = (T >> 16) + (1 if r < (T & 0xFFFF) else 0)
        carry = (T + 0xFFFF - r) >> 16
        assert carry == compare, (float(a), r)
        return carry
    if not a < F32(6.0):
        return 7
    mul = F32(2.0 ** 17) if a < 2 else (F32(2.0 ** 16) if a < 4 else F32(2.0 ** 15))
    T = int(math.ceil(float(F32(a * mul))))
    # ip = floor(a / step) for the steps 0.5 / 1 / 2 of the three ranges, so
    # the lower neighbour's E2M1 index is ip / ip + 2 / ip + 4; a fraction
    # above 1 - 2^-16 carries into ip, which then names the upper neighbour
    ip = T >> 16
    base = ip if a < 2 else (ip + 2 if a < 4 else ip + 4)
    return base + (1 if r < (T & 0xFFFF) else 0)


@pytest.mark.parametrize("grid", [0, 1])
def test_fixed_point_rule_equals_float_rule(oracle, grid):
    rng = np.random.default_rng(11 + grid)
    qmax = oracle.grid_qmax(grid)
    grid_pts = [oracle.grid_value(grid, m) for m in range(8)]
    mags = np.concatenate([
        rng.random(4000).astype(np.float32) * F32(qmax * 1.1),                  # incl. above qmax
        np.array(grid_pts, np.float32),                                           # exact grid points
        np.nextafter(np.array(grid_pts[1:], np.float32), F32(0)),                # just below them
        (rng.random(500) * 2.0 ** rng.integers(-30, 0, 500)).astype(np.float32),  # tiny values
    ])
    checked = 0
    for a in mags:
        a_c = F32(min(float(a), qmax))
        # the threshold of this a, and the draws around it
        if grid == 1:
            T = int(math.ceil(float(F32(min(F32(a * F32(2.0 ** 17)), F32(7 << 16))))))
        else:
            mul = 2.0 ** 17 if a < 2 else (2.0 ** 16 if a < 4 else 2.0 ** 15)
            T = int(math.ceil(float(F32(a * F32(mul))))) if a < 6 else 0
        thr = T & 0xFFFF
        rs = [int(v) for v in rng.integers(0, 2 ** 16, 4)] + \
             [(thr + d) & 0xFFFF for d in (-2, -1, 0, 1, 2)]
        for r in rs:
            assert fixed_point_code(grid, a, r) == oracle.round_sr(grid, a_c, r), (grid, float(a), r)
            checked += 1
    assert checked > 40000
