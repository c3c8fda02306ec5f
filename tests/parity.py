"""The parity bars, shared by the GPU tests.

  * Transform off: codes, block scales and tensor scales bit-exact (checked
    inline by the tests with array equality).
  * Transform on: the fp32 butterflies may round a value differently from
    the oracle's fp64 transform, which can move a code by one grid step.  At
    most 1e-4 of the codes of a tensor (or of the sampled rows of one) may
    differ, each by at most one step; counted over the whole comparison, so
    a small tensor must match exactly.
  * GEMMs: relative Frobenius error <= 1e-5 against the fp64 product of the
    dequantized operands the kernel consumed.  With the transform off those
    are the oracle's own operands (bit-exact codes); with it on they are the
    GPU's codes and scales, dequantized by the oracle, after the codes have
    passed the bar above against the oracle's.
"""
import numpy as np

CODE_FRAC = 1e-4
GEMM_TOL = 1e-5


def signed_index(codes):
    c = np.asarray(codes).astype(np.int32)
    return np.where(c & 8, -(c & 7), c & 7)


class CodeTally:
    """Accumulates code differences over several pieces of one comparison."""

    def __init__(self):
        self.n = 0
        self.diff = 0
        self.worst = 0

    def add(self, got, ref):
        d = np.abs(signed_index(got) - signed_index(ref))
        self.n += d.size
        self.diff += int((d > 0).sum())
        self.worst = max(self.worst, int(d.max()) if d.size else 0)

    def check(self, frac=CODE_FRAC):
        assert self.worst <= 1, "a code differs by %d grid steps" % self.worst
        assert self.diff <= frac * self.n, "%d of %d codes differ (> %g)" % (self.diff, self.n, frac)


def assert_codes_close(got, ref, frac=CODE_FRAC):
    t = CodeTally()
    t.add(got, ref)
    t.check(frac)


def rel_fro(c, ref):
    c = np.asarray(c, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(c - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_gemm_close(c, ref, tol=GEMM_TOL):
    err = rel_fro(c, ref)
    assert err <= tol, "relative Frobenius error %g > %g" % (err, tol)
