"""fp32 tolerance of the verify GEMM's outputs against the oracle.

The target: |dY| <= 1e-6 + 1e-5 |Y_oracle| elementwise.  Where one thread
block sums an output's groups in ascending order (always with
HQ_LAUNCH_EXACT_ORDER) the GPU's fp32 sum is the oracle's, bit for bit.
Where an output's K range is split between thread blocks, the blocks' partial
sums are combined in another order; any two summation orders of the same
fp32 terms differ by a few ulp of the partial sums, so an output that cancels
to near zero cannot meet 1e-5 relative to |Y| under any reordering.  For
those modes the relative part is taken against the magnitude of the sum
being formed, sx * sum_g |scale * P|, and the fraction of outputs that also
meet the elementwise target is measured and reported.
"""
import numpy as np

ATOL, RTOL = 1e-6, 1e-5


def sum_magnitude(ref):
    """sx[m] * sum_g |scale[n][g] * P[m][n][g]|: the size of the fp32 sum that forms Y[m][n]."""
    terms = np.abs(ref["scales"].astype(np.float64)[None] * ref["P"].astype(np.float64)).sum(-1)
    return np.abs(ref["sx"].astype(np.float64))[:, None] * terms


def strict_fraction(y, ref_out) -> float:
    """Fraction of outputs within 1e-6 + 1e-5 |Y_oracle| (the elementwise target)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref_out["Y"], dtype=np.float64)
    return float((np.abs(y - ref) <= ATOL + RTOL * np.abs(ref)).mean())


def assert_close(y, ref_out, min_strict: float = 0.99):
    """Every output within 1e-6 + 1e-5 * max(|Y|, sum magnitude) of the
    oracle, and at least `min_strict` of them within the elementwise target.
    Returns the measured elementwise fraction."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref_out["Y"], dtype=np.float64)
    err = np.abs(y - ref)
    mag = np.maximum(np.abs(ref), sum_magnitude(ref_out))
    lim = ATOL + RTOL * mag
    bad = err > lim
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; worst {np.max(err - lim):.3e}"
    frac = strict_fraction(y, ref_out)
    assert frac >= min_strict, f"only {frac:.5f} within the elementwise tolerance"
    return frac
