"""Agreement rules between the CUDA path and the oracle.

* indices on integer-grid inputs (fp32 scores exact): bit-exact sets;
* indices on Gaussian inputs: the selected sets may differ only by positions
  whose oracle score lies within 1e-5 (relative) of the k-th score;
* out: max-abs <= 1e-2 and relative L2 <= 2e-3 against the fp64 oracle.  The
  max-abs bound is read on the unit scale: |out - ref| <= 1e-2 * max(1, |ref|)
  element by element.  The output is bf16, whose rounding alone moves a value
  of magnitude v by up to 2^-9 v; outputs of the fp8 pools with fp32 or UE8M0
  scales reach tens or thousands, where an absolute 1e-2 is below half a
  bf16 ulp;
* lse: |lse - lse_ref| <= 1e-4 * max(1, |lse_ref|); -inf must match -inf.
When two index sets differ only by tolerated ties, out / lse are compared
with the oracle evaluated on the GPU's own set.
"""
import numpy as np

OUT_MAX_ABS = 1e-2
OUT_REL_L2 = 2e-3
LSE_TOL = 1e-4
TIE_REL = 1e-5


def sel_set(row):
    row = np.asarray(row)
    return set(int(x) for x in row[row >= 0])


def check_index_sets(gpu_row, ref_row, scores, k):
    """Returns None when the sets are equal, else asserts the tie rule and
    returns the GPU set (as a sorted array)."""
    g, r = sel_set(gpu_row), sel_set(ref_row)
    assert len(g) == len(r), (len(g), len(r))
    if g == r:
        return None
    s = np.asarray(scores, dtype=np.float64)
    kth = np.sort(s)[::-1][min(k, len(s)) - 1]
    scale = max(abs(kth), 1e-3 * np.abs(s).max())
    for p in g ^ r:
        assert abs(s[p] - kth) <= TIE_REL * scale, ("non-tie difference", p, s[p], kth)
    return np.array(sorted(g))


def check_out_lse(out, lse, ref_out, ref_lse, what=""):
    out = np.asarray(out, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    ref_lse = np.asarray(ref_lse, dtype=np.float64)
    assert out.shape == ref_out.shape, (out.shape, ref_out.shape)
    assert np.isfinite(out).all(), what + ": non-finite output"
    err = np.abs(out - ref_out) / np.maximum(1.0, np.abs(ref_out))
    assert err.max() <= OUT_MAX_ABS, (what, "max-abs (unit scale)", err.max())
    den = np.linalg.norm(ref_out)
    if den > 0:
        rel = np.linalg.norm(out - ref_out) / den
        assert rel <= OUT_REL_L2, (what, "rel-L2", rel)
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ninf), (what, "-inf lse mismatch")
    d = np.abs(lse[~ninf] - ref_lse[~ninf])
    tol = LSE_TOL * np.maximum(1.0, np.abs(ref_lse[~ninf]))
    assert (d <= tol).all(), (what, "lse", d.max())
