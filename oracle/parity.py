"""The GEMM parity criterion: how a GPU result is compared with the oracle.

TEST INFRASTRUCTURE ONLY (like the rest of this package): the tests and
``__graft_entry__.smoke()`` use it; the product library never imports it.

The target tolerance is max(1 ulp of the output format, 2^-7 |ref|) per
element, ref being the oracle's exactly accumulated, fp64-scaled value
before rounding.  Any kernel that accumulates in fp32 can exceed that
literal bound where an output nearly cancels (|ref| far below the size of
its terms): the error of summing K fp32 terms is bounded by
2 K 2^-24 sum |a_s b_s A B| (plus the final rounding), and that bound can be
larger than 2^-7 |ref|.  Such elements are accepted when they lie within
that summation bound and are rare (at most max(2, 1e-4 n) of n outputs).
Non-finite outputs must sit exactly where the oracle's are, with the same
sign for infinities.
"""
import numpy as np

from . import bf16_bits_to_f64, fp16_bits_to_f64, round_bf16, round_fp16


def out_to_f64(b: np.ndarray, out_dtype: int) -> np.ndarray:
    return bf16_bits_to_f64(b) if out_dtype == 0 else fp16_bits_to_f64(b)


def ulp_of(ref: np.ndarray, out_dtype: int) -> np.ndarray:
    """Spacing of the output format (bf16 or fp16) at |ref|, subnormals included."""
    mbits, emin = (7, -126) if out_dtype == 0 else (10, -14)
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** (emin - 1))))
    e = np.maximum(e, emin)
    return 2.0 ** (e - mbits)


def check_gemm(got_bits, exact, sumabs, K: int, out_dtype: int = 0, what: str = "",
               allow_nonfinite: bool = False):
    """Compare GPU output bits with the oracle's fp64 values; raises AssertionError.

    got_bits: uint16 output bits; exact: oracle value before rounding; sumabs:
    sum |a_s b_s A B| per element (from the oracle).  With allow_nonfinite, the
    oracle's non-finite elements (from non-finite scales) must be matched exactly
    (NaN by NaN, inf by an inf of the same sign); otherwise every output must be
    finite.  Returns a dict of statistics.
    """
    got = out_to_f64(got_bits, out_dtype)
    ref = np.asarray(exact, np.float64)
    fin = np.isfinite(ref)
    # finite values whose rounding to the output format overflows
    rounded = out_to_f64(round_bf16(ref) if out_dtype == 0 else round_fp16(ref), out_dtype)
    ref_rounded_inf = fin & np.isinf(rounded)
    if allow_nonfinite:
        nan_r, nan_g = np.isnan(ref), np.isnan(got)
        assert np.array_equal(nan_r, nan_g), f"{what}: NaN positions differ"
        inf_r = np.isinf(ref)
        assert np.array_equal(got[inf_r], ref[inf_r]), f"{what}: infinities differ"
    else:
        assert np.all(fin), f"{what}: the oracle produced non-finite values"
    # finite references that round beyond the format's range must come out as inf of that sign
    if ref_rounded_inf.any():
        assert np.array_equal(got[ref_rounded_inf], rounded[ref_rounded_inf]), f"{what}: overflow differs"
    sel = fin & ~ref_rounded_inf
    assert np.all(np.isfinite(got[sel])), f"{what}: non-finite outputs where the oracle is finite"
    g, r, sa = got[sel], ref[sel], np.asarray(sumabs, np.float64)[sel]
    diff = np.abs(g - r)
    ulp = ulp_of(r, out_dtype)
    lit = np.maximum(ulp, 2.0 ** -7 * np.abs(r))
    acc = ulp + 2.0 * K * 2.0 ** -24 * sa
    bad_lit = diff > lit
    bad = bad_lit & (diff > acc)
    stats = {
        "n": int(diff.size),
        "literal_violations": int(bad_lit.sum()),
        "hard_violations": int(bad.sum()),
        "max_rel_to_sumabs": float((diff / np.maximum(sa, 1e-300)).max()) if diff.size else 0.0,
    }
    assert stats["hard_violations"] == 0, (what, stats, np.argwhere(bad)[:5])
    assert stats["literal_violations"] <= max(2, 1e-4 * diff.size), (what, stats)
    return stats
