"""Shared parity measures for the GPU tests (test infrastructure).

Tolerances (stated by the benchmark specification of this library):
* FP16 decode: max |err| <= 1e-2 and relative L2 error <= 2e-3 against the
  fp64 oracle.
* FP8 context output: >= 99.9 % of elements within 2 E4M3 ulps of the
  oracle's exact value rounded to E4M3, and relative L2 error <= 3e-2 after
  dequantisation (check_ctx).  The ulp distance is the difference of the
  monotone code ordinals.  The "format floor" -- the relative L2 error of
  the exact result rounded to E4M3, the best any E4M3 output can do -- is
  printed beside it as a diagnostic only.
* check_ctx_format_floor is a separate, weaker check for inputs whose exact
  outputs lie among E4M3's subnormals (a 65536-key softmax at out_scale 1):
  there the format alone misses 3e-2, so it asserts the ulp bar and a
  relative L2 error within 1.05 x the floor, and says that 3e-2 is out of
  reach.  No test of a stated configuration uses it in place of check_ctx.
* Dequantisation: bit-exact.
"""
import numpy as np

import oracle

DECODE_MAX_ABS = 1e-2
DECODE_REL_L2 = 2e-3
CTX_ULPS = 2
CTX_FRAC_WITHIN = 0.999
CTX_REL_L2 = 3e-2


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def check_decode(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    rl = rel_l2(got, ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err.max() <= DECODE_MAX_ABS, f"{what}: max|err| {err.max():.3e} > {DECODE_MAX_ABS}"
    assert rl <= DECODE_REL_L2, f"{what}: rel-L2 {rl:.3e} > {DECODE_REL_L2}"
    return float(err.max()), rl


def e4m3_ordinal(codes):
    c = np.asarray(codes, dtype=np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def _ctx_measures(out_codes, ref):
    out_codes = np.asarray(out_codes, dtype=np.uint8)
    ref_codes = oracle.f64_to_e4m3(ref) if ref.size < 200000 else _fast_e4m3(ref)
    ulps = np.abs(e4m3_ordinal(out_codes) - e4m3_ordinal(ref_codes))
    frac = float((ulps <= CTX_ULPS).mean())
    table = oracle.e4m3_table()
    got = table[out_codes]
    rl = rel_l2(got, ref)
    floor = rel_l2(table[ref_codes], ref)  # best any E4M3 output can do
    return got, ulps, frac, rl, floor


def check_ctx(out_codes, ref, what=""):
    """out_codes: uint8 E4M3 from the GPU; ref: fp64 exact O / out_scale.
    Asserts the stated bar: >= 99.9 % within 2 ulps and rel-L2 <= 3e-2."""
    got, ulps, frac, rl, floor = _ctx_measures(out_codes, ref)
    print(f"{what}: within {CTX_ULPS} ulps {frac:.6f} (max {int(ulps.max())}), rel-L2 {rl:.4e} "
          f"(bound {CTX_REL_L2:.1e}; E4M3 format floor {floor:.4e}, diagnostic)")
    assert np.isfinite(got).all(), f"{what}: NaN in output"
    assert frac >= CTX_FRAC_WITHIN, f"{what}: only {frac:.5f} within {CTX_ULPS} ulps (max {ulps.max()})"
    assert rl <= CTX_REL_L2, f"{what}: rel-L2 {rl:.3e} > {CTX_REL_L2:.1e} (format floor {floor:.3e})"
    return frac, rl, int(ulps.max())


def check_ctx_format_floor(out_codes, ref, what=""):
    """The weaker check for outputs that E4M3 cannot hold to 3e-2 (see the
    module docstring): the ulp bar, and rel-L2 within 1.05 x the floor."""
    got, ulps, frac, rl, floor = _ctx_measures(out_codes, ref)
    print(f"{what}: within {CTX_ULPS} ulps {frac:.6f} (max {int(ulps.max())}), rel-L2 {rl:.4e} against "
          f"the format floor {floor:.4e}; the stated 3e-2 bound is {'met' if rl <= CTX_REL_L2 else 'NOT met'}")
    assert np.isfinite(got).all(), f"{what}: NaN in output"
    assert frac >= CTX_FRAC_WITHIN, f"{what}: only {frac:.5f} within {CTX_ULPS} ulps (max {ulps.max()})"
    assert rl <= 1.05 * floor, f"{what}: rel-L2 {rl:.3e} > 1.05 x format floor {floor:.3e}"
    return frac, rl, floor


def _fast_e4m3(ref):
    """Round to E4M3 by nearest table value (ties to the even code), for large arrays."""
    table = oracle.e4m3_table()
    pos = np.array([table[c] for c in range(0x7F)])  # 0 .. 448 ascending
    a = np.minimum(np.abs(ref), 448.0)
    idx = np.searchsorted(pos, a)  # pos[idx-1] < a <= pos[idx]
    idx = np.clip(idx, 1, len(pos) - 1)
    lo, hi = pos[idx - 1], pos[idx]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((idx % 2) == 0))
    code = np.where(pick_hi, idx, idx - 1)
    code = np.where(a == 0, 0, code)
    return (code | np.where(ref < 0, 0x80, 0)).astype(np.uint8)
