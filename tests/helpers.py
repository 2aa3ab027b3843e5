"""Comparison helpers for the tests (no finalize arithmetic here)."""
from __future__ import annotations

import json
import os

import numpy as np

# Acceptance bar for every output element: |got - ref| <= 2^-7 * |ref| + 1e-6
# (one BF16 ulp at the bottom of a binade), and at least 99% of the elements
# bit-exact.  NaN matches NaN only.
REL_TOL = 2.0 ** -7
ABS_TOL = 1e-6
MIN_EXACT = 0.99


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round through float32 (RNE twice; used only by independent checks)."""
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).copy()
    nan = np.isnan(u.view(np.float32))
    u += ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    out = (u >> 16).astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return f64_to_bf16_bits(np.asarray(x, dtype=np.float32).astype(np.float64))


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at each element (16 fewer significand bits than float32)."""
    f = np.abs(bf16_bits_to_f64(bits)).astype(np.float32)
    return np.spacing(f).astype(np.float64) * 65536.0


def compare_bf16(got: np.ndarray, ref: np.ndarray, *, rel: float = REL_TOL, abs_: float = ABS_TOL,
                 min_exact: float = MIN_EXACT, extra: np.ndarray | None = None) -> dict:
    """Element-wise check of BF16 bit arrays; returns stats, raises AssertionError.
    ``extra`` (same shape) widens the bound per element where an intermediate
    BF16 rounding propagates (the caller derives it)."""
    got = np.asarray(got, dtype=np.uint16)
    ref = np.asarray(ref, dtype=np.uint16)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    g = bf16_bits_to_f64(got)
    r = bf16_bits_to_f64(ref)
    exact = got == ref
    # +0 and -0 compare equal as values; count them as exact matches
    exact |= (g == 0) & (r == 0)
    nan_r, nan_g = np.isnan(r), np.isnan(g)
    exact |= nan_r & nan_g          # any NaN payload matches NaN
    assert np.array_equal(nan_r, nan_g), (
        f"NaN mismatch: ref NaN {int(nan_r.sum())}, got NaN {int(nan_g.sum())}, "
        f"first at {np.argwhere(nan_r != nan_g)[:4].tolist()}")
    fin = ~nan_r
    with np.errstate(invalid="ignore"):
        err = np.abs(g - r)
        bound = rel * np.abs(r) + abs_
        if extra is not None:
            bound = bound + extra
        bad = fin & ~(err <= bound)
    n = got.size
    stats = dict(n=n, exact_frac=float(exact.sum()) / max(n, 1),
                 max_abs_err=float(err[fin].max()) if fin.any() else 0.0,
                 n_bad=int(bad.sum()))
    if bad.any():
        where = np.argwhere(bad)[:5]
        detail = [(tuple(int(i) for i in w), float(g[tuple(w)]), float(r[tuple(w)])) for w in where]
        raise AssertionError(f"{int(bad.sum())} elements outside the 1-ulp bound: {detail}")
    log = os.environ.get("MF_PARITY_LOG")
    if log:  # optional record of the per-test statistics
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", ""), **stats}) + "\n")
    assert stats["exact_frac"] >= min_exact, f"bit-exact fraction {stats['exact_frac']:.6f} < {min_exact}"
    return stats
