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
    """Round float64 to BF16 in one step, to nearest with ties to even (used
    only by independent checks).  Normal range: the float64 encoding keeps its
    top 19 bits (sign, 11 exponent bits, the 7 fraction bits BF16 stores); the
    45 bits dropped round half to even, and a carry out of the fraction moves
    into the exponent as it should.  Below 2^-126 BF16 is subnormal with a fixed
    step of 2^-133: adding and subtracting 1.5 * 2^-81, whose float64 ulp is that
    step, makes the FPU round there.  Results past the BF16 maximum overflow to
    infinity in the final (exact otherwise) conversion to float32."""
    x = np.asarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    drop = np.uint64((1 << 45) - 1)
    kept = (u + ((u >> np.uint64(45)) & np.uint64(1)) + (drop >> np.uint64(1))) & ~drop
    y = kept.view(np.float64)
    tiny = np.abs(x) < 2.0 ** -126
    if tiny.any():
        c = 1.5 * 2.0 ** -81
        y = np.where(tiny, np.copysign((np.abs(x) + c) - c, x), y)
    with np.errstate(over="ignore"):
        f = y.astype(np.float32)
    out = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    out[np.isnan(x)] = 0x7FC0
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return f64_to_bf16_bits(np.asarray(x, dtype=np.float32).astype(np.float64))


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at each element (16 fewer significand bits than float32)."""
    f = np.abs(bf16_bits_to_f64(bits)).astype(np.float32)
    return np.spacing(f).astype(np.float64) * 65536.0


# With a widened bound (``extra``), at most this fraction of the elements may
# fall outside the plain bound above (at least one element is always allowed).
# The widening covers a BF16 rounding boundary that an intermediate value lands
# on from the other side (FP32 norm on the GPU, float64 in the oracle), which
# happens to about 1e-5 of the values; more than 1e-4 means a real error.
MAX_WIDENED_FRAC = 1e-4


def compare_bf16(got: np.ndarray, ref: np.ndarray, *, rel: float = REL_TOL, abs_: float = ABS_TOL,
                 min_exact: float = MIN_EXACT, extra: np.ndarray | None = None,
                 max_widened_frac: float = MAX_WIDENED_FRAC) -> dict:
    """Element-wise check of BF16 bit arrays; returns stats, raises AssertionError.
    ``extra`` (same shape) widens the bound per element where an intermediate
    BF16 rounding propagates (the caller derives it); the elements that need
    the widening (outside the plain bound, inside the widened one) are counted
    as ``n_widened`` and capped at ``max_widened_frac`` of the elements."""
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
        plain = rel * np.abs(r) + abs_
        bound = plain if extra is None else plain + extra
        bad = fin & ~(err <= bound)
        widened = fin & ~(err <= plain) & ~bad
    n = got.size
    stats = dict(n=n, exact_frac=float(exact.sum()) / max(n, 1),
                 max_abs_err=float(err[fin].max()) if fin.any() else 0.0,
                 n_bad=int(bad.sum()), n_widened=int(widened.sum()))
    if bad.any():
        where = np.argwhere(bad)[:5]
        detail = [(tuple(int(i) for i in w), float(g[tuple(w)]), float(r[tuple(w)])) for w in where]
        raise AssertionError(f"{int(bad.sum())} elements outside the 1-ulp bound: {detail}")
    log = os.environ.get("MF_PARITY_LOG")
    if log:  # optional record of the per-test statistics
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", ""), **stats}) + "\n")
    assert stats["exact_frac"] >= min_exact, f"bit-exact fraction {stats['exact_frac']:.6f} < {min_exact}"
    allowed = max(1, int(max_widened_frac * n))
    assert stats["n_widened"] <= allowed, (
        f"{stats['n_widened']} of {n} elements need the widened bound (at most {allowed}): "
        f"first at {np.argwhere(widened)[:4].tolist()}")
    return stats
