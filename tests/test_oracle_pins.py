"""Pins of the CPU oracle to facts other than itself (CPU only).

The pages print no worked values, so the pins are: hand-worked examples
(derivations in the comments), closed forms, invariants, special cases that
reduce to a library routine (PyTorch's BF16 rounding, its float64 RMSNorm),
and an independent float64 brute force on small inputs.  Each is chosen so a
plausible slip in the oracle -- a dropped term, a wrong sign or index, a
transposed operand, eps outside the square root, the gain in the wrong place,
a missing BF16 round in the Beam path -- fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import bf16_bits_to_f64, compare_bf16, f32_to_bf16_bits, f64_to_bf16_bits

ONE = np.uint16(0x3F80)


def bits(values):
    """BF16 bits of values that are exactly representable in BF16."""
    a = np.asarray(values, dtype=np.float32)
    b = f32_to_bf16_bits(a)
    assert np.array_equal(bf16_bits_to_f64(b), a.astype(np.float64)), "not a BF16 value"
    return b


def vals(b):
    return bf16_bits_to_f64(b).tolist()


# --------------------------------------------------------------------------
# BF16 rounding (the format: the upper 16 bits of binary32, RNE)

@pytest.mark.parametrize("x,expected", [
    (1.0, 0x3F80),
    (-1.5, 0xBFC0),
    (1.0 + 2 ** -8, 0x3F80),                # tie between 1 and 1+2^-7 -> even (1)
    (1.0 + 3 * 2 ** -8, 0x3F82),            # tie between 1+2^-7 and 1+2^-6 -> even
    (1.0 + 2 ** -8 + 2 ** -40, 0x3F81),     # just above the tie -> up
    (1.0 + 2 ** -8 - 2 ** -40, 0x3F80),     # just below the tie -> down
    (2 ** -133, 0x0001),                    # smallest subnormal
    (2 ** -134, 0x0000),                    # tie between 0 and 2^-133 -> even (0)
    (3 * 2 ** -134, 0x0002),                # tie between 1 and 2 quanta -> even (2)
    (-(2 ** -134) * 1.5, 0x8001),           # 0.75 quanta, negative
    ((2 - 2 ** -7) * 2 ** 127, 0x7F7F),     # largest finite BF16
    (2 ** 128 - 2 ** 119, 0x7F80),          # tie above the largest finite -> +inf
    (-(2 ** 129), 0xFF80),                  # overflow -> -inf
    (float("inf"), 0x7F80),
    (float("nan"), 0x7FC0),
    (-0.0, 0x8000),
    (0.0, 0x0000),
])
def test_bf16_rounding_table(x, expected):
    assert oracle.bf16_from_double(x) == expected


def _nearest_bf16_exact(x: float) -> int:
    """BF16 bits nearest to x in exact rational arithmetic (ties to the even
    code), by search over the sorted positive codes; 2^128 stands for +inf."""
    from fractions import Fraction
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    ax = Fraction(abs(x))
    codes = _POSITIVE_CODES
    value = (lambda c: Fraction(2) ** 128 if c == 0x7F80 else
             Fraction(float(bf16_bits_to_f64(np.uint16(c)))))
    lo, hi = 0, len(codes) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if value(codes[mid]) <= ax:
            lo = mid
        else:
            hi = mid
    dl, dh = ax - value(codes[lo]), value(codes[hi]) - ax
    if dl < 0:
        return sign | codes[lo]
    pick = codes[lo] if (dl < dh or (dl == dh and codes[lo] % 2 == 0)) else codes[hi]
    return sign | int(pick)


_POSITIVE_CODES = list(range(0, 0x7F81))


def test_independent_bf16_round_of_the_checks_is_exact():
    # the one-step float64 -> BF16 round that the brute-force checks use is
    # itself pinned: the hand table above, then exact rational rounding on
    # random magnitudes across the whole range, exact ties and their neighbours
    for x, expected in [(1.0 + 2 ** -8, 0x3F80), (1.0 + 3 * 2 ** -8, 0x3F82),
                        (2 ** -134, 0), (3 * 2 ** -134, 2), (-(2 ** -134) * 1.5, 0x8001),
                        (2 ** 128 - 2 ** 119, 0x7F80), (-(2 ** 129), 0xFF80), (-0.0, 0x8000),
                        (float("inf"), 0x7F80), (float("nan"), 0x7FC0)]:
        assert int(f64_to_bf16_bits(np.array([x]))[0]) == expected, x
    rng = np.random.default_rng(5)
    mags = rng.standard_normal(600) * 10.0 ** rng.integers(-44, 39, 600)
    codes = (rng.integers(0, 0x7F7F, 300).astype(np.uint32) << 16).view(np.float32)
    f = codes.astype(np.float64)
    half = np.spacing(np.abs(codes)).astype(np.float64) * 32768.0
    x = np.concatenate([mags, f + half, -(f + half), f + half * (1 + 2 ** -30),
                        f + half * (1 - 2 ** -30)])
    got = f64_to_bf16_bits(x)
    want = np.array([_nearest_bf16_exact(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5].ravel()


def test_bf16_rounding_matches_torch_on_float32_values():
    # every float32 value reduces the double -> BF16 rounding to PyTorch's
    # float -> BF16 conversion (a library routine); take random bit patterns
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    u[:8] = [0x00000001, 0x00008000, 0x007FFFFF, 0x7F7FFFFF, 0x7F7F8000, 0x3F808000, 0x3F818000, 0x80000000]
    f = u.view(np.float32)
    f = f[~np.isnan(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# tp_moe_finalize_rmsnorm: hand-worked examples

def _p1_inputs():
    # rows r0 = [1,2,3,4], r1 = [4,3,2,1]; token 0 uses slots (0, 1, -1)
    gemm2 = bits([[1, 2, 3, 4], [4, 3, 2, 1]])
    idx = np.array([[0, 1, -1]], dtype=np.int32)
    w = np.array([[0.5, 0.25, np.nan]], dtype=np.float32)   # NaN on the invalid slot
    return gemm2, idx, w


@pytest.mark.parametrize("before", [False, True])
def test_hand_example_unit_gain(before):
    # acc = 0.5*r0 + 0.25*r1 = [1.5, 1.75, 2.0, 2.25]
    # mean square = (2.25 + 3.0625 + 4 + 5.0625) / 4 = 3.59375, eps = 0
    # y = acc / sqrt(3.59375) = [0.791257, 0.923133, 1.055009, 1.186885]
    # BF16 (spacing 2^-8 below 1, 2^-7 above): [0.79296875, 0.921875, 1.0546875, 1.1875]
    gemm2, idx, w = _p1_inputs()
    nw = bits([1, 1, 1, 1])
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=0.0, gain_center=0.0,
                                      weight_before_norm=before)
    assert vals(out[0]) == [0.79296875, 0.921875, 1.0546875, 1.1875]


def test_hand_example_gain_after_norm():
    # norm_weight [0.5, -1, 2, 0] + gain_center 1 -> g = [1.5, 0, 3, 1]
    # after: y = acc / sqrt(3.59375) * g = [1.186885, 0, 3.165026, 1.186885]
    gemm2, idx, w = _p1_inputs()
    nw = bits([0.5, -1, 2, 0])
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=0.0, gain_center=1.0,
                                      weight_before_norm=False)
    assert vals(out[0]) == [1.1875, 0.0, 3.171875, 1.1875]


def test_hand_example_gain_before_norm():
    # before: v = acc * g = [2.25, 0, 6, 2.25]; mean square = (5.0625+36+5.0625)/4
    # = 11.53125; y = v / sqrt(11.53125) = [0.662589, 0, 1.766904, 0.662589]
    gemm2, idx, w = _p1_inputs()
    nw = bits([0.5, -1, 2, 0])
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=0.0, gain_center=1.0,
                                      weight_before_norm=True)
    assert vals(out[0]) == [0.6640625, 0.0, 1.765625, 0.6640625]


def test_negative_weight_and_values_sign():
    # acc = -0.5*[1,-2] + 1*[2,2] = [1.5, 3]; ms = (2.25+9)/2 = 5.625
    # y = acc/sqrt(5.625) = [0.632456, 1.264911] -> BF16 [0.6328125, 1.265625]
    gemm2 = bits([[1, -2], [2, 2]])
    idx = np.array([[0, 1]], dtype=np.int32)
    w = np.array([[-0.5, 1.0]], dtype=np.float32)
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, bits([1, 1]), eps=0.0, gain_center=0.0,
                                      weight_before_norm=False)
    assert vals(out[0]) == [0.6328125, 1.265625]


def test_hand_example_packed_routing_words():
    # the producer's packed words (expert_id << 16) | bf16 bits: expert 5 with
    # 0.5 (0x3F00), expert 40000 with 0.25 (0x3E80; the word is negative as
    # int32), and an invalid slot whose word holds a BF16 NaN -- the same sums
    # as the unit-gain hand example, so the same output
    gemm2, idx, _ = _p1_inputs()
    packed = np.array([[(5 << 16) | 0x3F00, (40000 << 16) | 0x3E80, (0xFFFF << 16) | 0x7FC0]],
                      dtype=np.uint32).view(np.int32)
    out = oracle.moe_finalize_rmsnorm(gemm2, packed, idx, bits([1, 1, 1, 1]), eps=0.0,
                                      gain_center=0.0, weight_before_norm=False)
    assert vals(out[0]) == [0.79296875, 0.921875, 1.0546875, 1.1875]


def test_packed_words_equal_bf16_weights():
    # the expert id in the high half never matters; the low half is the weight
    rng = np.random.default_rng(14)
    gemm2, idx, w, nw = _random_case(rng)
    wb = f32_to_bf16_bits(w)
    experts = rng.integers(0, 65536, size=w.shape).astype(np.uint32)
    packed = ((experts << 16) | wb.astype(np.uint32)).view(np.int32)
    for before in (False, True):
        a = oracle.moe_finalize_rmsnorm(gemm2, wb, idx, nw, eps=1e-6, gain_center=1.0,
                                        weight_before_norm=before)
        b = oracle.moe_finalize_rmsnorm(gemm2, packed, idx, nw, eps=1e-6, gain_center=1.0,
                                        weight_before_norm=before)
        assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# closed forms

@pytest.mark.parametrize("before", [False, True])
@pytest.mark.parametrize("c,eps,expected", [
    (1.0, 3.0, 0.5),          # 1/sqrt(1+3): eps inside the root (outside would give 0.25)
    (2.0, 12.0, 0.5),         # 2/sqrt(4+12)
    (-0.5, 0.75, -0.5),       # -0.5/sqrt(0.25+0.75)
    (3.0, 0.0, 1.0),
    (1.0, 1e-6, 1.0),         # 0.9999995 rounds to 1.0
])
def test_constant_rows_closed_form(c, eps, expected, before):
    # all 8 slots valid, every row = c, weights 1/8: acc = c exactly;
    # with g = 1, y = c / sqrt(c^2 + eps) for both orderings
    rows = np.full((8, 16), c, dtype=np.float32)
    gemm2 = bits(rows)
    idx = np.arange(8, dtype=np.int32)[None, :]
    w = np.full((1, 8), 0.125, dtype=np.float32)
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, bits(np.zeros(16)), eps=eps,
                                      gain_center=1.0, weight_before_norm=before)
    assert set(vals(out[0])) == {expected}


def test_constant_rows_with_gain_after_norm():
    # y_h = g_h * c / sqrt(c^2 + eps) with c = 1, eps = 3 -> 0.5 * g_h
    gemm2 = bits(np.ones((8, 4)))
    idx = np.arange(8, dtype=np.int32)[None, :]
    w = np.full((1, 8), 0.125, dtype=np.float32)
    nw = bits([0.5, 1.0, -3.0, 2.0])
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=3.0, gain_center=0.25,
                                      weight_before_norm=False)
    # g = [0.75, 1.25, -2.75, 2.25]
    assert vals(out[0]) == [0.375, 0.625, -1.375, 1.125]


@pytest.mark.parametrize("before", [False, True])
def test_all_invalid_slots_give_zero(before):
    # every slot invalid -> acc = 0 -> y = 0 * 1/sqrt(eps) * g = 0 everywhere
    # (-0 where the gain is negative); the NaN weights of invalid slots are
    # never read
    rng = np.random.default_rng(3)
    rows = 5
    gemm2 = f32_to_bf16_bits(rng.standard_normal((rows, 32)).astype(np.float32))
    idx = np.array([[-1, rows, np.iinfo(np.int32).min, np.iinfo(np.int32).max] * 2] * 3,
                   dtype=np.int32)
    w = np.full(idx.shape, np.nan, dtype=np.float32)
    nw = f32_to_bf16_bits(rng.standard_normal(32).astype(np.float32))
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=1e-6, gain_center=1.0,
                                      weight_before_norm=before)
    assert np.all(bf16_bits_to_f64(out) == 0.0)


def test_all_invalid_with_zero_eps_is_nan():
    # the degenerate case: 0 * 1/sqrt(0) = 0 * inf = NaN (the formula as written)
    gemm2 = bits(np.ones((2, 8)))
    idx = np.full((1, 8), -1, dtype=np.int32)
    w = np.ones((1, 8), dtype=np.float32)
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, bits(np.ones(8)), eps=0.0,
                                      gain_center=0.0, weight_before_norm=False)
    assert np.all(np.isnan(bf16_bits_to_f64(out)))


# --------------------------------------------------------------------------
# special cases that reduce to a library routine

@pytest.mark.parametrize("before", [False, True])
@pytest.mark.parametrize("slot,weight", [(0, 1.0), (3, 0.25), (7, 4.0), (5, -2.0)])
def test_single_valid_slot_is_textbook_rmsnorm(slot, weight, before):
    # one valid slot with a power-of-two weight w: acc = w * x exactly, and
    # RMSNorm with eps scales with it: rmsnorm(w x; eps) = sign(w) rmsnorm(x; eps / w^2).
    # Compare with PyTorch's float64 rms_norm on the gathered row.
    rng = np.random.default_rng(100 + slot)
    H, R = 4096, 40
    gemm2 = f32_to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    nw = f32_to_bf16_bits((0.1 * rng.standard_normal(H)).astype(np.float32))
    gc, eps = 1.0, 1e-3
    row = 17
    idx = np.full((1, 8), -1, dtype=np.int32)
    idx[0, slot] = row
    idx[0, (slot + 1) % 8] = R          # out of range by one: invalid
    w = rng.standard_normal((1, 8)).astype(np.float32)
    w[0, slot] = weight
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=eps, gain_center=gc,
                                      weight_before_norm=before)
    x = torch.from_numpy(bf16_bits_to_f64(gemm2[row])) * weight
    g = torch.from_numpy((bf16_bits_to_f64(nw).astype(np.float32) + np.float32(gc)).astype(np.float64))
    if before:
        y = torch.nn.functional.rms_norm(x * g, (H,), None, eps)
    else:
        y = torch.nn.functional.rms_norm(x, (H,), g, eps)
    ref = y.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    compare_bf16(out[0], ref, min_exact=0.999)


# --------------------------------------------------------------------------
# independent float64 brute force (vectorised numpy; no FP32 intermediates)

def _brute_tp(gemm2, w, idx, nw, eps, gc, before, hidden):
    rows = gemm2.shape[0]
    x = bf16_bits_to_f64(gemm2[:, :hidden])
    wf = w.astype(np.float64) if w.dtype == np.float32 else bf16_bits_to_f64(w)
    valid = (idx >= 0) & (idx < rows)
    safe = np.where(valid, idx, 0)
    contrib = np.where(valid[:, :, None], wf[:, :, None] * x[safe], 0.0)   # [T, K, H]
    acc = contrib.sum(axis=1)
    g = (bf16_bits_to_f64(nw).astype(np.float32) + np.float32(gc)).astype(np.float64)
    v = acc * g if before else acc
    r = 1.0 / np.sqrt((v * v).mean(axis=1, keepdims=True) + eps)
    y = v * r if before else acc * r * g
    return f64_to_bf16_bits(y)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("before", [False, True])
def test_oracle_matches_float64_brute_force(seed, before):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 9))
    K = int(rng.integers(1, 9))
    H = [8, 64, 4096][seed % 3]
    stride = H + 8 * int(rng.integers(0, 3))
    R = int(rng.integers(T * K, 3 * T * K + 2))
    gemm2 = f32_to_bf16_bits(rng.standard_normal((R, stride)).astype(np.float32) * 2)
    gemm2[:, H:] = 0x7FC0                                    # NaN padding columns
    idx = rng.integers(-3, R + 3, size=(T, K)).astype(np.int32)
    wdtype = "fp32" if seed % 2 else "bf16"
    w = rng.random((T, K)).astype(np.float32)
    if wdtype == "bf16":
        w = f32_to_bf16_bits(w)
    nw = f32_to_bf16_bits((0.1 * rng.standard_normal(H)).astype(np.float32))
    eps, gc = [1e-6, 1e-5, 0.5][seed % 3], [1.0, 0.0, 0.5][seed % 3]
    got = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=eps, gain_center=gc,
                                      weight_before_norm=before, hidden=H)
    ref = _brute_tp(gemm2, w, idx, nw, eps, gc, before, H)
    compare_bf16(got, ref, min_exact=0.99)


# --------------------------------------------------------------------------
# invariants

def _random_case(rng, T=6, K=8, H=64, R=60):
    gemm2 = f32_to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    idx = rng.integers(-2, R + 2, size=(T, K)).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    nw = f32_to_bf16_bits((0.1 * rng.standard_normal(H)).astype(np.float32))
    return gemm2, idx, w, nw


@pytest.mark.parametrize("before", [False, True])
def test_physical_row_order_does_not_matter(before):
    # permuting the physical rows and remapping the index map accordingly
    # leaves every output bit unchanged
    rng = np.random.default_rng(7)
    gemm2, idx, w, nw = _random_case(rng)
    R = gemm2.shape[0]
    perm = rng.permutation(R)              # new row j holds old row perm[j]
    inv = np.argsort(perm)
    idx2 = np.where((idx >= 0) & (idx < R), inv[np.clip(idx, 0, R - 1)], idx).astype(np.int32)
    a = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=before)
    b = oracle.moe_finalize_rmsnorm(np.ascontiguousarray(gemm2[perm]), w, idx2, nw, eps=1e-6,
                                    gain_center=1.0, weight_before_norm=before)
    assert np.array_equal(a, b)


def test_token_order_does_not_matter():
    rng = np.random.default_rng(8)
    gemm2, idx, w, nw = _random_case(rng)
    p = rng.permutation(idx.shape[0])
    a = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=False)
    b = oracle.moe_finalize_rmsnorm(gemm2, np.ascontiguousarray(w[p]), np.ascontiguousarray(idx[p]),
                                    nw, eps=1e-6, gain_center=1.0, weight_before_norm=False)
    assert np.array_equal(a[p], b)


def test_row_padding_is_never_read():
    # padded columns full of NaN and padding rows full of NaN leave the output
    # identical to the unpadded layout (the mean runs over `hidden` columns only)
    rng = np.random.default_rng(9)
    gemm2, idx, w, nw = _random_case(rng, H=64)
    R, H = gemm2.shape
    padded = np.full((R + 7, H + 24), 0x7FC0, dtype=np.uint16)
    padded[:R, :H] = gemm2
    idx2 = np.where(idx == R, R + 7, idx).astype(np.int32)   # keep out-of-range out of range
    a = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=True)
    b = oracle.moe_finalize_rmsnorm(padded, w, idx2, nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=True, hidden=H)
    assert np.array_equal(a, b)


def test_last_row_valid_first_past_end_invalid():
    # idx = rows-1 contributes, idx = rows does not
    gemm2 = bits([[1, 1], [2, -2], [5, 1]])
    nw = bits([1, 1])
    w = np.array([[1.0, 1.0]], dtype=np.float32)
    a = oracle.moe_finalize_rmsnorm(gemm2, w, np.array([[2, 3]], np.int32), nw, eps=0.0,
                                    gain_center=0.0, weight_before_norm=False)
    # acc = [5, 1]; ms = 13; y = [5, 1]/sqrt(13) = [1.386750, 0.277350]
    assert vals(a[0]) == [1.390625, 0.27734375]


def test_duplicate_index_equals_summed_weight():
    rng = np.random.default_rng(12)
    gemm2 = f32_to_bf16_bits(rng.standard_normal((4, 32)).astype(np.float32))
    nw = f32_to_bf16_bits(rng.standard_normal(32).astype(np.float32))
    a = oracle.moe_finalize_rmsnorm(gemm2, np.array([[0.25, 0.25]], np.float32),
                                    np.array([[3, 3]], np.int32), nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=False)
    b = oracle.moe_finalize_rmsnorm(gemm2, np.array([[0.5, 9.0]], np.float32),
                                    np.array([[3, -1]], np.int32), nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=False)
    assert np.array_equal(a, b)


def test_bf16_and_fp32_weights_with_equal_values_agree():
    rng = np.random.default_rng(13)
    gemm2, idx, w, nw = _random_case(rng)
    wb = f32_to_bf16_bits(w)
    wf = bf16_bits_to_f64(wb).astype(np.float32)
    a = oracle.moe_finalize_rmsnorm(gemm2, wb, idx, nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=True)
    b = oracle.moe_finalize_rmsnorm(gemm2, wf, idx, nw, eps=1e-6, gain_center=1.0,
                                    weight_before_norm=True)
    assert np.array_equal(a, b)


def test_reduction_is_fp32_in_slot_order():
    # the routing reduction stays in FP32 and adds the slots in ascending order:
    # column 0 holds 2^24, 1, -2^24.  FP32: 2^24 + 1 is a tie that rounds to
    # 2^24 (even), minus 2^24 gives 0.  A float64 sum (or the slots in another
    # order) gives 1.  Column 1 holds 0, 1, 0 and pins the scale:
    # FP32 acc = [0, 1] -> y = [0, sqrt(2)] -> BF16 [0, 1.4140625];
    # the other readings give acc = [1, 1] -> y = [1, 1].
    x = np.array([[2.0 ** 24, 0.0], [1.0, 1.0], [-(2.0 ** 24), 0.0]], dtype=np.float32)
    gemm2 = bits(x)
    idx = np.array([[0, 1, 2]], dtype=np.int32)
    w = np.ones((1, 3), dtype=np.float32)
    out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, bits([1, 1]), eps=0.0, gain_center=0.0,
                                      weight_before_norm=False)
    assert vals(out[0]) == [0.0, 1.4140625]


def test_reduction_fuses_each_slot_into_one_rounding():
    # each slot is one fused multiply-add (a single rounding of w * x + acc), the
    # reading the kernels reproduce bit for bit.  w = 1 + 2^-17 (FP32) on the
    # BF16 rows x0 = -(1 + 2^-7) and x1 = 1 + 2^-7 (every column):
    #   slot 0: w * x0 = -(1 + 2^-7 + 2^-17 + 2^-24), rounded (a tie, to even)
    #           to -(1 + 2^-7 + 2^-17) = acc
    #   slot 1: fused, w * x1 + acc = 2^-24 exactly; unfused, the product rounds
    #           to 1 + 2^-7 + 2^-17 first and the sum is 0.
    # With gain 1 and eps 2^-100, acc = 2^-24 in every column gives y = 1.0;
    # an unfused reduction gives acc = 0 and y = 0.
    x = np.array([[-(1 + 2.0 ** -7)] * 4, [1 + 2.0 ** -7] * 4], dtype=np.float32)
    w = np.full((1, 2), 1 + 2.0 ** -17, dtype=np.float32)
    idx = np.array([[0, 1]], dtype=np.int32)
    for before in (False, True):
        out = oracle.moe_finalize_rmsnorm(bits(x), w, idx, bits([1, 1, 1, 1]), eps=2.0 ** -100,
                                          gain_center=0.0, weight_before_norm=before)
        assert vals(out[0]) == [1.0] * 4
    # the same in Beam's reduction: BF16(2^-24) times scale 1 is 2^-24 exactly
    beam = oracle.beam_moe_finalize(bits(x)[None, :, :1].copy(), w, 1, routed_scale=1.0)
    assert vals(beam[0]) == [2.0 ** -24]


def test_gain_center_is_added_in_fp32():
    # the API page adds gain_center to norm_weight in FP32: with norm_weight 2^-30
    # and gain_center 1 + 2^-8, the FP32 sum drops 2^-30 (under half an FP32 ulp)
    # and g = 1 + 2^-8 exactly.  A constant row of ones with weight 1 and eps 0
    # gives acc / rms = 1, so y = g = 1 + 2^-8: a BF16 tie, to even -> 1.0.  A
    # float64 add keeps 1 + 2^-8 + 2^-30, which rounds up to 1 + 2^-7.
    out = oracle.moe_finalize_rmsnorm(bits([[1, 1, 1, 1]]), np.ones((1, 1), dtype=np.float32),
                                      np.zeros((1, 1), dtype=np.int32),
                                      bits([2.0 ** -30] * 4), eps=0.0,
                                      gain_center=1 + 2.0 ** -8, weight_before_norm=False)
    assert vals(out[0]) == [1.0] * 4


# --------------------------------------------------------------------------
# beam_moe_finalize

def test_beam_identity():
    # top_k 1, weight 1, scale 1, no norm: the output is the input, bit for bit
    rng = np.random.default_rng(20)
    x = f32_to_bf16_bits(rng.standard_normal((5, 1, 256)).astype(np.float32) * 3)
    w = np.ones((5, 1), dtype=np.float32)
    out = oracle.beam_moe_finalize(x, w, 5)
    assert np.array_equal(out, x[:, 0, :])


def test_beam_scale_is_an_fp32_product():
    # the scale multiplies the BF16 sum as PyTorch's BF16 tensor times a scalar:
    # one FP32 product, then BF16.  r = 1 + 2^-7 and the FP32 scale
    # s = 16712189 * 2^-24: r * s = 1 + 2^-8 + 5.8e-8 exactly, which FP32 rounds
    # to 1 + 2^-8 (the excess is under half an FP32 ulp); that is a BF16 tie,
    # to even -> 1.0.  A float64 product keeps the excess and rounds to 1 + 2^-7.
    x = bits([[[1 + 2.0 ** -7] * 4]])
    s = 16712189 * 2.0 ** -24
    assert float(np.float32(s)) == s
    out = oracle.beam_moe_finalize(x, np.ones((1, 1), dtype=np.float32), 1, routed_scale=s)
    assert vals(out[0]) == [1.0] * 4


def test_beam_rounds_sum_before_scale():
    # s = 1 + 2^-8 is a tie: BF16(s) = 1 (even); 1 * 2.5 = 2.5.
    # A single final rounding would give BF16(2.509765625) = 2.515625.
    x = bits([[[1.0], [2 ** -8]]])
    w = np.ones((1, 2), dtype=np.float32)
    out = oracle.beam_moe_finalize(x, w, 1, routed_scale=2.5)
    assert vals(out[0]) == [2.5]


def test_beam_rounds_scaled_value_before_norm():
    # x = [1, 1.0078125, 1.015625, 1.0234375] (K = 1, w = 1), scale 2.5:
    # v = BF16(2.5 x) = [2.5, 2.515625, 2.53125, 2.5625]   (2.51953125 -> 2.515625,
    # 2.5390625 -> 2.53125, 2.55859375 -> 2.5625, spacing 2^-6, ties to even)
    # y = v / sqrt(mean v^2 + 1e-6) = [0.989139, 0.995322, 1.001504, 1.013868]
    # -> BF16 [0.98828125, 0.99609375, 1.0, 1.015625]; without the round of v the
    # last element would be 1.0078125
    x = bits([[[1.0, 1.0078125, 1.015625, 1.0234375]]])
    w = np.ones((1, 1), dtype=np.float32)
    out = oracle.beam_moe_finalize(x, w, 1, routed_scale=2.5, post_weight=bits([1, 1, 1, 1]),
                                   post_eps=1e-6)
    assert vals(out[0]) == [0.98828125, 0.99609375, 1.0, 1.015625]


def test_beam_no_norm_is_two_rounds():
    # s = 0.5*1.5 + 0.5*2.25 = 1.875; BF16 exact; * 3 = 5.625 exact
    x = bits([[[1.5, -1.0], [2.25, 0.5]]])
    w = np.array([[0.5, 0.5]], dtype=np.float32)
    out = oracle.beam_moe_finalize(x, w, 1, routed_scale=3.0)
    assert vals(out[0]) == [5.625, -0.75]


def test_beam_norm_matches_library_rmsnorm():
    # top_k 1 with weight 1: the reduction is the identity, the scale is
    # PyTorch's BF16 tensor * scalar (FP32 product, RNE), the norm is float64
    # rms_norm with the BF16 weight
    rng = np.random.default_rng(21)
    T, H = 4, 7168
    x = f32_to_bf16_bits(rng.standard_normal((T, 1, H)).astype(np.float32))
    pw = f32_to_bf16_bits((1 + 0.05 * rng.standard_normal(H)).astype(np.float32))
    w = np.ones((T, 1), dtype=np.float32)
    out = oracle.beam_moe_finalize(x, w, T, routed_scale=2.5, post_weight=pw, post_eps=1e-6)
    xt = torch.from_numpy(x[:, 0, :].view(np.int16).copy()).view(torch.bfloat16)
    v = (xt * 2.5).double()
    y = torch.nn.functional.rms_norm(v, (H,), torch.from_numpy(bf16_bits_to_f64(pw)), 1e-6)
    ref = y.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    compare_bf16(out, ref, min_exact=0.999)


def test_beam_unweighted_norm_when_post_weight_absent():
    rng = np.random.default_rng(22)
    x = f32_to_bf16_bits(rng.standard_normal((3, 2, 256)).astype(np.float32))
    w = rng.random((3, 2)).astype(np.float32)
    a = oracle.beam_moe_finalize(x, w, 3, routed_scale=1.5, post_weight=None, post_eps=1e-5)
    b = oracle.beam_moe_finalize(x, w, 3, routed_scale=1.5, post_weight=bits(np.ones(256)),
                                 post_eps=1e-5)
    assert np.array_equal(a, b)


def test_beam_writes_only_live_rows():
    rng = np.random.default_rng(23)
    x = f32_to_bf16_bits(rng.standard_normal((6, 3, 256)).astype(np.float32))
    x[4:] = 0x7FC0                                      # dead rows: NaN, never read
    w = rng.random((6, 3)).astype(np.float32)
    w[4:] = np.nan
    out = np.full((6, 256), 0x1234, dtype=np.uint16)     # canary past the live rows
    oracle.beam_moe_finalize(x, w, 4, routed_scale=2.0, post_weight=None, post_eps=1e-6, out=out)
    assert np.all(out[4:] == 0x1234)
    assert not np.isnan(bf16_bits_to_f64(out[:4])).any()


def _brute_beam(x, w, live, scale, pw, eps):
    s = np.einsum("tkh,tk->th", bf16_bits_to_f64(x[:live]), w[:live].astype(np.float64))
    r = bf16_bits_to_f64(f64_to_bf16_bits(s))
    v = bf16_bits_to_f64(f32_to_bf16_bits((r * scale).astype(np.float32)))
    if eps is None:
        return f64_to_bf16_bits(v)
    y = v / np.sqrt((v * v).mean(axis=1, keepdims=True) + eps)
    if pw is not None:
        y = y * bf16_bits_to_f64(pw)
    return f64_to_bf16_bits(y)


@pytest.mark.parametrize("seed", range(4))
def test_beam_matches_float64_brute_force(seed):
    # the brute force sums in float64, so its BF16 round of the sum can differ
    # by one step from the FP32 sum's in rare ties; after a 1.0 scale that is
    # still one ulp, within the acceptance bound
    rng = np.random.default_rng(40 + seed)
    cap, K, H = 7, [1, 3, 8, 32][seed], [256, 512, 1024, 256][seed]
    live = int(rng.integers(1, cap + 1))
    x = f32_to_bf16_bits(rng.standard_normal((cap, K, H)).astype(np.float32))
    w = rng.random((cap, K)).astype(np.float32)
    pw = f32_to_bf16_bits((1 + 0.05 * rng.standard_normal(H)).astype(np.float32))
    eps = None if seed == 1 else 1e-6
    got = oracle.beam_moe_finalize(x, w, live, routed_scale=1.0,
                                   post_weight=pw if eps else None, post_eps=eps)
    ref = _brute_beam(x, w, live, 1.0, pw if eps else None, eps)
    compare_bf16(got, ref, min_exact=0.99)


def test_beam_reduction_equals_tp_gather_with_identity_map():
    # token-major rows with the identity route map idx[t,k] = t*K + k: the tp
    # oracle's FP32 reduction and the Beam oracle's are the same sum.  With
    # scale 1 and no BF16 tie in between, Beam(no norm) rounds that sum to BF16;
    # tp with g = 1 and a huge eps returns acc/sqrt(eps) -- compare the two
    # through the exact scaling by 2^k: eps = 2^40 gives y = acc * 2^-20.
    rng = np.random.default_rng(50)
    cap, K, H = 5, 4, 256
    x = f32_to_bf16_bits(rng.standard_normal((cap, K, H)).astype(np.float32))
    w = rng.random((cap, K)).astype(np.float32)
    beam = oracle.beam_moe_finalize(x, w, cap, routed_scale=1.0)
    gemm2 = np.ascontiguousarray(x.reshape(cap * K, H))
    idx = np.arange(cap * K, dtype=np.int32).reshape(cap, K)
    tp = oracle.moe_finalize_rmsnorm(gemm2, w, idx, bits(np.zeros(H)), eps=2.0 ** 40,
                                     gain_center=1.0, weight_before_norm=False)
    # mean square is tiny against 2^40, so y = acc * 2^-20 * (1 - tiny): compare
    # after undoing the power of two; the (1 - tiny) factor only matters at ties
    tp_scaled = bf16_bits_to_f64(tp) * 2.0 ** 20
    compare_bf16(f64_to_bf16_bits(tp_scaled), beam, min_exact=0.99)
    assert math.isfinite(float(tp_scaled.max()))


# --------------------------------------------------------------------------
# beam_moe_finalize_norm_residual_norm (the residual step is partly unpinned:
# hidden = BF16(s0 x + s1 residual) in FP32, normalized = BF16(RMSNorm(hidden)))

def _identity_beam(values):
    """expert_outputs with top_k 1 holding `values`, unit weights: the Beam
    finalize (scale 1, no norm) returns them unchanged."""
    x = bits([[list(v)] for v in values])
    return x, np.ones((x.shape[0], 1), dtype=np.float32)


def test_residual_add_hand_example():
    # x + r with scales (1, 1): 1.5 + 0.25 = 1.75; 1 + 2^-8 is a tie -> 1 (even);
    # -2 + 0.5 = -1.5; 3 - 3 = 0
    x, w = _identity_beam([[1.5, 1.0, -2.0, 3.0]])
    r = bits([[0.25, 2 ** -8, 0.5, -3.0]])
    hid, norm = oracle.beam_moe_finalize_norm_residual_norm(x, w, r)
    assert norm is None
    assert vals(hid[0]) == [1.75, 1.0, -1.5, 0.0]


def test_residual_scales_hand_example():
    # scales (2, 0.5): 2*1.5 + 0.5*1 = 3.5, 2*1 + 0.5*2 = 3, 2*-2 + 0.5*4 = -2,
    # 2*3 + 0.5*-8 = 2
    x, w = _identity_beam([[1.5, 1.0, -2.0, 3.0]])
    r = bits([[1.0, 2.0, 4.0, -8.0]])
    hid, _ = oracle.beam_moe_finalize_norm_residual_norm(x, w, r, scales=(2.0, 0.5))
    assert vals(hid[0]) == [3.5, 3.0, -2.0, 2.0]


def test_residual_sum_is_one_fp32_rounding():
    # reading: hidden = BF16(fma(s1, r, s0 * x)) in FP32.  x = 1, r = 2^-8 and
    # scales (1, 1 + 2^-23): s1 * r + x = 1 + 2^-8 + 2^-31 exactly, which FP32
    # rounds to 1 + 2^-8 (2^-31 is under half an FP32 ulp); that is a BF16 tie,
    # to even -> 1.0.  A float64 sum rounds to 1 + 2^-7.
    x, w = _identity_beam([[1.0] * 4])
    r = bits([[2.0 ** -8] * 4])
    hid, _ = oracle.beam_moe_finalize_norm_residual_norm(x, w, r, scales=(1.0, 1 + 2.0 ** -23))
    assert vals(hid[0]) == [1.0] * 4


def test_residual_next_norm_closed_form():
    # hidden = 0.5 + 0.5 = 1 everywhere; next norm with eps 3: 1/sqrt(1+3) = 0.5,
    # times next_weight [2, 1, -1, 0.5] -> [1, 0.5, -0.5, 0.25]
    x, w = _identity_beam([[0.5] * 4, [0.5] * 4])
    r = bits([[0.5] * 4, [0.5] * 4])
    hid, norm = oracle.beam_moe_finalize_norm_residual_norm(
        x, w, r, next_weight=bits([2.0, 1.0, -1.0, 0.5]), next_eps=3.0)
    assert np.all(hid == 0x3F80)
    assert vals(norm[0]) == vals(norm[1]) == [1.0, 0.5, -0.5, 0.25]


def test_residual_zero_reduces_to_beam_and_library_rmsnorm():
    # residual 0 and scales (1, 1): hidden is the Beam finalize output bit for
    # bit, and normalized is PyTorch's float64 rms_norm of it
    rng = np.random.default_rng(60)
    cap, K, H, T = 6, 4, 1024, 5
    x = f32_to_bf16_bits(rng.standard_normal((cap, K, H)).astype(np.float32))
    w = rng.random((cap, K)).astype(np.float32)
    pw = f32_to_bf16_bits((1 + 0.05 * rng.standard_normal(H)).astype(np.float32))
    nw = f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    r = np.zeros((T, H), dtype=np.uint16)
    hid, norm = oracle.beam_moe_finalize_norm_residual_norm(
        x, w, r, routed_scale=2.5, post_weight=pw, post_eps=1e-6, next_weight=nw, next_eps=1e-5)
    beam = oracle.beam_moe_finalize(x, w, T, routed_scale=2.5, post_weight=pw, post_eps=1e-6)
    assert np.array_equal(hid, beam)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(bf16_bits_to_f64(hid)), (H,),
                                       torch.from_numpy(bf16_bits_to_f64(nw)), 1e-5)
    compare_bf16(norm, ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16),
                 min_exact=0.999)


@pytest.mark.parametrize("seed", range(3))
def test_residual_matches_float64_brute_force(seed):
    rng = np.random.default_rng(70 + seed)
    cap, K, H = 7, [1, 5, 8][seed], [256, 768, 2048][seed]
    T = int(rng.integers(1, cap + 1))
    x = f32_to_bf16_bits(rng.standard_normal((cap, K, H)).astype(np.float32))
    w = rng.random((cap, K)).astype(np.float32)
    res = f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    nw = f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    s0, s1 = [(1.0, 1.0), (0.5, 2.0), (1.25, -0.75)][seed]
    hid, norm = oracle.beam_moe_finalize_norm_residual_norm(
        x, w, res, routed_scale=1.0, next_weight=nw, next_eps=1e-6, scales=(s0, s1))
    fin = _brute_beam(x, w, T, 1.0, None, None)
    h = s0 * bf16_bits_to_f64(fin) + s1 * bf16_bits_to_f64(res)
    compare_bf16(hid, f64_to_bf16_bits(h), min_exact=0.99)
    hv = bf16_bits_to_f64(hid)
    y = hv / np.sqrt((hv * hv).mean(axis=1, keepdims=True) + 1e-6) * bf16_bits_to_f64(nw)
    compare_bf16(norm, f64_to_bf16_bits(y), min_exact=0.99)
