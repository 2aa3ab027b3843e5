"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Every case runs the same seeded inputs through both and compares every
output element: |gpu - oracle| <= 2^-7 |oracle| + 1e-6 and at least 99% of
the elements bit-exact (the Beam path without normalisation must match bit
for bit).  Outputs carry canary rows past their end that must stay untouched.
"""
import functools

import numpy as np
import pytest

import oracle
import synth_inputs as si
from gpu_common import CANARY, dev_bf16, host_bits, oracle_beam, oracle_tp, run_beam, run_tp
from helpers import bf16_bits_to_f64, bf16_ulp, compare_bf16

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]

TP_VARIANTS = ("cluster", "token_cta", "bulk", "auto")
BEAM_VARIANTS = ("token_cta", "bulk", "auto")


# ---------------------------------------------------------------------------
# the five workloads

@functools.lru_cache(maxsize=None)
def c_small():
    return si.finalize_16_tokens()


@functools.lru_cache(maxsize=1)
def c_padded():
    return si.finalize_4096_tokens_padded(poison_padding=True)


@functools.lru_cache(maxsize=None)
def c_decode(T):
    return si.finalize_decode(T)


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_finalize_16_tokens(cuda_lib, variant):
    case = c_small()
    compare_bf16(run_tp(cuda_lib, case, variant), oracle_tp(case))


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_finalize_4096_tokens_padded_stride_bf16_weights(cuda_lib, variant):
    case = c_padded()
    got = run_tp(cuda_lib, case, variant)
    assert not np.isnan(bf16_bits_to_f64(got)).any(), "padding (NaN) leaked into the output"
    compare_bf16(got, oracle_tp(case))


@pytest.mark.parametrize("T", si.DECODE_TOKENS)
@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_finalize_decode_sizes(cuda_lib, T, variant):
    case = c_decode(T)
    compare_bf16(run_tp(cuda_lib, case, variant), oracle_tp(case))


def test_automatic_choice_by_waves(cuda_lib):
    # between 9 and 1023 tokens the register kernel (2 CTAs per SM) runs unless
    # the bulk-staged kernel (3 CTAs per SM) needs fewer waves of the device's SMs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    def waves(t, per_sm):
        return -(-t // (per_sm * sms))
    for T in (1, 8, 9, 100, 2 * sms, 2 * sms + 1, 3 * sms, 3 * sms + 1, 4 * sms, 5 * sms,
              1023, 1024, 5000):
        if T <= 8:
            want = "cluster"
        elif T >= 1024:
            want = "bulk"
        else:
            want = "bulk" if waves(T, 3) < waves(T, 2) else "token_cta"
        assert cuda_lib.select_finalize_variant(T) == want, T
    for T in (2 * sms + 1, 5 * sms):   # one token count of each choice, against the oracle
        case = si.tp_case(f"waves_{T}", T, indexed_rows=T * 8 + 9, invalid_frac=0.02,
                          weights_dtype="fp32", seed=T)
        compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


@functools.lru_cache(maxsize=1)
def c_roofline():
    return si.finalize_32768_tokens(weight_before_norm=False)


@pytest.mark.parametrize("before", [False, True])
def test_finalize_32768_tokens_full_size(cuda_lib, before):
    # the bandwidth workload in the launch configuration the benchmark times
    # (automatic choice), every output element against the oracle
    case = c_roofline()
    assert cuda_lib.select_finalize_variant(case.num_tokens) == "bulk"
    got = run_tp(cuda_lib, case, "auto", before=before)
    stats = compare_bf16(got, oracle_tp(case, before=before))
    assert stats["n"] == 32768 * 4096


@functools.lru_cache(maxsize=1)
def c_beam():
    return si.beam_8000_live(poison_dead_rows=True)


@pytest.mark.parametrize("variant", BEAM_VARIANTS)
def test_beam_8000_live(cuda_lib, variant):
    case = c_beam()
    got = run_beam(cuda_lib, case, variant)
    assert not np.isnan(bf16_bits_to_f64(got)).any(), "dead rows (NaN) leaked into the output"
    compare_bf16(got, oracle_beam(case))


# ---------------------------------------------------------------------------
# edge cases: finalize + RMSNorm

def small_case(T, *, stride=4096, wdt="fp32", seed=1, before=False, eps=1e-6):
    return si.tp_case(f"edge_T{T}", T, indexed_rows=T * 8 + 3, row_stride=stride,
                      invalid_frac=0.05, weights_dtype=wdt, seed=seed, weight_before_norm=before,
                      eps=eps)


@pytest.mark.parametrize("T", [2, 37, 65, 300, 1023, 1024, 1500])
@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_ragged_token_counts(cuda_lib, T, variant):
    case = small_case(T, seed=T, before=bool(T % 2), wdt="bf16" if T % 3 == 0 else "fp32")
    compare_bf16(run_tp(cuda_lib, case, variant), oracle_tp(case))


# Token counts around the multi-token CTAs of the staged hidden-4096 kernel,
# used from five waves of resident CTAs up (152 SMs x 3 CTAs = 456 on GB300:
# 2280 tokens is the first multi-token launch; 2600 drops a partial wave of
# multi-token CTAs, 3284 keeps one).  Rows of stride 4160 with NaN padding
# columns and padding rows; 5% invalid slots, so a row's mbarrier skips
# tokens and its phase must still be tracked.
@pytest.mark.parametrize("T", [2279, 2280, 2281, 2600, 3284, 4567, 9001])
@pytest.mark.parametrize("wdt", ["fp32", "bf16", "packed"])
def test_multi_token_ctas(cuda_lib, T, wdt):
    case = si.tp_case(f"multi{T}{wdt}", T, indexed_rows=T * 8, padding_rows=64, row_stride=4160,
                      invalid_frac=0.05, weights_dtype=wdt, weight_before_norm=T % 2 == 1,
                      seed=T, poison_padding=True)
    assert cuda_lib.select_finalize_variant(T) == "bulk"
    compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


def test_kernel_name_reports_the_multi_token_kernel(cuda_lib):
    # five waves of the staged kernel's resident CTAs (three per SM) and more
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    first = 5 * 3 * sms
    assert cuda_lib.finalize_kernel_name(first - 1) == "tp_token_bulk_kernel"
    assert cuda_lib.finalize_kernel_name(first) == "tp_token_bulk_multi_kernel"
    assert cuda_lib.finalize_kernel_name(32768) == "tp_token_bulk_multi_kernel"
    assert cuda_lib.finalize_kernel_name(32768, variant="token_cta") == "tp_token_cta_kernel"
    # the residual op takes three tokens per CTA from five waves (two CTAs per
    # SM at hidden 7168); plain Beam keeps one token per CTA
    first = 5 * 2 * sms
    assert cuda_lib.beam_kernel_name(first - 1, 8, 7168, residual=True) == "beam_token_bulk_kernel"
    assert cuda_lib.beam_kernel_name(first, 8, 7168, residual=True) == \
        "beam_token_bulk_multi_kernel"
    assert cuda_lib.beam_kernel_name(8000, 8, 7168, residual=True) == \
        "beam_token_bulk_multi_kernel"
    assert cuda_lib.beam_kernel_name(8000, 8, 7168) == "beam_token_bulk_kernel"
    assert cuda_lib.beam_kernel_name(8000, 16, 7168, residual=True) == "beam_token_bulk_kernel"
    assert cuda_lib.beam_kernel_name(8000, 8, 8192, residual=True) == "beam_token_bulk_kernel"
    assert cuda_lib.beam_kernel_name(8000, 8, 3072, residual=True) == "beam_token_bulk_kernel"


def test_multi_token_ctas_half_the_slots_invalid(cuda_lib):
    # many slots skipped in a row: the per-row phases diverge across tokens
    T = 3500
    case = si.tp_case("multi_sparse", T, indexed_rows=T * 8, invalid_frac=0.5,
                      weights_dtype="fp32", seed=7)
    compare_bf16(run_tp(cuda_lib, case, "bulk"), oracle_tp(case))


def test_multi_token_ctas_with_and_without_programmatic_launch(cuda_lib):
    case = small_case(3000, seed=44)
    assert cuda_lib.finalize_kernel_name(3000) == "tp_token_bulk_multi_kernel"
    try:
        cuda_lib.set_programmatic_launch(False)
        off = run_tp(cuda_lib, case, "bulk")
    finally:
        cuda_lib.set_programmatic_launch(True)
    on = run_tp(cuda_lib, case, "bulk")
    assert np.array_equal(off, on)
    compare_bf16(on, oracle_tp(case))


def test_multi_token_ctas_read_the_previous_calls_output(cuda_lib):
    # a Beam call writes the 2400 rows that a 3000-token finalize (three tokens
    # per CTA) gathers right after it on the same stream, with programmatic launch
    T1, K1, T2 = 2400, 2, 3000
    beam = si.beam_case("chain_multi", T1, K1, 4096, T1, routed_scale=1.5, post_weight=False,
                        post_eps=None, seed=45)
    x, w1 = dev_bf16(beam.expert_outputs), torch.from_numpy(beam.weights).cuda()
    mid = torch.empty((T1, 4096), dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(46)
    idx2 = rng.integers(-1, T1, size=(T2, 8)).astype(np.int32)
    w2 = rng.random((T2, 8)).astype(np.float32)
    nw = f32_bits(rng.standard_normal(4096) * 0.1)
    out = torch.empty((T2, 4096), dtype=torch.bfloat16, device="cuda")
    idx2_d, w2_d, nw_d = torch.from_numpy(idx2).cuda(), torch.from_numpy(w2).cuda(), dev_bf16(nw)
    for _ in range(3):
        mid.fill_(float("nan"))
        torch.cuda.synchronize()
        cuda_lib.beam_moe_finalize(x, w1, mid, beam.routed_scale)
        cuda_lib.moe_finalize_rmsnorm(mid, w2_d, idx2_d, nw_d, out, eps=1e-6, gain_center=1.0,
                                      weight_before_norm=False)
        torch.cuda.synchronize()
        assert not np.isnan(bf16_bits_to_f64(host_bits(out))).any()
    ref1 = oracle_beam(beam)
    ref2 = oracle.moe_finalize_rmsnorm(ref1, w2, idx2, nw, eps=1e-6, gain_center=1.0,
                                       weight_before_norm=False)
    compare_bf16(host_bits(out), ref2)


def test_multi_token_ctas_in_a_graph_and_on_two_streams(cuda_lib):
    cases = [small_case(2600, seed=47), small_case(2600, seed=48)]
    c0 = cases[0]
    g, w, idx, nw = (dev_bf16(c0.gemm2), torch.from_numpy(c0.weights).cuda(),
                     torch.from_numpy(c0.idx).cuda(), dev_bf16(c0.norm_weight))
    out = torch.empty((2600, 4096), dtype=torch.bfloat16, device="cuda")

    def call():
        cuda_lib.moe_finalize_rmsnorm(g, w, idx, nw, out, eps=c0.eps, gain_center=c0.gain_center,
                                      weight_before_norm=c0.weight_before_norm)
    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st), torch.cuda.graph(graph, stream=st):
        call()
    torch.cuda.synchronize()
    for c in cases:
        g.copy_(dev_bf16(c.gemm2))
        w.copy_(torch.from_numpy(c.weights).cuda())
        idx.copy_(torch.from_numpy(c.idx).cuda())
        nw.copy_(dev_bf16(c.norm_weight))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        compare_bf16(host_bits(out), oracle_tp(c))
    # two launches in flight at once on two streams, different buffers
    c1 = cases[1]
    g1, w1, i1 = dev_bf16(c1.gemm2), torch.from_numpy(c1.weights).cuda(), torch.from_numpy(c1.idx).cuda()
    nw1 = dev_bf16(c1.norm_weight)
    out1 = torch.empty_like(out)
    g.copy_(dev_bf16(c0.gemm2))
    w.copy_(torch.from_numpy(c0.weights).cuda())
    idx.copy_(torch.from_numpy(c0.idx).cuda())
    nw.copy_(dev_bf16(c0.norm_weight))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        cuda_lib.moe_finalize_rmsnorm(g, w, idx, nw, out, eps=c0.eps, gain_center=c0.gain_center,
                                      weight_before_norm=c0.weight_before_norm, stream=s1)
        cuda_lib.moe_finalize_rmsnorm(g1, w1, i1, nw1, out1, eps=c1.eps, gain_center=c1.gain_center,
                                      weight_before_norm=c1.weight_before_norm, stream=s2)
    torch.cuda.synchronize()
    compare_bf16(host_bits(out), oracle_tp(c0))
    compare_bf16(host_bits(out1), oracle_tp(c1))


def _tie_case(rows, w, nw, *, eps, gc, before, T=3):
    # T tokens, each gathering the same rows in its first slots; the other of its
    # 8 slots are invalid (-1), so every hidden-4096 kernel applies
    n = rows.shape[0]
    idx = np.full((T, 8), -1, dtype=np.int32)
    idx[:, :n] = np.arange(n, dtype=np.int32)
    wt = np.zeros((T, 8), dtype=np.float32)
    wt[:, :n] = w
    return si.TpCase("tie", f32_bits(rows), wt, idx, f32_bits(nw), 4096, eps, gc, before)


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_fp32_rounding_ties_match_the_oracle(cuda_lib, variant):
    # inputs on which FP32 and float64 arithmetic round to different BF16 values
    # (derivations in the oracle pins): one rounding per slot of the reduction,
    # and the FP32 add of the gain center.  Every kernel must give the oracle's
    # bits exactly: 1.0 in every element.
    one_plus = np.float32(1 + 2.0 ** -7)
    fma_rows = np.stack([np.full(4096, -one_plus), np.full(4096, one_plus)]).astype(np.float32)
    fma_w = np.full(2, 1 + 2.0 ** -17, dtype=np.float32)
    for before in (False, True):
        case = _tie_case(fma_rows, fma_w, np.ones(4096), eps=2.0 ** -100, gc=0.0, before=before)
        got, ref = run_tp(cuda_lib, case, variant), oracle_tp(case)
        assert np.all(ref == 0x3F80) and np.array_equal(got, ref)
    case = _tie_case(np.ones((1, 4096), dtype=np.float32), np.ones(1, dtype=np.float32),
                     np.full(4096, 2.0 ** -30), eps=0.0, gc=1 + 2.0 ** -8, before=False)
    got, ref = run_tp(cuda_lib, case, variant), oracle_tp(case)
    assert np.all(ref == 0x3F80) and np.array_equal(got, ref)


@pytest.mark.parametrize("variant", BEAM_VARIANTS)
def test_beam_fp32_scale_tie_matches_the_oracle(cuda_lib, variant):
    # the FP32 product of the BF16 sum and the scale lands exactly on a BF16 tie
    # (1 + 2^-8 -> 1.0); a float64 product would give 1 + 2^-7
    x = f32_bits(np.full((4, 1, 256), 1 + 2.0 ** -7, dtype=np.float32))
    case = si.BeamCase("tie", x, np.ones((4, 1), dtype=np.float32), 4,
                       16712189 * 2.0 ** -24, None, None, meta={})
    got, ref = run_beam(cuda_lib, case, variant), oracle_beam(case)
    assert np.all(ref == 0x3F80) and np.array_equal(got, ref)


def test_residual_fp32_sum_tie_matches_the_oracle(cuda_lib):
    # hidden = BF16(fma(1 + 2^-23, 2^-8, 1)) = BF16(1 + 2^-8) = 1.0 in FP32
    case = si.BeamCase("tie", f32_bits(np.ones((4, 1, 256), dtype=np.float32)),
                       np.ones((4, 1), dtype=np.float32), 4, 1.0, None, None, meta={})
    res = f32_bits(np.full((4, 256), 2.0 ** -8, dtype=np.float32))
    h, _, _ = run_residual(cuda_lib, case, res, post=False, nxt=None, scales=(1.0, 1 + 2.0 ** -23))
    rh, _ = oracle.beam_moe_finalize_norm_residual_norm(case.expert_outputs, case.weights, res,
                                                        scales=(1.0, 1 + 2.0 ** -23))
    assert np.all(rh == 0x3F80) and np.array_equal(h, rh)


def test_fewer_tokens_than_sms(cuda_lib):
    case = small_case(5, seed=5)
    for v in ("bulk", "token_cta", "cluster"):
        compare_bf16(run_tp(cuda_lib, case, v), oracle_tp(case))


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_zero_tokens_is_a_no_op(cuda_lib, variant):
    case = small_case(3)
    g = dev_bf16(case.gemm2)
    out = torch.full((2, 4096), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    cuda_lib.moe_finalize_rmsnorm(g, torch.empty((0, 8), device="cuda"),
                                  torch.empty((0, 8), dtype=torch.int32, device="cuda"),
                                  dev_bf16(case.norm_weight), out[:0], eps=1e-6, gain_center=1.0,
                                  weight_before_norm=False, variant=variant)
    torch.cuda.synchronize()
    assert np.all(host_bits(out) == CANARY)


def _special_index_case(before):
    # tokens whose slots are all invalid, the boundary indices rows-1 / rows,
    # INT32_MIN / INT32_MAX, duplicated indices and NaN weights on invalid slots
    case = small_case(24, seed=7, before=before)
    R = case.gemm2.shape[0]
    idx = case.idx.copy()
    w = case.weights.copy()
    idx[0, :] = [-1, R, np.iinfo(np.int32).min, np.iinfo(np.int32).max, -7, R + 5, -1, R]
    w[0, :] = np.nan
    idx[1, :] = [R - 1, R, R - 1, -1, 0, 0, R + 1, 3]
    w[1, 1] = w[1, 3] = w[1, 6] = np.nan
    idx[2, :] = 5                                     # one row eight times
    idx[3, :] = -1
    idx[3, 7] = 11                                    # only the last slot valid
    idx[4, :] = -1
    idx[4, 0] = 12                                    # only the first slot valid
    case.idx, case.weights = np.ascontiguousarray(idx), np.ascontiguousarray(w)
    return case


@pytest.mark.parametrize("before", [False, True])
@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_special_indices(cuda_lib, variant, before):
    case = _special_index_case(before)
    got = run_tp(cuda_lib, case, variant)
    assert np.all(bf16_bits_to_f64(got[0]) == 0.0)   # all-invalid token -> exact zeros
    compare_bf16(got, oracle_tp(case))


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_all_invalid_with_zero_eps_gives_nan(cuda_lib, variant):
    # the degenerate case of the formula: 0 * 1/sqrt(0); both sides give NaN
    case = small_case(4, seed=8, eps=0.0)
    case.idx[:] = -1
    got = run_tp(cuda_lib, case, variant)
    assert np.isnan(bf16_bits_to_f64(got)).all()
    compare_bf16(got, oracle_tp(case))


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_no_rows_at_all(cuda_lib, variant):
    # gemm2 with zero rows: every index is out of range
    case = small_case(3, seed=9)
    case.gemm2 = np.zeros((0, 4096), dtype=np.uint16)
    got = run_tp(cuda_lib, case, variant)
    assert np.all(bf16_bits_to_f64(got) == 0.0)


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_wide_row_stride(cuda_lib, variant):
    case = si.tp_case("stride8192", 40, indexed_rows=400, padding_rows=9, row_stride=8192,
                      invalid_frac=0.1, weights_dtype="fp32", seed=10, poison_padding=True)
    got = run_tp(cuda_lib, case, variant)
    compare_bf16(got, oracle_tp(case))


@pytest.mark.parametrize("variant", ("token_cta", "bulk"))
def test_extreme_values(cuda_lib, variant):
    # large magnitudes (sigma 1e15) and tiny ones (sigma 1e-15): the FP32
    # reduction and the FP32 sum of squares stay finite and normal, and match
    # (beyond |acc| ~ 2^57 the FP32 sum of squares of 4096 values overflows)
    for sigma, seed in ((1e15, 11), (1e-15, 12)):
        case = si.tp_case("extreme", 64, indexed_rows=512, sigma=sigma, invalid_frac=0.02,
                          weights_dtype="fp32", seed=seed, eps=0.0)
        compare_bf16(run_tp(cuda_lib, case, variant), oracle_tp(case))


def test_non_default_stream(cuda_lib):
    case = small_case(50, seed=13)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = run_tp(cuda_lib, case, "auto", stream=s)
    compare_bf16(got, oracle_tp(case))


# ---------------------------------------------------------------------------
# other sizes (hidden 256..8192, top_k 1..32) and packed routing words

@pytest.mark.parametrize("H,K", [(256, 1), (256, 32), (7168, 8), (8192, 32), (4096, 4),
                                 (2048, 16), (7936, 3), (1536, 5), (4096, 8), (512, 32),
                                 (768, 7), (1024, 8), (1024, 32), (1280, 2), (1536, 32),
                                 (1792, 20)])
@pytest.mark.parametrize("wdt", ["fp32", "bf16", "packed"])
def test_generic_sizes(cuda_lib, H, K, wdt):
    T = 37
    case = si.tp_case(f"generic_{H}_{K}", T, hidden=H, top_k=K, indexed_rows=T * K + 5,
                      padding_rows=3, row_stride=H + 16, invalid_frac=0.1, weights_dtype=wdt,
                      seed=H + K, weight_before_norm=bool(K % 2), poison_padding=True)
    case.idx[0, :] = -1                                  # one token with no valid slot
    variants = ("auto", "bulk") if (H, K) != (4096, 8) else TP_VARIANTS
    for v in variants:
        compare_bf16(run_tp(cuda_lib, case, v), oracle_tp(case))


# Other sizes at five waves and more with a token in one staged piece run
# several tokens per CTA (tp_generic_bulk_multi_kernel): hidden 7168 x 8 from
# 1520 tokens on GB300 (two CTAs per SM), 3072 x 8 and 2304 x 8 (one chunk per
# thread), 1280 x 10 (small rows, ten per piece); 5% invalid slots.
# With small tokens at hidden 2048..7168 (top_k 1..3) the buffer holds two
# tokens: 8000 x 7168 x 1, 7000 x 7168 x 2, 6000 x 6144 x 3, 16000 x 4096 x 1,
# 16000 x 2048 x 2.
@pytest.mark.parametrize("T,H,K", [(1600, 7168, 8), (4000, 3072, 8), (5000, 2304, 8),
                                   (9000, 1280, 10), (8000, 7168, 1), (7000, 7168, 2),
                                   (6000, 6144, 3), (16000, 4096, 1), (16000, 2048, 2)])
@pytest.mark.parametrize("wdt", ["fp32", "bf16", "packed"])
def test_generic_multi_token_ctas(cuda_lib, T, H, K, wdt):
    case = si.tp_case(f"gmulti{T}{wdt}", T, hidden=H, top_k=K, indexed_rows=T * K + 5,
                      padding_rows=3, row_stride=H + 8, invalid_frac=0.05, weights_dtype=wdt,
                      weight_before_norm=T % 2 == 0, seed=T + H, poison_padding=True)
    assert cuda_lib.finalize_kernel_name(T, H, K) == "tp_generic_bulk_multi_kernel"
    compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


# Hidden 256..1024 at five waves of resident warps and more, a token in one
# slice piece (top_k <= 8, or 16 at hidden 256): three tokens per warp
# (tp_warp_bulk_multi_kernel); the last CTA's second warp may have no token.
@pytest.mark.parametrize("T,H,K", [(30001, 256, 8), (30000, 256, 16), (25001, 512, 8),
                                   (15000, 768, 8), (13000, 1024, 6)])
@pytest.mark.parametrize("wdt", ["fp32", "bf16", "packed"])
def test_warp_multi_token(cuda_lib, T, H, K, wdt):
    case = si.tp_case(f"wmulti{T}{H}{wdt}", T, hidden=H, top_k=K, indexed_rows=T * K + 5,
                      padding_rows=3, row_stride=H + 8, invalid_frac=0.05, weights_dtype=wdt,
                      weight_before_norm=T % 2 == 1, seed=T + H, poison_padding=True)
    assert cuda_lib.finalize_kernel_name(T, H, K) == "tp_warp_bulk_multi_kernel"
    compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


def test_warp_multi_token_sparse_and_empty_tokens(cuda_lib):
    # 60% invalid slots: some tokens have no valid row at all (the warp's
    # barrier then skips a phase) -- their output is exactly zero
    T, H, K = 30000, 512, 4
    case = si.tp_case("wmulti_sparse", T, hidden=H, top_k=K, indexed_rows=T * K,
                      invalid_frac=0.6, weights_dtype="fp32", seed=10)
    assert (np.all((case.idx < 0) | (case.idx >= case.gemm2.shape[0]), axis=1)).sum() > 100
    compare_bf16(run_tp(cuda_lib, case, "bulk"), oracle_tp(case))


def test_generic_multi_token_ctas_half_the_slots_invalid(cuda_lib):
    T, H, K = 2000, 7168, 8
    case = si.tp_case("gmulti_sparse", T, hidden=H, top_k=K, indexed_rows=T * K,
                      invalid_frac=0.5, weights_dtype="fp32", seed=9)
    compare_bf16(run_tp(cuda_lib, case, "bulk"), oracle_tp(case))


def test_generic_two_token_slots_with_empty_tokens(cuda_lib):
    # two token slots at 7168 x 2 with half the slots invalid: about a quarter
    # of the tokens have no valid row (their slot's barriers do not move on)
    # and give exactly zero
    T, H, K = 8000, 7168, 2
    case = si.tp_case("gtwo_sparse", T, hidden=H, top_k=K, indexed_rows=T * K,
                      invalid_frac=0.5, weights_dtype="bf16", weight_before_norm=True, seed=12)
    empty = np.all((case.idx < 0) | (case.idx >= case.gemm2.shape[0]), axis=1)
    assert empty.sum() > 1000
    assert cuda_lib.finalize_kernel_name(T, H, K) == "tp_generic_bulk_multi_kernel"
    got = run_tp(cuda_lib, case, "auto")
    compare_bf16(got, oracle_tp(case))
    assert np.all(got[empty] == 0)


def test_two_token_slot_kernels_with_and_without_programmatic_launch(cuda_lib):
    # the generic finalize and Beam with two token slots per CTA give the same
    # bits with programmatic launch off and on
    tcase = si.tp_case("gtwo_pdl", 8000, hidden=7168, top_k=2, indexed_rows=16000,
                       invalid_frac=0.05, weights_dtype="fp32", seed=14)
    bcase = si.beam_case("btwo_pdl", 3100, 2, 7168, 3100, routed_scale=2.5, seed=15)
    assert cuda_lib.finalize_kernel_name(8000, 7168, 2) == "tp_generic_bulk_multi_kernel"
    assert cuda_lib.beam_kernel_name(3100, 2, 7168) == "beam_token_bulk_multi_kernel"
    got = {}
    try:
        for pdl in (False, True):
            cuda_lib.set_programmatic_launch(pdl)
            got[pdl] = (run_tp(cuda_lib, tcase, "auto"), run_beam(cuda_lib, bcase, "auto"))
    finally:
        cuda_lib.set_programmatic_launch(True)
    assert all(np.array_equal(a, b) for a, b in zip(got[False], got[True]))
    compare_bf16(got[True][0], oracle_tp(tcase))
    compare_bf16(got[True][1], oracle_beam(bcase))


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_packed_routing_words_specialised(cuda_lib, variant):
    case = si.tp_case("packed", 300, indexed_rows=2500, invalid_frac=0.03, weights_dtype="packed",
                      seed=31)
    assert case.weights.dtype == np.int32 and (case.weights < 0).sum() == 0
    compare_bf16(run_tp(cuda_lib, case, variant), oracle_tp(case))
    # high expert ids (negative words) change nothing
    case.weights = (case.weights.view(np.uint32) | np.uint32(0xF0000000)).view(np.int32)
    compare_bf16(run_tp(cuda_lib, case, variant), oracle_tp(case))


def test_other_sizes_reject_register_and_cluster_kernels(cuda_lib):
    case = si.tp_case("generic_reject", 4, hidden=2048, top_k=8, seed=32)
    for v in ("token_cta", "cluster"):
        with pytest.raises(cuda_lib.MoeFinalizeError) as e:
            run_tp(cuda_lib, case, v)
        assert e.value.status == 8


def test_unsupported_hidden_raises(cuda_lib):
    g = torch.zeros(16, 2000, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.MoeFinalizeError) as e:
        cuda_lib.moe_finalize_rmsnorm(g, torch.zeros(2, 8, device="cuda"),
                                      torch.zeros(2, 8, dtype=torch.int32, device="cuda"),
                                      torch.zeros(2000, dtype=torch.bfloat16, device="cuda"),
                                      torch.zeros(2, 2000, dtype=torch.bfloat16, device="cuda"),
                                      eps=1e-6, gain_center=1.0, weight_before_norm=False)
    assert e.value.status == 5


# ---------------------------------------------------------------------------
# edge cases: Beam

@pytest.mark.parametrize("K,H", [(1, 256), (32, 256), (8, 8192), (3, 7936), (5, 1536), (32, 8192),
                                 (2, 2560), (8, 4096), (32, 1024), (7, 768), (8, 512),
                                 # several pieces per token: per-row barriers, then small rows
                                 (16, 2048), (24, 3072), (32, 1536)])
@pytest.mark.parametrize("variant", BEAM_VARIANTS)
def test_beam_shapes(cuda_lib, K, H, variant):
    case = si.beam_case(f"beam_{K}_{H}", 40, K, H, 37, routed_scale=2.5, seed=K * 1000 + H,
                        poison_dead_rows=True)
    compare_bf16(run_beam(cuda_lib, case, variant), oracle_beam(case))


# Beam launches of many waves with the token in one staged piece, at hidden
# 2048-7168 with two chunks per thread or one (2304), dead rows poisoned; the
# several-tokens kernel with two token slots (top_k 1..6 at hidden 7168: CTAs
# of two tokens only, or three-slot-deep groups first; small tokens at 4096..5632
# in the build for three CTAs per SM) or one (5120 x 8).
ONE, MULTI = "beam_token_bulk_kernel", "beam_token_bulk_multi_kernel"


@pytest.mark.parametrize("T,H,K,kernel", [
    (1600, 7168, 8, ONE), (6000, 2048, 8, ONE), (4000, 4096, 4, ONE), (3000, 2304, 8, ONE),
    (2600, 7168, 1, MULTI), (3100, 7168, 1, MULTI), (2500, 7168, 4, MULTI),
    (5000, 7168, 2, MULTI), (3000, 7168, 3, MULTI), (6000, 5120, 8, MULTI),
    (3000, 5632, 8, MULTI), (4000, 6656, 6, MULTI), (1000, 7168, 2, ONE),
    # the build for three CTAs per SM (under 80 KB in flight with one token per CTA)
    (16000, 4096, 1, MULTI), (8000, 4608, 1, MULTI), (8000, 5632, 2, MULTI),
    (8000, 4096, 2, ONE), (6000, 6144, 3, ONE)])
def test_beam_many_waves(cuda_lib, T, H, K, kernel):
    case = si.beam_case(f"bwaves{T}", T + 7, K, H, T, routed_scale=2.5, seed=T + H + K,
                        poison_dead_rows=True)
    assert cuda_lib.beam_kernel_name(T, K, H) == kernel
    compare_bf16(run_beam(cuda_lib, case, "auto"), oracle_beam(case))


def test_beam_multi_token_ctas_without_norm_and_unweighted(cuda_lib):
    # the several-tokens kernel with the post-norm off (bit-exact) and an
    # unweighted post-norm
    T, H, K = 3100, 7168, 2
    assert cuda_lib.beam_kernel_name(T, K, H) == MULTI
    case = si.beam_case("bmulti_nonorm", T, K, H, T, routed_scale=1.5, post_weight=False,
                        post_eps=None, seed=77)
    assert np.array_equal(run_beam(cuda_lib, case, "auto"), oracle_beam(case))
    case = si.beam_case("bmulti_unweighted", T, K, H, T, routed_scale=1.5, post_weight=False,
                        post_eps=1e-6, seed=78)
    compare_bf16(run_beam(cuda_lib, case, "auto"), oracle_beam(case))


@pytest.mark.parametrize("variant", BEAM_VARIANTS)
def test_beam_without_norm_is_bit_exact(cuda_lib, variant):
    case = si.beam_case("beam_nonorm", 300, 8, 7168, 290, routed_scale=2.5, post_weight=False,
                        post_eps=None, seed=21, poison_dead_rows=True)
    got = run_beam(cuda_lib, case, variant)
    assert np.array_equal(got, oracle_beam(case))


@pytest.mark.parametrize("variant", BEAM_VARIANTS)
def test_beam_unweighted_norm(cuda_lib, variant):
    case = si.beam_case("beam_unweighted", 200, 4, 2048, 200, routed_scale=0.75,
                        post_weight=False, post_eps=1e-5, seed=22)
    compare_bf16(run_beam(cuda_lib, case, variant), oracle_beam(case))


@pytest.mark.parametrize("live", [0, 1, 151, 152, 153, 1000])
def test_beam_live_counts(cuda_lib, live):
    case = si.beam_case("beam_live", 1000, 8, 1024, live, routed_scale=2.5, seed=23,
                        poison_dead_rows=True)
    got = run_beam(cuda_lib, case, "auto")
    if live:
        compare_bf16(got, oracle_beam(case))


def test_beam_extra_weight_rows(cuda_lib):
    case = si.beam_case("beam_wrows", 64, 8, 512, 10, routed_scale=1.0, seed=24)
    compare_bf16(run_beam(cuda_lib, case, "bulk"), oracle_beam(case))


def test_beam_matches_tp_reduction_on_identity_map(cuda_lib):
    # token-major rows with the identity route map: Beam without norm and scale
    # 1 rounds the same FP32 sums that the tp path normalises; check the GPU
    # Beam output against the Beam oracle and the tp GPU output against the
    # tp oracle on the very same rows
    cap, K, H = 64, 8, 4096
    case = si.beam_case("beam_identity", cap, K, H, cap, routed_scale=1.0, post_weight=False,
                        post_eps=None, seed=25)
    assert np.array_equal(run_beam(cuda_lib, case, "bulk"), oracle_beam(case))
    tp = si.TpCase("identity", np.ascontiguousarray(case.expert_outputs.reshape(cap * K, H)),
                   case.weights, np.arange(cap * K, dtype=np.int32).reshape(cap, K),
                   np.zeros(H, dtype=np.uint16), H, 1e-6, 1.0, False)
    compare_bf16(run_tp(cuda_lib, tp, "bulk"), oracle_tp(tp))


# ---------------------------------------------------------------------------
# failure detection (a bounded wait that gives up; no fault, no hang)

def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    assert cuda_lib.device_status(clear=True) == 0
    cuda_lib.selftest_wait_timeout(20_000_000)        # 20 ms
    assert cuda_lib.device_status(clear=False) == 7   # MF_ERR_DEVICE_TIMEOUT
    assert cuda_lib.device_status(clear=True) == 7
    assert cuda_lib.device_status(clear=True) == 0
    case = small_case(8, seed=30)
    compare_bf16(run_tp(cuda_lib, case, "bulk"), oracle_tp(case))


# ---------------------------------------------------------------------------
# programmatic dependent launch

@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_programmatic_launch_on_and_off_agree(cuda_lib, variant):
    case = small_case(300, seed=40)
    try:
        cuda_lib.set_programmatic_launch(False)
        off = run_tp(cuda_lib, case, variant)
    finally:
        cuda_lib.set_programmatic_launch(True)
    on = run_tp(cuda_lib, case, variant)
    assert np.array_equal(off, on)
    compare_bf16(on, oracle_tp(case))


@pytest.mark.parametrize("variant", ("cluster", "token_cta", "bulk"))
def test_dependent_calls_see_each_others_output(cuda_lib, variant):
    # call 1 (Beam finalize without norm, bit-exact with its oracle) writes the
    # rows that call 2 (finalize + RMSNorm) gathers; both are launched back to
    # back on one stream with programmatic dependent launch, so call 2 must
    # wait for call 1.  Expected: the two oracles chained.
    assert cuda_lib.programmatic_launch()
    T1, K1 = 64, 4
    beam = si.beam_case("chain", T1, K1, 4096, T1, routed_scale=1.5, post_weight=False,
                        post_eps=None, seed=41)
    x = dev_bf16(beam.expert_outputs)
    w1 = torch.from_numpy(beam.weights).cuda()
    mid = torch.empty((T1, 4096), dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(42)
    T2 = 48
    idx2 = rng.integers(-1, T1, size=(T2, 8)).astype(np.int32)
    w2 = rng.random((T2, 8)).astype(np.float32)
    nw = f32_bits(rng.standard_normal(4096) * 0.1)
    out = torch.empty((T2, 4096), dtype=torch.bfloat16, device="cuda")
    idx2_d, w2_d, nw_d = torch.from_numpy(idx2).cuda(), torch.from_numpy(w2).cuda(), dev_bf16(nw)
    for _ in range(3):
        mid.fill_(float("nan"))
        torch.cuda.synchronize()
        cuda_lib.beam_moe_finalize(x, w1, mid, beam.routed_scale)
        cuda_lib.moe_finalize_rmsnorm(mid, w2_d, idx2_d, nw_d, out, eps=1e-6, gain_center=1.0,
                                      weight_before_norm=True, variant=variant)
        torch.cuda.synchronize()
        got = host_bits(out)
        assert not np.isnan(bf16_bits_to_f64(got)).any(), "call 2 read call 1's output too early"
    ref1 = oracle_beam(beam)
    assert np.array_equal(host_bits(mid), ref1)
    ref2 = oracle.moe_finalize_rmsnorm(ref1, w2, idx2, nw, eps=1e-6, gain_center=1.0,
                                       weight_before_norm=True)
    compare_bf16(got, ref2)


def f32_bits(a):
    u = np.asarray(a, dtype=np.float32).view(np.uint32).copy()
    u += ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# CUDA graphs: calls captured once (after a first call outside capture) and
# replayed with new inputs written into the captured buffers

@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_graph_replay_with_new_inputs(cuda_lib, variant):
    cases = [small_case(200, seed=50), small_case(200, seed=51)]
    a = cases[0]
    g = dev_bf16(a.gemm2)
    w = torch.from_numpy(a.weights).cuda()
    idx = torch.from_numpy(a.idx).cuda()
    nw = dev_bf16(a.norm_weight)
    out = torch.empty((200, 4096), dtype=torch.bfloat16, device="cuda")

    def call():
        cuda_lib.moe_finalize_rmsnorm(g, w, idx, nw, out, eps=a.eps, gain_center=a.gain_center,
                                      weight_before_norm=a.weight_before_norm, variant=variant)

    call()                                   # first call outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s), torch.cuda.graph(graph, stream=s):
        call()
    torch.cuda.synchronize()
    for c in cases:
        g.copy_(dev_bf16(c.gemm2))
        w.copy_(torch.from_numpy(c.weights).cuda())
        idx.copy_(torch.from_numpy(c.idx).cuda())
        nw.copy_(dev_bf16(c.norm_weight))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        compare_bf16(host_bits(out), oracle_tp(c))



# ---------------------------------------------------------------------------
# beam_moe_finalize_norm_residual_norm (residual step: a reading of the pages)

def residual_bounds(case, h_ref, n_ref, *, post, scales, next_eps, next_weight):
    """Widened bounds for the residual op.  With the Beam post-norm on, the
    finalized value f = BF16(v * rs * post_weight) comes from an FP32 norm on
    the GPU and a float64 one in the oracle, so f may land one BF16 ulp apart
    (about 1e-5 of elements); hidden = BF16(s0 f + s1 r) then differs by up to
    |s0| ulp(f) on top of its own rounding, which can be many ulps of hidden
    where s0 f and s1 r cancel.  The next norm scales that by rn * next_weight.
    Each output's own BF16 round then adds up to half an ulp of the GPU's value
    (at most 2^-8 of it) to that difference, which the plain bound, relative to
    the oracle's value, does not cover where the oracle's value is 0 (s0 f and
    s1 r cancelling exactly): the widening carries a factor 1 + 2^-7 for it.
    Without the post-norm f is bit-exact and no widening applies."""
    if not post:
        return None, None
    T = h_ref.shape[0]
    f_ref = oracle.beam_moe_finalize(case.expert_outputs, case.weights, T,
                                     routed_scale=case.routed_scale,
                                     post_weight=case.post_weight, post_eps=1e-6)
    s0 = 1.0 if scales is None else scales[0]
    own_round = 1.0 + 2.0 ** -7
    eh = abs(s0) * bf16_ulp(f_ref)
    if n_ref is None:
        return eh * own_round, None
    hv = bf16_bits_to_f64(h_ref)
    rn = 1.0 / np.sqrt((hv * hv).mean(axis=1, keepdims=True) + next_eps)
    g = np.abs(bf16_bits_to_f64(next_weight)) if next_weight is not None else 1.0
    return eh * own_round, (eh + bf16_ulp(h_ref)) * rn * g * own_round


def run_residual(mf, case, residual_bits, *, post, nxt, scales, inplace=False, tokens=None):
    cap, K, H = case.expert_outputs.shape
    x = dev_bf16(case.expert_outputs.reshape(cap * K, H))
    w = torch.from_numpy(case.weights).cuda()
    r = dev_bf16(residual_bits)
    pw = dev_bf16(case.post_weight) if (post and case.post_weight is not None) else None
    nw = dev_bf16(case.post_weight[::-1].copy()) if nxt == "weighted" else None
    hid_out = r if inplace else None
    h, n = mf.beam_moe_finalize_norm_residual_norm(
        x, w, r, pw, 1e-6 if post else None, nw, 1e-5 if nxt else None, scales,
        case.routed_scale, hidden=hid_out)
    torch.cuda.synchronize()
    if inplace:
        assert h.data_ptr() == r.data_ptr()
    return host_bits(h), (host_bits(n) if n is not None else None), nw


@pytest.mark.parametrize("post", [True, False])
@pytest.mark.parametrize("nxt", [None, "weighted", "plain"])
@pytest.mark.parametrize("scales", [None, (0.5, 2.0)])
def test_residual_norm_matches_oracle(cuda_lib, post, nxt, scales):
    cap, K, H, T = 300, 8, 7168, 290
    case = si.beam_case("resid", cap, K, H, T, routed_scale=2.5, seed=60, poison_dead_rows=True)
    res = si.normal_bf16((T, H), 1.0, 61, 1)
    h, n, _ = run_residual(cuda_lib, case, res, post=post, nxt=nxt, scales=scales)
    rh, rn = oracle.beam_moe_finalize_norm_residual_norm(
        case.expert_outputs, case.weights, res, routed_scale=2.5,
        post_weight=case.post_weight if post else None, post_eps=1e-6 if post else None,
        next_weight=case.post_weight[::-1].copy() if nxt == "weighted" else None,
        next_eps=1e-5 if nxt else None, scales=scales)
    eh, en = residual_bounds(case, rh, rn, post=post, scales=scales, next_eps=1e-5,
                             next_weight=case.post_weight[::-1].copy() if nxt == "weighted" else None)
    compare_bf16(h, rh, extra=eh)
    if nxt:
        compare_bf16(n, rn, extra=en)
    else:
        assert n is None and rn is None
    if not post:
        assert np.array_equal(h, rh)   # no norm on the way to hidden: bit-exact


@pytest.mark.parametrize("K,H", [(1, 256), (32, 8192), (3, 7936), (16, 2048), (32, 1024),
                                 (5, 768)])
def test_residual_norm_shapes_and_in_place(cuda_lib, K, H):
    cap, T = 40, 37
    case = si.beam_case("resid_shapes", cap, K, H, T, routed_scale=1.5, seed=K + H)
    res = si.normal_bf16((T, H), 2.0, 62, 1)
    h, n, nw = run_residual(cuda_lib, case, res, post=True, nxt="weighted", scales=(1.25, -0.75),
                            inplace=True)
    rh, rn = oracle.beam_moe_finalize_norm_residual_norm(
        case.expert_outputs, case.weights, res, routed_scale=1.5, post_weight=case.post_weight,
        post_eps=1e-6, next_weight=case.post_weight[::-1].copy(), next_eps=1e-5,
        scales=(1.25, -0.75))
    eh, en = residual_bounds(case, rh, rn, post=True, scales=(1.25, -0.75), next_eps=1e-5,
                             next_weight=case.post_weight[::-1].copy())
    compare_bf16(h, rh, extra=eh)
    compare_bf16(n, rn, extra=en)


MANY_WAVES = [  # T, H, K, post, next norm, scales, in place, expected kernel
    (1600, 7168, 8, True, "weighted", (1.25, -0.75), False, "beam_token_bulk_multi_kernel"),
    (1600, 7168, 8, True, "weighted", (1.25, -0.75), True, "beam_token_bulk_multi_kernel"),
    (1700, 7168, 8, False, None, None, False, "beam_token_bulk_multi_kernel"),
    (1650, 7168, 5, True, "plain", (0.5, 2.0), True, "beam_token_bulk_multi_kernel"),
    (2500, 4096, 8, True, "weighted", None, False, "beam_token_bulk_multi_kernel"),
    (2200, 5632, 6, True, "weighted", (1.25, -0.75), False, "beam_token_bulk_multi_kernel"),
    # its extra registers would cost a CTA per SM here: one token per CTA
    (2200, 5120, 6, True, "weighted", (1.25, -0.75), False, "beam_token_bulk_kernel"),
    (1000, 7168, 8, True, "weighted", (1.25, -0.75), False, "beam_token_bulk_kernel"),
]


@pytest.mark.parametrize("T,H,K,post,nxt,scales,inplace,kernel", MANY_WAVES)
def test_residual_norm_many_waves(cuda_lib, T, H, K, post, nxt, scales, inplace, kernel):
    # five waves of tokens and more: three tokens per CTA at hidden 4096..7168
    # (with the post-norm off, the next norm off, the hidden output in place)
    case = si.beam_case("resid_waves", T + 3, K, H, T, routed_scale=2.5, seed=64 + T + H,
                        poison_dead_rows=True)
    assert cuda_lib.beam_kernel_name(T, K, H, residual=True) == kernel
    res = si.normal_bf16((T, H), 1.0, 65, 1)
    nwt = case.post_weight[::-1].copy() if nxt == "weighted" else None
    h, n, _ = run_residual(cuda_lib, case, res, post=post, nxt=nxt, scales=scales,
                           inplace=inplace)
    rh, rn = oracle.beam_moe_finalize_norm_residual_norm(
        case.expert_outputs, case.weights, res, routed_scale=2.5,
        post_weight=case.post_weight if post else None, post_eps=1e-6 if post else None,
        next_weight=nwt, next_eps=1e-5 if nxt else None, scales=scales)
    eh, en = residual_bounds(case, rh, rn, post=post, scales=scales, next_eps=1e-5,
                             next_weight=nwt)
    compare_bf16(h, rh, extra=eh)
    if nxt:
        compare_bf16(n, rn, extra=en)
    else:
        assert n is None and rn is None
    if not post:
        assert np.array_equal(h, rh)


def test_residual_multi_token_ctas_after_a_producer_pdl_and_graph(cuda_lib):
    # three tokens per CTA: the residual is written by a Beam call (no post-norm:
    # bit-exact) right before each call on the same stream; programmatic launch
    # off and on give the same bits, and so do two replays of a captured graph
    T, K, H = 1700, 8, 7168
    assert cuda_lib.beam_kernel_name(T, K, H, residual=True) == "beam_token_bulk_multi_kernel"
    case = si.beam_case("resid_modes", T + 2, K, H, T, routed_scale=2.5, seed=90,
                        poison_dead_rows=True)
    src = si.beam_case("resid_modes_src", T, 2, H, T, routed_scale=1.5, post_weight=False,
                       post_eps=None, seed=91)
    x, w = dev_bf16(case.expert_outputs.reshape(-1, H)), torch.from_numpy(case.weights).cuda()
    pw, nwt = dev_bf16(case.post_weight), case.post_weight[::-1].copy()
    nw = dev_bf16(nwt)
    xs, ws = dev_bf16(src.expert_outputs), torch.from_numpy(src.weights).cuda()
    r = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    hid = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    nrm = torch.empty_like(hid)

    def call():
        cuda_lib.beam_moe_finalize(xs, ws, r, src.routed_scale)
        cuda_lib.beam_moe_finalize_norm_residual_norm(x, w, r, pw, 1e-6, nw, 1e-5, (1.25, -0.75),
                                                      2.5, hidden=hid, normalized=nrm)

    def fresh():
        for t in (r, hid, nrm):
            t.fill_(float("nan"))
        torch.cuda.synchronize()

    got = {}
    try:
        for pdl in (False, True):
            cuda_lib.set_programmatic_launch(pdl)
            fresh()
            call()
            torch.cuda.synchronize()
            got[pdl] = (host_bits(hid), host_bits(nrm))
    finally:
        cuda_lib.set_programmatic_launch(True)
    assert all(np.array_equal(a, b) for a, b in zip(got[False], got[True]))
    graph = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st), torch.cuda.graph(graph, stream=st):
        call()
    for _ in range(2):
        fresh()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(hid), got[True][0])
        assert np.array_equal(host_bits(nrm), got[True][1])
    res_ref = oracle_beam(src)
    rh, rn = oracle.beam_moe_finalize_norm_residual_norm(
        case.expert_outputs, case.weights, res_ref, routed_scale=2.5,
        post_weight=case.post_weight, post_eps=1e-6, next_weight=nwt, next_eps=1e-5,
        scales=(1.25, -0.75))
    eh, en = residual_bounds(case, rh, rn, post=True, scales=(1.25, -0.75), next_eps=1e-5,
                             next_weight=nwt)
    compare_bf16(got[True][0], rh, extra=eh)
    compare_bf16(got[True][1], rn, extra=en)


def test_residual_norm_zero_tokens(cuda_lib):
    case = si.beam_case("resid0", 4, 2, 256, 4, seed=63)
    x = dev_bf16(case.expert_outputs.reshape(8, 256))
    r = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    h, n = cuda_lib.beam_moe_finalize_norm_residual_norm(
        x, torch.from_numpy(case.weights).cuda(), r, None, None, None, 1e-6, None)
    assert h.shape == (0, 256) and n.shape == (0, 256)


# ---------------------------------------------------------------------------
# concurrency and size

def test_concurrent_calls_on_two_streams(cuda_lib):
    # the library keeps no per-call state: two calls in flight at once on two
    # streams (different inputs and outputs) both give the oracle's result
    cases = [small_case(700, seed=80), si.beam_case("conc", 600, 8, 7168, 590, seed=81)]
    tp, beam = cases
    g, w, idx, nw = (dev_bf16(tp.gemm2), torch.from_numpy(tp.weights).cuda(),
                     torch.from_numpy(tp.idx).cuda(), dev_bf16(tp.norm_weight))
    x, bw, pw = (dev_bf16(beam.expert_outputs), torch.from_numpy(beam.weights).cuda(),
                 dev_bf16(beam.post_weight))
    out1 = torch.empty((700, 4096), dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty((590, 7168), dtype=torch.bfloat16, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(4):
        cuda_lib.moe_finalize_rmsnorm(g, w, idx, nw, out1, eps=tp.eps, gain_center=tp.gain_center,
                                      weight_before_norm=tp.weight_before_norm, stream=s1)
        cuda_lib.beam_moe_finalize(x, bw, out2, beam.routed_scale, pw, beam.post_eps, stream=s2)
    torch.cuda.synchronize()
    compare_bf16(host_bits(out1), oracle_tp(tp))
    compare_bf16(host_bits(out2), oracle_beam(beam))


@pytest.mark.parametrize("hidden", [256, 512])
@pytest.mark.parametrize("T", [1, 3, 4, 5, 9])
def test_warp_per_token_partial_ctas(cuda_lib, T, hidden):
    # hidden <= 1024 runs one warp per token, two per CTA: token counts that leave
    # the last CTA partly empty
    case = si.tp_case("warp_partial", T, hidden=hidden, top_k=8, indexed_rows=T * 8 + 2,
                      invalid_frac=0.1, weights_dtype="fp32", seed=90 + T)
    compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


def test_many_tokens_small_hidden(cuda_lib):
    # 300000 tokens (a large grid) on the warp-per-token path
    T = 300_000
    case = si.tp_case("many", T, hidden=256, top_k=8, indexed_rows=T * 8, invalid_frac=0.01,
                      weights_dtype="bf16", seed=82)
    compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_consumes_output_of_preceding_torch_kernels(cuda_lib, variant):
    # PyTorch kernels (which know nothing of programmatic launch) write the rows,
    # the index map and the weights right before the call on the same stream
    case = small_case(256, seed=95)
    g0 = dev_bf16(case.gemm2)
    idx0 = torch.from_numpy(case.idx).cuda()
    w0 = torch.from_numpy(case.weights).cuda()
    nw = dev_bf16(case.norm_weight)
    out = torch.empty((256, 4096), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        torch.cuda.synchronize()
        g = g0 * 2                      # exact in BF16: an exponent step
        idx = idx0.clone()
        w = w0 * 1.0
        cuda_lib.moe_finalize_rmsnorm(g, w, idx, nw, out, eps=case.eps,
                                      gain_center=case.gain_center,
                                      weight_before_norm=case.weight_before_norm, variant=variant)
        torch.cuda.synchronize()
    rows2 = f32_bits((bf16_bits_to_f64(case.gemm2) * 2).astype(np.float32))  # on the host
    doubled = si.TpCase("doubled", rows2, case.weights, case.idx, case.norm_weight,
                        case.hidden, case.eps, case.gain_center, case.weight_before_norm)
    compare_bf16(host_bits(out), oracle_tp(doubled))


@pytest.mark.parametrize("variant", TP_VARIANTS)
def test_nan_and_inf_in_valid_rows_propagate_like_the_oracle(cuda_lib, variant):
    # a NaN in a gathered row makes the token's mean square NaN: the whole token
    # is NaN.  An Inf makes the mean square Inf, so 1/rms = 0: the token is 0
    # except where its sum is Inf (Inf * 0 = NaN).  Same on both sides; tokens
    # that do not gather those rows are unaffected.
    case = small_case(40, seed=96)
    g = case.gemm2.copy()
    nan_row, inf_row = int(case.idx[3, 0]), int(case.idx[9, 2])
    g[nan_row, 5] = 0x7FC0
    g[inf_row, 100] = 0x7F80
    case.gemm2 = g
    got = run_tp(cuda_lib, case, variant)
    ref = oracle_tp(case)
    r9 = bf16_bits_to_f64(ref[9])
    assert np.isnan(bf16_bits_to_f64(ref[3])).all()
    assert np.argwhere(np.isnan(r9)).ravel().tolist() == [100] and np.all(r9[~np.isnan(r9)] == 0)
    compare_bf16(got, ref)


@pytest.mark.parametrize("variant", ("token_cta", "bulk", "cluster"))
def test_subnormal_inputs(cuda_lib, variant):
    # BF16 subnormal rows (no flush to zero on either side)
    case = si.tp_case("subnormal", 32, indexed_rows=300, sigma=3e-39, invalid_frac=0.02,
                      weights_dtype="fp32", seed=97, eps=1e-30)
    assert (case.gemm2 & 0x7F80 == 0).mean() > 0.5     # mostly subnormal BF16 values
    compare_bf16(run_tp(cuda_lib, case, variant), oracle_tp(case))
