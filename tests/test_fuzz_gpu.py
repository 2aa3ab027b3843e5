"""Seeded random configurations of every operation and kernel against the
oracle (GPU), and calls from several host threads at once.

MF_FUZZ_SEEDS=N runs N seeds of each random test instead of the default
counts (a wide sweep: MF_FUZZ_SEEDS=300 python -m pytest tests/test_fuzz_gpu.py)."""
import os
import threading

import numpy as np
import pytest

import synth_inputs as si
from gpu_common import dev_bf16, host_bits, oracle_beam, oracle_tp, run_beam, run_tp
from helpers import compare_bf16

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def _seeds(default):
    return range(int(os.environ.get("MF_FUZZ_SEEDS", default)))


def _random_tp(seed):
    rng = np.random.default_rng(1000 + seed)
    specialised = rng.random() < 0.5
    H = 4096 if specialised else int(rng.integers(1, 33)) * 256
    K = 8 if specialised else int(rng.integers(1, 33))
    T = int(rng.choice([1, 2, 7, 33, 150, 1023, 1024, 1500]))
    stride = H + 8 * int(rng.integers(0, 4))
    extra_rows = int(rng.integers(0, 50))
    case = si.tp_case(f"fuzz{seed}", T, hidden=H, top_k=K, indexed_rows=T * K + extra_rows,
                      padding_rows=int(rng.integers(0, 5)), row_stride=stride,
                      sigma=float(rng.choice([0.5, 1.0, 3.0])),
                      invalid_frac=float(rng.choice([0.0, 0.05, 0.5])),
                      weights_dtype=str(rng.choice(["fp32", "bf16", "packed"])),
                      norm_mu=float(rng.choice([0.0, 1.0])), gain_center=float(rng.choice([0.0, 1.0, -0.5])),
                      eps=float(rng.choice([1e-6, 1e-5, 0.1])),
                      weight_before_norm=bool(rng.random() < 0.5), seed=seed,
                      poison_padding=True)
    variants = ["auto", "bulk"] + (["token_cta", "cluster"] if specialised else [])
    return case, variants


@pytest.mark.parametrize("seed", _seeds(32))
def test_fuzz_finalize(cuda_lib, seed):
    case, variants = _random_tp(seed)
    ref = oracle_tp(case)
    for v in variants:
        compare_bf16(run_tp(cuda_lib, case, v), ref)


@pytest.mark.parametrize("seed", _seeds(8))
def test_fuzz_finalize_multi_token(cuda_lib, seed):
    # hidden 4096 / top-k 8 at token counts where the staged kernel takes three
    # tokens per CTA (from five waves of resident CTAs: 2280 on GB300)
    rng = np.random.default_rng(5000 + seed)
    T = int(rng.integers(2280, 6001))
    case = si.tp_case(f"fuzz_multi{seed}", T, indexed_rows=T * 8 + int(rng.integers(0, 50)),
                      padding_rows=int(rng.integers(0, 5)),
                      row_stride=4096 + 8 * int(rng.integers(0, 4)),
                      sigma=float(rng.choice([0.5, 1.0, 3.0])),
                      invalid_frac=float(rng.choice([0.0, 0.05, 0.5])),
                      weights_dtype=str(rng.choice(["fp32", "bf16", "packed"])),
                      gain_center=float(rng.choice([0.0, 1.0, -0.5])),
                      eps=float(rng.choice([1e-6, 1e-5, 0.1])),
                      weight_before_norm=bool(rng.random() < 0.5), seed=seed,
                      poison_padding=True)
    compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


@pytest.mark.parametrize("seed", _seeds(8))
def test_fuzz_finalize_many_tokens_other_sizes(cuda_lib, seed):
    # other sizes at token counts where the generic and warp-per-token kernels
    # take several tokens per CTA or warp (when a token fits one piece)
    rng = np.random.default_rng(6000 + seed)
    H = int(rng.choice([256, 512, 768, 1024, 1280, 2048, 2304, 3072, 7168]))
    K = int(rng.integers(1, 17 if H == 256 else 9))
    T = int(rng.integers(22000, 36000)) if H <= 1024 else int(rng.integers(3100, 9000))
    case = si.tp_case(f"fuzz_many{seed}", T, hidden=H, top_k=K, indexed_rows=T * K + 7,
                      padding_rows=int(rng.integers(0, 5)), row_stride=H + 8 * int(rng.integers(0, 4)),
                      invalid_frac=float(rng.choice([0.0, 0.05, 0.5])),
                      weights_dtype=str(rng.choice(["fp32", "bf16", "packed"])),
                      gain_center=float(rng.choice([0.0, 1.0])), eps=float(rng.choice([1e-6, 0.1])),
                      weight_before_norm=bool(rng.random() < 0.5), seed=seed, poison_padding=True)
    compare_bf16(run_tp(cuda_lib, case, "auto"), oracle_tp(case))


@pytest.mark.parametrize("seed", _seeds(24))
def test_fuzz_beam(cuda_lib, seed):
    rng = np.random.default_rng(2000 + seed)
    H = int(rng.integers(1, 33)) * 256
    K = int(rng.integers(1, 33))
    cap = int(rng.integers(1, 200))
    live = int(rng.integers(0, cap + 1))
    norm = bool(rng.random() < 0.7)
    case = si.beam_case(f"bfuzz{seed}", cap, K, H, live, routed_scale=float(rng.choice([1.0, 2.5, 0.375])),
                        post_weight=norm and bool(rng.random() < 0.5),  # a weight needs its eps
                        post_eps=1e-6 if norm else None,
                        seed=seed, poison_dead_rows=True)
    if live == 0:
        return
    ref = oracle_beam(case)
    for v in ("auto", "token_cta"):
        compare_bf16(run_beam(cuda_lib, case, v), ref)


@pytest.mark.parametrize("seed", _seeds(4))
def test_fuzz_beam_many_tokens(cuda_lib, seed):
    # token counts and sizes where plain Beam may take several tokens per CTA
    # (hidden 4096..7168 with two chunks per thread, a token in one piece)
    rng = np.random.default_rng(8000 + seed)
    H = int(rng.choice([4096, 4608, 5120, 5632, 6144, 6656, 7168]))
    K = int(rng.integers(1, 9))
    T = int(rng.integers(2500, 4000))
    norm = bool(rng.random() < 0.7)
    weighted = bool(rng.random() < 0.8) and norm  # post_weight only with the norm
    case = si.beam_case(f"bfuzzm{seed}", T + int(rng.integers(0, 5)), K, H, T,
                        routed_scale=float(rng.choice([1.0, 2.5])), seed=seed,
                        post_weight=weighted, post_eps=1e-6 if norm else None,
                        poison_dead_rows=True)
    assert cuda_lib.beam_kernel_name(T, K, H) in ("beam_token_bulk_kernel",
                                                  "beam_token_bulk_multi_kernel")
    got, ref = run_beam(cuda_lib, case, "auto"), oracle_beam(case)
    compare_bf16(got, ref)
    if not norm:
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("seed", _seeds(16))
def test_fuzz_residual_norm(cuda_lib, seed):
    import oracle
    import test_parity_gpu as tpg
    rng = np.random.default_rng(3000 + seed)
    H = int(rng.integers(1, 33)) * 256
    K = int(rng.integers(1, 33))
    T = int(rng.integers(1, 160))
    post = bool(rng.random() < 0.7)
    nxt = [None, "weighted", "plain"][int(rng.integers(0, 3))]
    scales = None if rng.random() < 0.5 else (float(rng.choice([0.5, 1.25, -0.75])),
                                               float(rng.choice([2.0, 1.0, -0.5])))
    case = si.beam_case(f"rfuzz{seed}", T + int(rng.integers(0, 5)), K, H, T,
                        routed_scale=float(rng.choice([1.0, 2.5])), seed=seed)
    res = si.normal_bf16((T, H), float(rng.choice([0.5, 2.0])), seed, 9)
    h, n, _ = tpg.run_residual(cuda_lib, case, res, post=post, nxt=nxt, scales=scales,
                               inplace=bool(rng.random() < 0.3))
    nw = case.post_weight[::-1].copy() if nxt == "weighted" else None
    rh, rn = oracle.beam_moe_finalize_norm_residual_norm(
        case.expert_outputs, case.weights, res, routed_scale=case.routed_scale,
        post_weight=case.post_weight if post else None, post_eps=1e-6 if post else None,
        next_weight=nw, next_eps=1e-5 if nxt else None, scales=scales)
    eh, en = tpg.residual_bounds(case, rh, rn, post=post, scales=scales, next_eps=1e-5,
                                 next_weight=nw)
    compare_bf16(h, rh, extra=eh)
    if nxt:
        compare_bf16(n, rn, extra=en)
    if not post:
        assert np.array_equal(h, rh)   # no norm on the way to hidden: bit-exact


@pytest.mark.parametrize("seed", _seeds(4))
def test_fuzz_residual_norm_many_tokens(cuda_lib, seed):
    # token counts where the residual op may take three tokens per CTA (hidden
    # 4096..7168 with two chunks per thread, a token in one piece; one token per
    # CTA where the several-tokens kernel would cost a CTA per SM)
    import oracle
    import test_parity_gpu as tpg
    rng = np.random.default_rng(7000 + seed)
    H = int(rng.choice([4096, 4608, 5120, 5632, 6144, 6656, 7168]))
    K = int(rng.integers(1, 9))
    T = int(rng.integers(2300, 3500))
    post = bool(rng.random() < 0.7)
    nxt = [None, "weighted", "plain"][int(rng.integers(0, 3))]
    scales = None if rng.random() < 0.5 else (float(rng.choice([0.5, 1.25, -0.75])),
                                               float(rng.choice([2.0, 1.0, -0.5])))
    case = si.beam_case(f"rfuzzm{seed}", T + int(rng.integers(0, 5)), K, H, T,
                        routed_scale=float(rng.choice([1.0, 2.5])), seed=seed,
                        poison_dead_rows=True)
    assert cuda_lib.beam_kernel_name(T, K, H, residual=True) in ("beam_token_bulk_kernel",
                                                                "beam_token_bulk_multi_kernel")
    res = si.normal_bf16((T, H), float(rng.choice([0.5, 2.0])), seed, 9)
    h, n, _ = tpg.run_residual(cuda_lib, case, res, post=post, nxt=nxt, scales=scales,
                               inplace=bool(rng.random() < 0.3))
    nw = case.post_weight[::-1].copy() if nxt == "weighted" else None
    rh, rn = oracle.beam_moe_finalize_norm_residual_norm(
        case.expert_outputs, case.weights, res, routed_scale=case.routed_scale,
        post_weight=case.post_weight if post else None, post_eps=1e-6 if post else None,
        next_weight=nw, next_eps=1e-5 if nxt else None, scales=scales)
    eh, en = tpg.residual_bounds(case, rh, rn, post=post, scales=scales, next_eps=1e-5,
                                 next_weight=nw)
    compare_bf16(h, rh, extra=eh)
    if nxt:
        compare_bf16(n, rn, extra=en)
    if not post:
        assert np.array_equal(h, rh)


def test_calls_from_several_host_threads(cuda_lib):
    # four host threads, each with its own stream and inputs, calling at once
    cases = [small_case_for_thread(i) for i in range(4)]
    refs = [oracle_tp(c) for c in cases]
    results = [None] * 4
    errors = []

    def worker(i):
        try:
            c = cases[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                g, w = dev_bf16(c.gemm2), torch.from_numpy(c.weights).cuda()
                idx, nw = torch.from_numpy(c.idx).cuda(), dev_bf16(c.norm_weight)
                out = torch.empty((c.num_tokens, 4096), dtype=torch.bfloat16, device="cuda")
                for _ in range(20):
                    cuda_lib.moe_finalize_rmsnorm(g, w, idx, nw, out, eps=c.eps,
                                                  gain_center=c.gain_center,
                                                  weight_before_norm=c.weight_before_norm,
                                                  stream=s)
                s.synchronize()
                results[i] = host_bits(out)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for got, ref in zip(results, refs):
        compare_bf16(got, ref)


def small_case_for_thread(i):
    return si.tp_case(f"thread{i}", [5, 70, 600, 1200][i], indexed_rows=[5, 70, 600, 1200][i] * 8,
                      invalid_frac=0.05, weights_dtype="fp32", seed=300 + i,
                      weight_before_norm=bool(i % 2))
