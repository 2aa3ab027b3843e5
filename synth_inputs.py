"""Seeded synthetic inputs for the MoE finalize path (shared by tests and bench).

This module only draws random numbers and lays them out; it holds none of the
finalize arithmetic.  The same bytes go to the CPU oracle and to the CUDA
library.  Every tensor comes from numpy's PCG64 generator, seeded from
``SeedSequence([seed, tensor_id])`` and split into a fixed number of chunks
(each with its own spawned stream), so the bytes depend on the seed and the
shape only, not on how many threads draw them.

The workloads mirror the shapes and distributions of the pages' operation:

* flashinfer.comm.tp_moe_finalize_rmsnorm: hidden 4096, top-k 8, BF16 GEMM2
  rows grouped by expert (the permuted layout) with optional padding rows and a padded row
  stride (a multiple of 8 elements), an int32 index map with negative or
  out-of-range entries, BF16 or FP32 routing weights, a BF16 norm weight.
* beam_moe_finalize: token-major BF16 [capacity, top_k, hidden], FP32
  weights [capacity, top_k], live_tokens <= capacity.

BF16 tensors are numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BF16_NAN = np.uint16(0x7FC0)

# tensor ids for SeedSequence([seed, id])
_ID_ROWS, _ID_IDX, _ID_INVALID, _ID_LOGITS, _ID_NORM, _ID_EXPERT = 1, 2, 3, 4, 5, 6

_CHUNK = 1 << 24  # elements per independently seeded chunk


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to BF16 (nearest, ties to even); bit patterns."""
    u = a.view(np.uint32).copy()
    u += ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return (u >> 16).astype(np.uint16)


def normal_bf16(shape, sigma: float, seed: int, tensor_id: int, mu: float = 0.0) -> np.ndarray:
    """BF16 bits of mu + sigma * N(0, 1), drawn in float32 chunks on all host cores."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    kids = np.random.SeedSequence([seed, tensor_id]).spawn(nchunks)

    def work(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(kids[c]))
        a = g.standard_normal(hi - lo, dtype=np.float32)
        if sigma != 1.0:
            a *= np.float32(sigma)
        if mu != 0.0:
            a += np.float32(mu)
        out[lo:hi] = _f32_to_bf16_bits(a)

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def softmax_weights(tokens: int, top_k: int, seed: int, dtype: str) -> np.ndarray:
    """Routing weights: softmax over top_k N(0,1) logits per token, in double,
    then cast to float32 ("fp32") or to BF16 bits ("bf16")."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _ID_LOGITS])))
    logits = g.standard_normal((tokens, top_k))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    p = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    if dtype == "fp32":
        return np.ascontiguousarray(p)
    assert dtype == "bf16"
    return _f32_to_bf16_bits(p)


def pack_topk(weights_bf16: np.ndarray, seed: int, num_experts: int = 256) -> np.ndarray:
    """int32 routing words ``(expert_id << 16) | bf16 bits`` (the producer MoE's
    packed topk_ids layout) holding the given BF16 weights and random expert
    ids in [0, num_experts)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _ID_EXPERT])))
    experts = g.integers(0, num_experts, size=weights_bf16.shape).astype(np.uint32)
    return ((experts << 16) | weights_bf16.astype(np.uint32)).view(np.int32)


def permutation_index(tokens: int, top_k: int, indexed_rows: int, total_rows: int,
                      invalid_frac: float, seed: int) -> np.ndarray:
    """int32 [tokens, top_k]: a random injective map into rows [0, indexed_rows),
    with round(invalid_frac * tokens * top_k) slots, chosen without
    replacement, replaced by -1 or total_rows (a fair coin each)."""
    n = tokens * top_k
    assert n <= indexed_rows <= total_rows
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _ID_IDX])))
    idx = g.permutation(indexed_rows)[:n].astype(np.int32)
    n_bad = int(round(invalid_frac * n))
    if n_bad:
        g2 = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _ID_INVALID])))
        pos = g2.choice(n, size=n_bad, replace=False)
        coin = g2.integers(0, 2, size=n_bad)
        idx[pos] = np.where(coin == 0, -1, total_rows).astype(np.int32)
    return idx.reshape(tokens, top_k)


@dataclass
class TpCase:
    """Inputs of one tp_moe_finalize_rmsnorm call (host arrays)."""
    name: str
    gemm2: np.ndarray          # uint16 [rows, row_stride]
    weights: np.ndarray        # float32, uint16 (BF16) or int32 (packed) [T, K]
    idx: np.ndarray            # int32 [T, K]
    norm_weight: np.ndarray    # uint16 [hidden]
    hidden: int
    eps: float
    gain_center: float
    weight_before_norm: bool
    meta: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return self.idx.shape[0]

    @property
    def top_k(self) -> int:
        return self.idx.shape[1]


@dataclass
class BeamCase:
    """Inputs of one beam_moe_finalize call (host arrays)."""
    name: str
    expert_outputs: np.ndarray  # uint16 [capacity, K, H]
    weights: np.ndarray         # float32 [capacity, K]
    live_tokens: int
    routed_scale: float
    post_weight: np.ndarray | None
    post_eps: float | None
    meta: dict = field(default_factory=dict)


def tp_case(name: str, tokens: int, *, hidden: int = 4096, top_k: int = 8,
            indexed_rows: int | None = None, padding_rows: int = 0, row_stride: int | None = None,
            sigma: float = 1.0, invalid_frac: float = 0.0, weights_dtype: str = "fp32",
            norm_mu: float = 0.0, norm_sigma: float = 0.1, gain_center: float = 1.0,
            eps: float = 1e-6, weight_before_norm: bool = False, seed: int = 0,
            poison_padding: bool = False) -> TpCase:
    """A tp_moe_finalize_rmsnorm workload.  Rows [0, indexed_rows) are the
    ones the index map may reference; ``padding_rows`` more rows follow them
    (never indexed); columns [hidden, row_stride) are row padding.  With
    ``poison_padding`` every padding element is a BF16 NaN, otherwise zero."""
    indexed_rows = tokens * top_k if indexed_rows is None else indexed_rows
    row_stride = hidden if row_stride is None else row_stride
    rows = indexed_rows + padding_rows
    live = normal_bf16((indexed_rows, hidden), sigma, seed, _ID_ROWS)
    if row_stride == hidden and padding_rows == 0:
        gemm2 = live
    else:
        fill = BF16_NAN if poison_padding else np.uint16(0)
        gemm2 = np.full((rows, row_stride), fill, dtype=np.uint16)
        gemm2[:indexed_rows, :hidden] = live
        del live
    idx = permutation_index(tokens, top_k, indexed_rows, rows, invalid_frac, seed)
    if weights_dtype == "packed":
        weights = pack_topk(softmax_weights(tokens, top_k, seed, "bf16"), seed)
    else:
        weights = softmax_weights(tokens, top_k, seed, weights_dtype)
    norm_weight = normal_bf16((hidden,), norm_sigma, seed, _ID_NORM, mu=norm_mu)
    return TpCase(name, gemm2, weights, idx, norm_weight, hidden, eps, gain_center,
                  weight_before_norm, meta=dict(indexed_rows=indexed_rows, rows=rows,
                                                row_stride=row_stride, sigma=sigma,
                                                invalid_frac=invalid_frac, seed=seed))


def beam_case(name: str, capacity: int, top_k: int, hidden: int, live_tokens: int, *,
              routed_scale: float = 1.0, post_weight: bool = True, post_eps: float | None = 1e-6,
              post_weight_sigma: float = 0.05, seed: int = 0,
              poison_dead_rows: bool = False) -> BeamCase:
    """A beam_moe_finalize workload; rows t >= live_tokens of expert_outputs
    are BF16 NaN when ``poison_dead_rows`` (they must never be read)."""
    x = normal_bf16((capacity, top_k, hidden), 1.0, seed, _ID_ROWS)
    if poison_dead_rows and live_tokens < capacity:
        x[live_tokens:] = BF16_NAN
    w = softmax_weights(capacity, top_k, seed, "fp32")
    pw = normal_bf16((hidden,), post_weight_sigma, seed, _ID_NORM, mu=1.0) if post_weight else None
    return BeamCase(name, x, w, live_tokens, routed_scale, pw, post_eps,
                    meta=dict(capacity=capacity, seed=seed))


# ---------------------------------------------------------------------------
# The five workloads of this path.

def finalize_16_tokens() -> TpCase:
    """16 tokens: gemm2 [128, 4096] ~N(0,1); idx = permutation of 0..127 with
    5% of slots -1 or 128; FP32 softmax weights; norm_weight ~N(0, 0.1);
    gain_center 1.0, eps 1e-6, norm weight after the RMS."""
    return tp_case("finalize_T16", 16, indexed_rows=128, invalid_frac=0.05,
                   weights_dtype="fp32", gain_center=1.0, eps=1e-6, weight_before_norm=False)


def finalize_4096_tokens_padded(poison_padding: bool = True) -> TpCase:
    """4096 tokens: gemm2 [36864, 4160] (row stride 4160, 4096 live columns,
    4096 padding rows never indexed); idx = permutation of the 32768 real rows,
    2% invalid; BF16 softmax weights; eps 1e-5, norm weight before the RMS."""
    return tp_case("finalize_T4096_stride4160", 4096, indexed_rows=32768, padding_rows=4096,
                   row_stride=4160, invalid_frac=0.02, weights_dtype="bf16", gain_center=1.0,
                   eps=1e-5, weight_before_norm=True, poison_padding=poison_padding)


def beam_8000_live(poison_dead_rows: bool = True) -> BeamCase:
    """Beam: expert_outputs [8192, 8, 7168] ~N(0,1); FP32 softmax weights;
    live 8000; routed_scale 2.5; post_weight ~1+N(0, 0.05); post_eps 1e-6."""
    return beam_case("beam_cap8192_live8000_H7168", 8192, 8, 7168, 8000, routed_scale=2.5,
                     post_weight=True, post_eps=1e-6, poison_dead_rows=poison_dead_rows)


DECODE_TOKENS = (1, 8, 32, 128)


def finalize_decode(tokens: int) -> TpCase:
    """Decode sizes: rows = 10 * tokens ~N(0,1); a random injective map (8T of
    the 10T rows used), 3% invalid; FP32 weights; gain_center 0.0, eps 1e-6,
    norm weight after the RMS.  The norm weight is ~1+N(0, 0.1), so that the
    effective gain stays near 1 with gain_center 0."""
    return tp_case(f"finalize_decode_T{tokens}", tokens, indexed_rows=10 * tokens,
                   invalid_frac=0.03, weights_dtype="fp32", norm_mu=1.0, norm_sigma=0.1,
                   gain_center=0.0, eps=1e-6, weight_before_norm=False, seed=0)


ROOFLINE_TOKENS = 32768
ROOFLINE_INDEXED_ROWS = 262144
ROOFLINE_PADDING_ROWS = 26214   # 10% unused padding rows: 288358 rows in all


def finalize_32768_tokens(weight_before_norm: bool = False) -> TpCase:
    """Bandwidth workload: 32768 tokens, gemm2 [288358, 4096] ~N(0, 2)
    (262144 indexed rows plus 26214 never-indexed padding rows); random
    permutation map with 1% invalid; FP32 weights; norm_weight ~N(0, 0.1);
    gain_center 1.0, eps 1e-6."""
    return tp_case(f"finalize_T32768_{'before' if weight_before_norm else 'after'}",
                   ROOFLINE_TOKENS, indexed_rows=ROOFLINE_INDEXED_ROWS,
                   padding_rows=ROOFLINE_PADDING_ROWS, sigma=2.0, invalid_frac=0.01,
                   weights_dtype="fp32", gain_center=1.0, eps=1e-6,
                   weight_before_norm=weight_before_norm)


def algorithmic_bytes_tp(tokens: int, hidden: int = 4096, top_k: int = 8,
                         weight_bytes: int = 4) -> int:
    """K*H*2 gathered + H*2 written + K*4 index + K*sizeof(w), per token."""
    return tokens * (top_k * hidden * 2 + hidden * 2 + top_k * 4 + top_k * weight_bytes)


def algorithmic_bytes_beam(live_tokens: int, hidden: int, top_k: int) -> int:
    """K*H*2 read + H*2 written + K*4 weight bytes, per live token."""
    return live_tokens * (top_k * hidden * 2 + hidden * 2 + top_k * 4)


def algorithmic_bytes_beam_residual(tokens: int, hidden: int, top_k: int, next_norm: bool) -> int:
    """Beam bytes plus the residual read, the hidden write and (with the next
    norm) the normalized write, per token."""
    return tokens * (top_k * hidden * 2 + top_k * 4 + hidden * 2 * (3 if next_norm else 2))
