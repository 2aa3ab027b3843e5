"""GB300 (sm_103a) MoE finalize + RMSNorm and Beam finalize.

Thin Python binding over the C ABI of ``libmoe_finalize.so``
(include/moe_finalize.h): it checks tensor metadata, reads pointers, sizes
and the current CUDA stream, and calls the library.  Every arithmetic step
runs in the library's CUDA kernels; PyTorch only supplies device memory and
streams.  There is no CPU fallback: without the built library the calls raise.

* ``moe_finalize_rmsnorm`` (alias ``tp_moe_finalize_rmsnorm``) follows
  flashinfer.comm.tp_moe_finalize_rmsnorm (API page), on one GPU.
* ``beam_moe_finalize`` follows vllm.models.beam.nvidia.moe_finalize,
  beam_moe_finalize.
* ``beam_moe_finalize_norm_residual_norm`` follows the same page's function of
  that name on one GPU (its residual step is a reading; see the C header).
"""
from __future__ import annotations


import torch

from ._abi import (MF_DTYPE_BF16, MF_DTYPE_FP32, MF_DTYPE_PACKED_TOPK, VARIANT_NAMES, VARIANTS, MoeFinalizeError,
                   check, lib)

__all__ = [
    "moe_finalize_rmsnorm", "tp_moe_finalize_rmsnorm", "beam_moe_finalize",
    "beam_moe_finalize_norm_residual_norm", "MoeFinalizeError",
    "device_status", "selftest_wait_timeout", "select_finalize_variant", "select_beam_variant",
    "finalize_kernel_name", "beam_kernel_name", "finalize_data_movement",
    "version", "set_programmatic_launch", "programmatic_launch", "HIDDEN", "TOP_K",
]

HIDDEN = 4096
TOP_K = 8


_BF16 = torch.bfloat16
_WEIGHT_DTYPES = {torch.bfloat16: MF_DTYPE_BF16, torch.float32: MF_DTYPE_FP32,
                  torch.int32: MF_DTYPE_PACKED_TOPK}


def _stream_ptr(stream, device) -> int:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return s.cuda_stream


def _on_device(dev: torch.device, fn, *args) -> int:
    """Call fn with dev as the current CUDA device (switching only if needed)."""
    if dev.index is None or dev.index == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


def _req(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _variant(name: str) -> int:
    v = VARIANTS.get(name)
    if v is None:
        raise ValueError(f"unknown variant {name!r}; one of {sorted(VARIANTS)}")
    return v


def moe_finalize_rmsnorm(gemm2_permuted: torch.Tensor, expert_weights: torch.Tensor,
                         expanded_idx_to_permuted_idx: torch.Tensor, norm_weight: torch.Tensor,
                         output: torch.Tensor, *, eps: float, gain_center: float,
                         weight_before_norm: bool, variant: str = "auto",
                         stream: torch.cuda.Stream | None = None) -> None:
    """Finalize + RMSNorm into ``output`` (BF16 [num_tokens, hidden]).

    gemm2_permuted: BF16 (rows, >= 4096), unit last-dim stride, row stride a
    multiple of 8.  expert_weights: (num_tokens, top_k) BF16, FP32, or int32
    packed routing words ``(expert_id << 16) | bf16 weight bits`` (the
    producer MoE's topk_ids).  expanded_idx_to_permuted_idx: int32
    (num_tokens, top_k); negative or out-of-range entries contribute zero.
    norm_weight: BF16 (hidden,).  hidden 4096 with top_k 8, or hidden
    256..8192 (a multiple of 256) with top_k 1..32.
    Asynchronous on ``stream`` (default: the current stream).
    """
    g, w, idx, nw, out = gemm2_permuted, expert_weights, expanded_idx_to_permuted_idx, \
        norm_weight, output
    wdt, row_stride, dev = _finalize_operands(g, w, idx, out)
    if nw.dim() != 1 or nw.dtype != _BF16 or not nw.is_contiguous():
        raise ValueError("norm_weight must be a contiguous 1-D BF16 tensor")
    if nw.shape[0] != out.shape[1]:
        raise ValueError("norm_weight and output disagree on hidden")
    if nw.device != dev:
        raise ValueError("all tensors must be on the same CUDA device")
    st = _on_device(dev, lib().moe_finalize_rmsnorm_variant,
                    g.data_ptr(), g.shape[0], row_stride, w.data_ptr(), wdt, idx.data_ptr(),
                    nw.data_ptr(), out.data_ptr(), out.shape[0], out.shape[1], idx.shape[1],
                    float(eps), float(gain_center), 1 if weight_before_norm else 0,
                    _variant(variant), _stream_ptr(stream, dev))
    check(st, "moe_finalize_rmsnorm")


def _finalize_operands(g, w, idx, out):
    """Metadata checks shared by the finalize calls; returns the weights' dtype
    code, gemm2's row stride and the device."""
    gs, os_, ids = g.shape, out.shape, idx.shape
    wdt = _WEIGHT_DTYPES.get(w.dtype)
    if len(gs) != 2 or g.dtype != _BF16 or (g.stride(1) != 1 and gs[1] > 1):
        raise ValueError("gemm2_permuted must be a 2-D BF16 tensor with unit last-dim stride")
    if len(os_) != 2 or out.dtype != _BF16 or not out.is_contiguous():
        raise ValueError("output must be a contiguous 2-D BF16 tensor")
    if len(ids) != 2 or idx.dtype != torch.int32 or not idx.is_contiguous():
        raise ValueError("expanded_idx_to_permuted_idx must be a contiguous 2-D int32 tensor")
    if wdt is None or not w.is_contiguous() or w.shape != ids:
        raise ValueError("expert_weights must be contiguous BF16, FP32 or packed int32 with the "
                         "index map's shape")
    if os_[0] != ids[0]:
        raise ValueError("output and the index map disagree on num_tokens")
    if gs[1] < os_[1]:
        # a narrowed view would otherwise let the kernel read past its columns
        raise ValueError("gemm2_permuted has fewer columns than output's hidden")
    dev = out.device
    if dev.type != "cuda" or g.device != dev or w.device != dev or idx.device != dev:
        raise ValueError("all tensors must be on the same CUDA device")
    row_stride = g.stride(0) if gs[0] > 1 else max(gs[1], g.stride(0))
    return wdt, row_stride, dev


def finalize_data_movement(gemm2_permuted: torch.Tensor, expert_weights: torch.Tensor,
                           expanded_idx_to_permuted_idx: torch.Tensor, output: torch.Tensor, *,
                           stream: torch.cuda.Stream | None = None) -> None:
    """Measurement aid: the memory traffic of ``moe_finalize_rmsnorm`` at hidden
    4096 / top_k 8 on the same operands, without its arithmetic (``output``
    receives a meaningless bit pattern).  Timed beside the finalize, it shows
    what the finalize adds to the cost of the bytes themselves."""
    g, w, idx, out = gemm2_permuted, expert_weights, expanded_idx_to_permuted_idx, output
    if out.dim() != 2 or idx.dim() != 2 or out.shape[1] != HIDDEN or idx.shape[1] != TOP_K:
        raise ValueError(f"the data-movement kernel covers hidden {HIDDEN} with top_k {TOP_K}")
    wdt, row_stride, dev = _finalize_operands(g, w, idx, out)
    st = _on_device(dev, lib().mf_finalize_data_movement, g.data_ptr(), g.shape[0], row_stride,
                    w.data_ptr(), wdt, idx.data_ptr(), out.data_ptr(), out.shape[0],
                    _stream_ptr(stream, dev))
    check(st, "finalize_data_movement")


tp_moe_finalize_rmsnorm = moe_finalize_rmsnorm


def beam_moe_finalize(expert_outputs: torch.Tensor, expert_weights: torch.Tensor,
                      output: torch.Tensor, routed_scale: float = 1.0,
                      post_weight: torch.Tensor | None = None, post_eps: float | None = None, *,
                      variant: str = "auto",
                      stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Beam finalize of the live rows (``output.shape[0]``) into ``output``.

    expert_outputs: contiguous BF16 [capacity, top_k, hidden].  expert_weights:
    contiguous FP32 [>= live, top_k].  output: contiguous BF16 [live, hidden].
    post_eps None omits the normalisation; post_weight None with post_eps set
    is an unweighted RMSNorm.  Returns ``output``.
    """
    x, w, out = expert_outputs, expert_weights, output
    _req(x.dim() == 3 and w.dim() == 2 and out.dim() == 2, "expected 3-D, 2-D, 2-D tensors")
    _req(x.dtype == torch.bfloat16 and out.dtype == torch.bfloat16 and w.dtype == torch.float32,
         "expert_outputs/output must be BF16 and expert_weights FP32")
    _req(x.is_contiguous() and w.is_contiguous() and out.is_contiguous(),
         "expert_outputs, expert_weights and output must be contiguous")
    cap, top_k, hidden = x.shape
    _req(out.shape[1] == hidden and w.shape[1] == top_k, "shapes disagree on hidden or top_k")
    dev = out.device
    _req(dev.type == "cuda" and x.device == dev and w.device == dev,
         "all tensors must be on the same CUDA device")
    pw_ptr = None
    if post_weight is not None:
        _req(post_eps is not None, "post_weight requires post_eps")
        _req(post_weight.shape == (hidden,) and post_weight.is_contiguous() and
             post_weight.dtype == torch.bfloat16 and post_weight.device == dev,
             "post_weight must be a contiguous BF16 [hidden] tensor on the output's device")
        pw_ptr = post_weight.data_ptr()
    st = _on_device(dev, lib().beam_moe_finalize_variant,
                    x.data_ptr(), cap, w.data_ptr(), w.shape[0], out.data_ptr(), out.shape[0],
                    top_k, hidden, float(routed_scale), pw_ptr, float(post_eps or 0.0),
                    int(post_eps is not None), _variant(variant), _stream_ptr(stream, dev))
    check(st, "beam_moe_finalize")
    return out


def beam_moe_finalize_norm_residual_norm(
        gemm2_permuted: torch.Tensor, expert_weights: torch.Tensor, residual: torch.Tensor,
        post_weight: torch.Tensor | None, post_eps: float | None,
        next_weight: torch.Tensor | None, next_eps: float | None,
        scales: tuple[float, float] | None, routed_scale: float = 1.0, *,
        hidden: torch.Tensor | None = None, normalized: torch.Tensor | None = None,
        stream: torch.cuda.Stream | None = None) -> tuple[torch.Tensor, torch.Tensor | None]:
    """Beam finalize of the first ``residual.shape[0]`` tokens, then the residual
    add and the next RMSNorm, in one kernel.  Returns ``(hidden, normalized)``;
    ``normalized`` is None without ``next_eps``.

    gemm2_permuted: contiguous BF16 [capacity * top_k, hidden] token-major rows
    (or [capacity, top_k, hidden]); expert_weights: FP32 [capacity, top_k];
    residual: BF16 [tokens, hidden].  hidden = BF16(s0 * finalized + s1 *
    residual) with scales (s0, s1), (1, 1) when None; ``hidden`` may be
    ``residual`` itself.
    """
    # the C ABI rejects the same combination (MF_ERR_INVALID)
    _req(normalized is None or next_eps is not None,
         "normalized is only written by the next norm: pass next_eps with it")
    w, r = expert_weights, residual
    _req(w.dim() == 2 and w.dtype == torch.float32 and w.is_contiguous(),
         "expert_weights must be a contiguous 2-D FP32 tensor")
    cap, top_k = w.shape
    _req(r.dim() == 2 and r.dtype == torch.bfloat16 and r.is_contiguous(),
         "residual must be a contiguous 2-D BF16 tensor")
    tokens, hid_size = r.shape
    x = gemm2_permuted
    _req(x.dtype == torch.bfloat16 and x.is_contiguous() and x.numel() == cap * top_k * hid_size,
         "gemm2_permuted must be contiguous BF16 [capacity * top_k, hidden]")
    dev = r.device
    _req(dev.type == "cuda" and x.device == dev and w.device == dev,
         "all tensors must be on the same CUDA device")
    for wt, eps in ((post_weight, post_eps), (next_weight, next_eps)):
        if wt is not None:
            _req(eps is not None, "a norm weight requires its eps")
            _req(wt.shape == (hid_size,) and wt.is_contiguous() and wt.dtype == torch.bfloat16
                 and wt.device == dev, "norm weights must be contiguous BF16 [hidden]")
    if hidden is None:
        hidden = torch.empty_like(r)
    if normalized is None and next_eps is not None:
        normalized = torch.empty_like(r)
    for o in (hidden, normalized):
        if o is not None:
            _req(o.shape == r.shape and o.dtype == torch.bfloat16 and o.is_contiguous() and
                 o.device == dev, "outputs must be contiguous BF16 like residual")
    s0, s1 = scales if scales is not None else (1.0, 1.0)
    st = _on_device(dev, lib().beam_moe_finalize_norm_residual_norm,
                    x.data_ptr(), cap, w.data_ptr(), cap, r.data_ptr(), tokens, top_k, hid_size,
                    float(routed_scale), None if post_weight is None else post_weight.data_ptr(),
                    float(post_eps or 0.0), int(post_eps is not None),
                    None if next_weight is None else next_weight.data_ptr(),
                    float(next_eps or 0.0), int(next_eps is not None), float(s0), float(s1),
                    hidden.data_ptr(), None if normalized is None else normalized.data_ptr(),
                    _stream_ptr(stream, dev))
    check(st, "beam_moe_finalize_norm_residual_norm")
    return hidden, normalized


def select_finalize_variant(num_tokens: int, hidden: int = HIDDEN, top_k: int = TOP_K) -> str:
    """Kernel the automatic choice runs for these sizes."""
    return VARIANT_NAMES[lib().mf_select_finalize_variant(int(num_tokens), int(hidden),
                                                          int(top_k))]


def select_beam_variant(live_tokens: int, top_k: int, hidden: int) -> str:
    return VARIANT_NAMES[lib().mf_select_beam_variant(int(live_tokens), int(top_k), int(hidden))]


def finalize_kernel_name(num_tokens: int, hidden: int = HIDDEN, top_k: int = TOP_K,
                         variant: str = "auto") -> str:
    """Name of the CUDA kernel a moe_finalize_rmsnorm call of these sizes launches
    on the current device ("" if none would)."""
    return lib().mf_finalize_kernel_name(int(num_tokens), int(hidden), int(top_k),
                                         _variant(variant)).decode()


def beam_kernel_name(live_tokens: int, top_k: int, hidden: int, variant: str = "auto",
                     residual: bool = False) -> str:
    """Name of the CUDA kernel a beam_moe_finalize call (or, with ``residual``,
    beam_moe_finalize_norm_residual_norm) of these sizes launches."""
    return lib().mf_beam_kernel_name(int(live_tokens), int(top_k), int(hidden), _variant(variant),
                                     int(bool(residual))).decode()


def device_status(clear: bool = True) -> int:
    """Synchronise the current device and return its status word as a status
    code (0, or 7 = MF_ERR_DEVICE_TIMEOUT if a bounded wait gave up)."""
    return int(lib().mf_device_status(int(bool(clear))))


def selftest_wait_timeout(timeout_ns: int = 10_000_000,
                          stream: torch.cuda.Stream | None = None) -> None:
    """Launch the failure-detection self-test (a wait that must give up)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    check(lib().mf_selftest_wait_timeout(int(timeout_ns), _stream_ptr(stream, dev)),
          "mf_selftest_wait_timeout")


def set_programmatic_launch(enable: bool) -> None:
    """Turn programmatic dependent launch on or off for later calls (default on)."""
    lib().mf_set_programmatic_launch(int(bool(enable)))


def programmatic_launch() -> bool:
    return bool(lib().mf_get_programmatic_launch())


def version() -> int:
    return int(lib().mf_version())
