"""CPU oracle for the MoE finalize (+ RMSNorm) path and its Beam variant.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``moe_finalize_rmsnorm_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``moe_finalize_oracle.c`` (plain C, one element at a
time); this module builds it with gcc and marshals numpy arrays into it.
Every function follows the pages:

* ``moe_finalize_rmsnorm`` -- flashinfer.comm.tp_moe_finalize_rmsnorm
  (API page: description and parameter list).
* ``beam_moe_finalize`` -- vllm.models.beam.nvidia.moe_finalize,
  beam_moe_finalize (docstring and source).
* ``beam_moe_finalize_norm_residual_norm`` -- vllm.models.beam.nvidia.
  moe_finalize, beam_moe_finalize_norm_residual_norm: Beam finalize, then the
  residual step of its unfused reference.  PARTLY UNPINNED: the residual step
  (beam_norm_residual_norm) is not on the pages; it is read as
  hidden = BF16(s0 x + s1 residual) in FP32 and normalized = BF16(RMSNorm(hidden)).
* ``bf16_from_double`` -- the BF16 format itself (upper half of binary32),
  round-to-nearest-even.

All BF16 tensors are passed as ``numpy.uint16`` bit patterns.

Parity of the oracle with the pages' own kernels is unpinned (the pages ship
no kernels or numbers); the oracle itself is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_finalize_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# A prebuilt oracle library to load instead (the mutation tests point this at a
# copy of the oracle with one planted mistake, to check that the pins catch it).
_OVERRIDE = os.environ.get("MF_ORACLE_SO")
if _OVERRIDE:
    _LIB = _OVERRIDE
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA, no shared code with the GPU path)."""
    if _OVERRIDE:
        return _LIB
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, i64, i32, f32, c_int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_float, ctypes.c_int)
            lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_moe_finalize_rmsnorm.argtypes = [
                vp, i64, i64, vp, c_int, vp, vp, vp, i64, i32, i32, f32, f32, c_int]
            lib.oracle_moe_finalize_rmsnorm.restype = c_int
            lib.oracle_beam_moe_finalize.argtypes = [
                vp, vp, vp, i64, i32, i32, f32, vp, f32, c_int]
            lib.oracle_beam_moe_finalize.restype = c_int
            lib.oracle_beam_moe_finalize_norm_residual_norm.argtypes = [
                vp, vp, vp, i64, i32, i32, f32, vp, f32, c_int, vp, f32, c_int, f32, f32, vp, vp]
            lib.oracle_beam_moe_finalize_norm_residual_norm.restype = c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def bf16_from_double(x: float) -> int:
    """BF16 bit pattern of x rounded to nearest, ties to even (NaN -> 0x7FC0)."""
    return int(_load().oracle_bf16_from_double(float(x)))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits)))


def moe_finalize_rmsnorm(gemm2: np.ndarray, weights: np.ndarray, idx: np.ndarray,
                         norm_weight: np.ndarray, *, eps: float, gain_center: float,
                         weight_before_norm: bool, hidden: int | None = None,
                         out: np.ndarray | None = None) -> np.ndarray:
    """Oracle of tp_moe_finalize_rmsnorm.

    gemm2: uint16 [rows, row_stride] (BF16 bits; the first ``hidden`` columns
    are live, default all).  weights [T, top_k]: float32, uint16 (BF16 bits),
    or int32 packed routing words ``(expert_id << 16) | bf16 bits`` (the
    topk_ids format of trtllm_fp8_per_tensor_scale_routed_moe).  idx: int32 [T, top_k].  norm_weight: uint16 [hidden].
    Returns uint16 [T, hidden].
    """
    assert gemm2.dtype == np.uint16 and gemm2.ndim == 2
    assert idx.dtype == np.int32 and idx.ndim == 2 and weights.shape == idx.shape
    assert weights.dtype in (np.float32, np.uint16, np.int32)
    rows, row_stride = gemm2.shape
    hidden = row_stride if hidden is None else int(hidden)
    assert 0 < hidden <= row_stride and norm_weight.shape == (hidden,)
    t, k = idx.shape
    if out is None:
        out = np.empty((t, hidden), dtype=np.uint16)
    assert out.shape == (t, hidden) and out.dtype == np.uint16
    rc = _load().oracle_moe_finalize_rmsnorm(
        _ptr(gemm2), rows, row_stride, _ptr(weights),
        {np.dtype(np.uint16): 0, np.dtype(np.float32): 1, np.dtype(np.int32): 2}[weights.dtype],
        _ptr(idx), _ptr(norm_weight), _ptr(out), t, hidden, k, float(eps),
        float(gain_center), int(bool(weight_before_norm)))
    if rc != 0:
        raise MemoryError("oracle could not allocate its row buffers")
    return out


def beam_moe_finalize(expert_outputs: np.ndarray, weights: np.ndarray, live_tokens: int, *,
                      routed_scale: float = 1.0, post_weight: np.ndarray | None = None,
                      post_eps: float | None = None,
                      out: np.ndarray | None = None) -> np.ndarray:
    """Oracle of beam_moe_finalize.

    expert_outputs: uint16 [capacity, top_k, hidden] (BF16 bits).  weights:
    float32 [>= live_tokens, top_k].  post_weight: uint16 [hidden] or None.
    post_eps None means no normalisation.  Returns uint16 [live_tokens, hidden].
    """
    assert expert_outputs.dtype == np.uint16 and expert_outputs.ndim == 3
    cap, k, hidden = expert_outputs.shape
    assert weights.dtype == np.float32 and weights.ndim == 2 and weights.shape[1] == k
    assert 0 <= live_tokens <= cap and weights.shape[0] >= live_tokens
    if post_weight is not None:
        assert post_eps is not None and post_weight.shape == (hidden,)
        assert post_weight.dtype == np.uint16
    if out is None:
        out = np.empty((live_tokens, hidden), dtype=np.uint16)
    assert out.shape[0] >= live_tokens and out.shape[1] == hidden
    if live_tokens == 0:
        return out
    rc = _load().oracle_beam_moe_finalize(
        _ptr(expert_outputs), _ptr(weights), _ptr(out), live_tokens, k, hidden,
        float(routed_scale), _ptr(post_weight), float(post_eps or 0.0),
        int(post_eps is not None))
    if rc != 0:
        raise MemoryError("oracle could not allocate its row buffers")
    return out


def beam_moe_finalize_norm_residual_norm(
        expert_outputs: np.ndarray, weights: np.ndarray, residual: np.ndarray, *,
        routed_scale: float = 1.0, post_weight: np.ndarray | None = None,
        post_eps: float | None = None, next_weight: np.ndarray | None = None,
        next_eps: float | None = None,
        scales: tuple[float, float] | None = None) -> tuple[np.ndarray, np.ndarray | None]:
    """Oracle of beam_moe_finalize_norm_residual_norm (partly unpinned).

    expert_outputs: uint16 [capacity, top_k, hidden]; weights: float32
    [>= tokens, top_k]; residual: uint16 [tokens, hidden] (tokens = live rows).
    Returns (hidden, normalized); normalized is None without next_eps.
    """
    assert expert_outputs.dtype == np.uint16 and expert_outputs.ndim == 3
    cap, k, hidden = expert_outputs.shape
    assert residual.dtype == np.uint16 and residual.ndim == 2 and residual.shape[1] == hidden
    tokens = residual.shape[0]
    assert tokens <= cap and weights.dtype == np.float32 and weights.shape[0] >= tokens
    for w, e in ((post_weight, post_eps), (next_weight, next_eps)):
        if w is not None:
            assert e is not None and w.shape == (hidden,) and w.dtype == np.uint16
    s0, s1 = scales if scales is not None else (1.0, 1.0)
    hid = np.empty((tokens, hidden), dtype=np.uint16)
    norm = np.empty((tokens, hidden), dtype=np.uint16) if next_eps is not None else None
    if tokens == 0:
        return hid, norm
    rc = _load().oracle_beam_moe_finalize_norm_residual_norm(
        _ptr(expert_outputs), _ptr(weights), _ptr(residual), tokens, k, hidden,
        float(routed_scale), _ptr(post_weight), float(post_eps or 0.0), int(post_eps is not None),
        _ptr(next_weight), float(next_eps or 0.0), int(next_eps is not None), float(s0),
        float(s1), _ptr(hid), _ptr(norm))
    if rc != 0:
        raise MemoryError("oracle could not allocate its row buffers")
    return hid, norm
