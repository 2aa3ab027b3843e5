"""Host-side checks of the C ABI (CPU only: nothing here reaches a kernel).

Every call below breaks exactly one rule of the contract in
include/moe_finalize.h, so validation rejects it before any CUDA call; the
pointers are fake (never dereferenced).
"""
import ctypes
import glob
import os
import re

import pytest

from moe_finalize_rmsnorm_gb300 import _abi
from moe_finalize_rmsnorm_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, NULL, SHAPE, ALIGN, DTYPE, UNSUP, CUDA, TIMEOUT, INVALID = range(9)

A = 0x10000          # a fake 16-byte-aligned address (never dereferenced)
MIS = 0x10008        # a fake 8-byte-but-not-16-byte-aligned address


@pytest.fixture(scope="module")
def lib():
    build()
    return _abi.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    assert {"moe_finalize_rmsnorm", "beam_moe_finalize", "mf_status_string",
            "mf_device_status"} <= names
    assert names == set(_abi.SIGNATURES), names ^ set(_abi.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_programmatic_launch_switch(lib):
    assert lib.mf_get_programmatic_launch() == 1          # on by default
    lib.mf_set_programmatic_launch(0)
    assert lib.mf_get_programmatic_launch() == 0
    lib.mf_set_programmatic_launch(5)
    assert lib.mf_get_programmatic_launch() == 1


def test_status_strings(lib):
    for code in range(9):
        assert lib.mf_status_string(code)
    assert lib.mf_status_string(0) == b"ok"
    assert lib.mf_version() >= 100


def tp(lib, gemm2=A, rows=100, stride=4096, w=A, wdt=1, idx=A, nw=A, out=A, T=4, H=4096, K=8,
       variant=0):
    return lib.moe_finalize_rmsnorm_variant(gemm2, rows, stride, w, wdt, idx, nw, out, T, H, K,
                                            1e-6, 1.0, 0, variant, None)


def test_tp_validation(lib):
    # sizes: 4096 / 8 (specialised) or hidden 256..8192 step 256, top_k 1..32
    assert tp(lib, H=128) == UNSUP
    assert tp(lib, H=8448) == UNSUP
    assert tp(lib, H=4000) == UNSUP
    assert tp(lib, K=0) == UNSUP
    assert tp(lib, K=33) == UNSUP
    assert tp(lib, K=4, variant=1) == INVALID     # register kernel only for 4096 / 8
    assert tp(lib, H=2048, variant=3) == INVALID  # cluster kernel only for 4096 / 8
    assert tp(lib, H=2048, stride=2044) == SHAPE
    assert tp(lib, stride=4095) == SHAPE          # shorter than hidden
    assert tp(lib, stride=4100) == SHAPE          # not a multiple of 8
    assert tp(lib, T=-1) == SHAPE
    assert tp(lib, rows=-1) == SHAPE
    assert tp(lib, wdt=3) == DTYPE
    assert tp(lib, variant=9) == INVALID
    assert tp(lib, gemm2=None) == NULL
    assert tp(lib, w=None) == NULL
    assert tp(lib, idx=None) == NULL
    assert tp(lib, nw=None) == NULL
    assert tp(lib, out=None) == NULL
    for kw in ("gemm2", "w", "idx", "nw", "out"):
        assert tp(lib, **{kw: MIS}) == ALIGN, kw
    # zero tokens: a no-op, whatever the pointers
    assert tp(lib, gemm2=None, w=None, idx=None, nw=None, out=None, T=0) == OK


def beam(lib, x=A, cap=10, w=A, wrows=10, out=A, live=5, K=8, H=7168, scale=2.5, pw=A, eps=1e-6,
         norm=1, variant=0):
    return lib.beam_moe_finalize_variant(x, cap, w, wrows, out, live, K, H, scale, pw, eps, norm,
                                         variant, None)


def test_beam_validation(lib):
    assert beam(lib, K=0) == UNSUP
    assert beam(lib, K=33) == UNSUP
    assert beam(lib, H=128) == UNSUP
    assert beam(lib, H=8448) == UNSUP
    assert beam(lib, H=4000) == UNSUP              # not a multiple of 256
    assert beam(lib, live=11) == SHAPE             # more live rows than capacity
    assert beam(lib, live=-1) == SHAPE
    assert beam(lib, wrows=4) == SHAPE             # fewer weight rows than live rows
    assert beam(lib, norm=0) == INVALID            # post_weight without post_eps
    assert beam(lib, variant=3) == INVALID         # no cluster variant for Beam
    assert beam(lib, x=None) == NULL
    assert beam(lib, w=None) == NULL
    assert beam(lib, out=None) == NULL
    assert beam(lib, x=MIS) == ALIGN
    assert beam(lib, out=MIS) == ALIGN
    assert beam(lib, pw=MIS) == ALIGN
    assert beam(lib, w=A + 2) == ALIGN             # FP32 weights need 4-byte alignment
    assert beam(lib, x=None, w=None, out=None, live=0) == OK


def test_binding_rejects_bad_tensors_before_the_library():
    torch = pytest.importorskip("torch")
    import moe_finalize_rmsnorm_gb300 as mf
    g = torch.zeros(16, 4096, dtype=torch.bfloat16)
    w = torch.zeros(2, 8)
    idx = torch.zeros(2, 8, dtype=torch.int32)
    nw = torch.zeros(4096, dtype=torch.bfloat16)
    out = torch.zeros(2, 4096, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        mf.moe_finalize_rmsnorm(g, w, idx, nw, out, eps=1e-6, gain_center=1.0,
                                weight_before_norm=False)
    with pytest.raises(ValueError, match="int32"):
        mf.moe_finalize_rmsnorm(g, w, idx.long(), nw, out, eps=1e-6, gain_center=1.0,
                                weight_before_norm=False)
    with pytest.raises(ValueError, match="variant"):
        mf._variant("fastest")
    x = torch.zeros(4, 8, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        mf.beam_moe_finalize(x, torch.zeros(4, 8), torch.zeros(4, 256, dtype=torch.bfloat16),
                             post_weight=torch.ones(256, dtype=torch.bfloat16), post_eps=1e-6)
    with pytest.raises(ValueError, match="FP32"):
        mf.beam_moe_finalize(x, torch.zeros(4, 8).double(),
                             torch.zeros(4, 256, dtype=torch.bfloat16))


def test_status_error_carries_the_code(lib):
    e = _abi.MoeFinalizeError(SHAPE, "where")
    assert e.status == SHAPE and "MF_ERR_SHAPE" in str(e)
    with pytest.raises(_abi.MoeFinalizeError):
        _abi.check(ALIGN, "x")


def test_ctypes_signatures_match_header_arity():
    # every declared parameter list has as many entries as the ctypes table
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "moe_finalize.h")).read(),
                  flags=re.S)
    for name, (_, args) in _abi.SIGNATURES.items():
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(args), (name, len(params), len(args))
    assert ctypes.sizeof(ctypes.c_void_p) == 8


def resid(lib, x=A, cap=10, w=A, wrows=10, r=A, T=5, K=8, H=7168, pw=A, pn=1, nw=A, nn=1,
          hid=A, nrm=A):
    return lib.beam_moe_finalize_norm_residual_norm(x, cap, w, wrows, r, T, K, H, 2.5, pw, 1e-6,
                                                    pn, nw, 1e-6, nn, 1.0, 1.0, hid, nrm, None)


def test_residual_norm_validation(lib):
    assert resid(lib, K=33) == UNSUP
    assert resid(lib, H=300) == UNSUP
    assert resid(lib, T=11) == SHAPE               # more tokens than capacity
    assert resid(lib, wrows=4) == SHAPE
    assert resid(lib, pn=0) == INVALID             # post_weight without its eps
    assert resid(lib, nn=0) == INVALID             # next_weight without its eps
    assert resid(lib, nw=None, nn=0) == INVALID    # normalized output without the next norm
    assert resid(lib, r=None) == NULL
    assert resid(lib, hid=None) == NULL
    assert resid(lib, nrm=None) == NULL            # next norm without its output
    assert resid(lib, r=MIS) == ALIGN
    assert resid(lib, nrm=MIS) == ALIGN
    assert resid(lib, nw=MIS) == ALIGN
    assert resid(lib, x=None, w=None, r=None, hid=None, nrm=None, T=0) == OK


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # the product path has no CPU fallback: without the built library every
    # entry point raises instead of computing anything
    import torch
    import moe_finalize_rmsnorm_gb300 as mf
    from moe_finalize_rmsnorm_gb300 import _abi
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB", str(tmp_path / "libmoe_finalize.so"))
    with pytest.raises(ImportError, match="no CPU fallback"):
        _abi.lib()
    with pytest.raises(ImportError):
        mf.select_finalize_variant(32768)
    g = torch.zeros((16, 4096), dtype=torch.bfloat16)
    with pytest.raises((ImportError, ValueError, RuntimeError)):
        mf.moe_finalize_rmsnorm(g, torch.ones((2, 8)), torch.zeros((2, 8), dtype=torch.int32),
                                torch.ones(4096, dtype=torch.bfloat16),
                                torch.empty((2, 4096), dtype=torch.bfloat16),
                                eps=1e-6, gain_center=0.0, weight_before_norm=False)


def _no_library_call():
    raise AssertionError("the binding reached the library before rejecting its arguments")


def test_binding_rejects_normalized_without_next_eps(monkeypatch):
    # the C ABI returns MF_ERR_INVALID for a normalized output without the next
    # norm; the binding raises for the same combination before calling it
    import torch
    import moe_finalize_rmsnorm_gb300 as mf
    monkeypatch.setattr(mf, "lib", _no_library_call)
    x = torch.zeros((4 * 2, 256), dtype=torch.bfloat16)
    w = torch.ones((4, 2))
    r = torch.zeros((3, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="next_eps"):
        mf.beam_moe_finalize_norm_residual_norm(x, w, r, None, None, None, None, None,
                                                normalized=torch.empty_like(r))


def test_binding_rejects_gemm2_narrower_than_hidden(monkeypatch):
    # a narrowed view keeps the parent's row stride: without the column check the
    # row-stride rule alone would let the kernel read columns outside the view
    import torch
    import moe_finalize_rmsnorm_gb300 as mf
    monkeypatch.setattr(mf, "lib", _no_library_call)
    g = torch.zeros((16, 4096), dtype=torch.bfloat16)[:, :2048]
    assert g.stride(0) == 4096
    with pytest.raises(ValueError, match="fewer columns"):
        mf.moe_finalize_rmsnorm(g, torch.ones((2, 8)), torch.zeros((2, 8), dtype=torch.int32),
                                torch.ones(4096, dtype=torch.bfloat16),
                                torch.empty((2, 4096), dtype=torch.bfloat16),
                                eps=1e-6, gain_center=0.0, weight_before_norm=False)


def test_kernel_names_without_a_device(lib):
    # the launch a call would make, by size and variant; without a device the
    # wave tests of the automatic choice are skipped
    name = lambda *a: lib.mf_finalize_kernel_name(*a).decode()
    assert name(1, 4096, 8, 0) == name(8, 4096, 8, 3) == "tp_cluster_kernel"
    assert name(16, 4096, 8, 0) == name(9, 4096, 8, 1) == "tp_token_cta_kernel"
    assert name(5000, 4096, 8, 2) in ("tp_token_bulk_kernel", "tp_token_bulk_multi_kernel")
    assert name(100, 512, 32, 0) == "tp_warp_bulk_kernel"
    assert name(100, 1280, 8, 2) == "tp_generic_bulk_kernel"
    assert name(0, 4096, 8, 0) == name(5, 300, 8, 0) == name(5, 512, 8, 1) == ""
    beam = lambda *a: lib.mf_beam_kernel_name(*a).decode()
    assert beam(10, 8, 7168, 0, 0) == beam(10, 8, 7168, 1, 1) == "beam_token_bulk_kernel"
    assert beam(10, 8, 7168, 1, 0) == "beam_token_cta_kernel"
    assert beam(10, 8, 512, 0, 0) == "beam_warp_bulk_kernel"
    assert beam(0, 8, 512, 0, 0) == beam(10, 33, 512, 0, 0) == ""


def test_data_movement_validation(lib):
    # the measurement aid takes the finalize's operands at hidden 4096 / top_k 8
    def dm(gemm2=A, rows=100, stride=4096, w=A, wdt=1, idx=A, out=A, T=5):
        return lib.mf_finalize_data_movement(gemm2, rows, stride, w, wdt, idx, out, T, None)
    assert dm(stride=4095) == SHAPE
    assert dm(stride=4100) == SHAPE
    assert dm(T=-1) == SHAPE
    assert dm(rows=-1) == SHAPE
    assert dm(T=1 << 31) == SHAPE
    assert dm(wdt=3) == DTYPE
    for kw in ("gemm2", "w", "idx", "out"):
        assert dm(**{kw: None}) == NULL, kw
        assert dm(**{kw: MIS}) == ALIGN, kw
    assert dm(gemm2=None, w=None, idx=None, out=None, T=0) == OK


def test_binding_data_movement_covers_4096_by_8_only(monkeypatch):
    import torch
    import moe_finalize_rmsnorm_gb300 as mf
    monkeypatch.setattr(mf, "lib", _no_library_call)
    g = torch.zeros((16, 2048), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="hidden 4096"):
        mf.finalize_data_movement(g, torch.ones((2, 8)), torch.zeros((2, 8), dtype=torch.int32),
                                  torch.empty((2, 2048), dtype=torch.bfloat16))
