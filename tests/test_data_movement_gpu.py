"""The data-movement measurement kernel (mf_finalize_data_movement) on GB300.

What it stores is the XOR of the 32-bit words it read (each valid row's words,
the weight's bits in the first word of every chunk), so a numpy XOR over the
same operands checks that it moves exactly the finalize's bytes: every valid
row, every weight, no invalid slot and no padding column.  No finalize
arithmetic is involved on either side.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import CANARY, dev_bf16, host_bits

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]

H = 4096


def _weight_bits(w: np.ndarray) -> np.ndarray:
    """The weight as the kernel holds it, as FP32 bits."""
    if w.dtype == np.float32:
        return w.view(np.uint32)
    if w.dtype == np.uint16:  # BF16
        return w.astype(np.uint32) << 16
    return (w.view(np.uint32) & 0xFFFF) << 16  # packed routing word: its low half


def expected_xor(case: si.TpCase) -> np.ndarray:
    rows = case.gemm2.shape[0]
    words = np.ascontiguousarray(case.gemm2[:, :H]).view(np.uint32).reshape(rows, H // 8, 4)
    valid = (case.idx >= 0) & (case.idx < rows)
    picked = words[np.where(valid, case.idx, 0)]                       # [T, K, 512, 4]
    picked = np.where(valid[:, :, None, None], picked, np.uint32(0))
    acc = np.bitwise_xor.reduce(picked, axis=1)                          # [T, 512, 4]
    wb = np.where(valid, _weight_bits(case.weights), np.uint32(0))
    acc[:, :, 0] ^= np.bitwise_xor.reduce(wb, axis=1)[:, None]
    return acc.view(np.uint16).reshape(case.num_tokens, H)


def run_data_movement(mf, case: si.TpCase) -> np.ndarray:
    T = case.num_tokens
    g = dev_bf16(case.gemm2)[:, :H]
    w = dev_bf16(case.weights) if case.weights.dtype == np.uint16 else \
        torch.from_numpy(case.weights).cuda()
    idx = torch.from_numpy(case.idx).cuda()
    buf = torch.full((T + 2, H), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    mf.finalize_data_movement(g, w, idx, buf[:T])
    torch.cuda.synchronize()
    assert mf.device_status(clear=True) == 0
    got = host_bits(buf)
    assert np.all(got[T:] == CANARY), "output canary overwritten"
    return got[:T]


@pytest.mark.parametrize("weights_dtype", ["fp32", "bf16", "packed"])
def test_data_movement_reads_exactly_the_finalize_operands(cuda_lib, weights_dtype):
    mf = cuda_lib
    case = si.tp_case("dm", 1000, indexed_rows=8000, padding_rows=200, row_stride=4160,
                      invalid_frac=0.05, weights_dtype=weights_dtype, poison_padding=True,
                      seed=71)
    np.testing.assert_array_equal(run_data_movement(mf, case), expected_xor(case))


def test_data_movement_zero_tokens_and_all_invalid(cuda_lib):
    mf = cuda_lib
    case = si.tp_case("dm0", 0, indexed_rows=64)
    assert run_data_movement(mf, case).shape == (0, H)
    case = si.tp_case("dm_invalid", 20, indexed_rows=200, seed=3)
    case.idx[:] = -1
    got = run_data_movement(mf, case)
    assert np.all(got == 0)
