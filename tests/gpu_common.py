"""Helpers shared by the GPU parity tests: device/host BF16 transfers and one
call of each operation through the library (with canary rows after the
output) or through the oracle.  No finalize arithmetic here."""
import numpy as np
import torch

import oracle

CANARY = 0x1234


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_tp(mf, case, variant, *, before=None, stream=None):
    before = case.weight_before_norm if before is None else before
    T, H = case.num_tokens, case.hidden
    g = dev_bf16(case.gemm2)[:, :H] if case.gemm2.size else \
        torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    w = dev_bf16(case.weights) if case.weights.dtype == np.uint16 else \
        torch.from_numpy(case.weights).cuda()
    idx = torch.from_numpy(case.idx).cuda()
    nw = dev_bf16(case.norm_weight)
    buf = torch.full((T + 2, H), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    out = buf[:T]
    mf.moe_finalize_rmsnorm(g, w, idx, nw, out, eps=case.eps, gain_center=case.gain_center,
                            weight_before_norm=before, variant=variant, stream=stream)
    torch.cuda.synchronize()
    got = host_bits(buf)
    assert np.all(got[T:] == CANARY), "output canary overwritten"
    return got[:T]


def oracle_tp(case, before=None):
    before = case.weight_before_norm if before is None else before
    return oracle.moe_finalize_rmsnorm(case.gemm2, case.weights, case.idx, case.norm_weight,
                                       eps=case.eps, gain_center=case.gain_center,
                                       weight_before_norm=before, hidden=case.hidden)


def run_beam(mf, case, variant, live=None):
    live = case.live_tokens if live is None else live
    cap, K, H = case.expert_outputs.shape
    x = dev_bf16(case.expert_outputs)
    w = torch.from_numpy(case.weights).cuda()
    pw = dev_bf16(case.post_weight) if case.post_weight is not None else None
    buf = torch.full((live + 2, H), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    out = buf[:live]
    r = mf.beam_moe_finalize(x, w, out, case.routed_scale, pw, case.post_eps, variant=variant)
    assert r.data_ptr() == out.data_ptr()
    torch.cuda.synchronize()
    got = host_bits(buf)
    assert np.all(got[live:] == CANARY), "output canary overwritten"
    return got[:live]


def oracle_beam(case, live=None):
    live = case.live_tokens if live is None else live
    return oracle.beam_moe_finalize(case.expert_outputs, case.weights, live,
                                    routed_scale=case.routed_scale, post_weight=case.post_weight,
                                    post_eps=case.post_eps)
