"""Write tests/golden/oracle_regression.json: small inputs and the oracle's
outputs for them, so that any later change to the oracle's arithmetic shows
up as a failing test (and has to be justified).

Calls only ``oracle``; the inputs are written out in full, so the fixture does
not depend on the random generator's version.  Run from the repo root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def f32_bits_to_bf16(a):
    u = a.astype(np.float32).view(np.uint32).copy()
    u += ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return (u >> 16).astype(np.uint16)


def main():
    rng = np.random.default_rng(2024)
    cases = []
    for before in (False, True):
        for wdt in ("fp32", "bf16"):
            T, K, H, stride, R = 3, 8, 32, 40, 20
            gemm2 = f32_bits_to_bf16(rng.standard_normal((R, stride)) * 2)
            gemm2[:, H:] = 0x7FC0
            idx = rng.integers(-2, R + 2, size=(T, K)).astype(np.int32)
            w = rng.random((T, K)).astype(np.float32)
            if wdt == "bf16":
                w = f32_bits_to_bf16(w)
            nw = f32_bits_to_bf16(0.1 * rng.standard_normal(H))
            out = oracle.moe_finalize_rmsnorm(gemm2, w, idx, nw, eps=1e-5, gain_center=1.0,
                                              weight_before_norm=before, hidden=H)
            cases.append(dict(op="tp", hidden=H, eps=1e-5, gain_center=1.0,
                              weight_before_norm=before, weights_dtype=wdt,
                              gemm2=gemm2.tolist(), idx=idx.tolist(),
                              weights=(w.view(np.uint32) if wdt == "fp32" else w).tolist(),
                              norm_weight=nw.tolist(), output=out.tolist()))
    for has_norm, pw_on in ((False, False), (True, False), (True, True)):
        cap, K, H, live = 4, 3, 256, 3
        x = f32_bits_to_bf16(rng.standard_normal((cap, K, H)))
        w = rng.random((cap, K)).astype(np.float32)
        pw = f32_bits_to_bf16(1 + 0.05 * rng.standard_normal(H)) if pw_on else None
        eps = 1e-6 if has_norm else None
        out = oracle.beam_moe_finalize(x, w, live, routed_scale=2.5, post_weight=pw,
                                       post_eps=eps)
        cases.append(dict(op="beam", live_tokens=live, routed_scale=2.5, post_eps=eps,
                          expert_outputs=x.tolist(), weights=w.view(np.uint32).tolist(),
                          post_weight=None if pw is None else pw.tolist(),
                          output=out.tolist()))
    doc = dict(
        source="tests/golden/make_golden.py (calls only the oracle)",
        note="BF16 tensors are uint16 bit patterns; fp32 weights are uint32 bit patterns",
        cites=["flashinfer.comm.tp_moe_finalize_rmsnorm (API page)",
               "vllm.models.beam.nvidia.moe_finalize, beam_moe_finalize"],
        cases=cases)
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(doc, f, separators=(",", ":"))


if __name__ == "__main__":
    main()
