"""The oracle still produces the outputs frozen in tests/golden/ (CPU only)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "oracle_regression.json")


def test_oracle_regression_fixture():
    with open(GOLDEN) as f:
        doc = json.load(f)
    assert len(doc["cases"]) == 7
    for case in doc["cases"]:
        want = np.array(case["output"], dtype=np.uint16)
        if case["op"] == "tp":
            w = np.array(case["weights"], dtype=np.uint32 if case["weights_dtype"] == "fp32"
                         else np.uint16)
            if case["weights_dtype"] == "fp32":
                w = w.view(np.float32)
            got = oracle.moe_finalize_rmsnorm(
                np.array(case["gemm2"], dtype=np.uint16), w,
                np.array(case["idx"], dtype=np.int32),
                np.array(case["norm_weight"], dtype=np.uint16), eps=case["eps"],
                gain_center=case["gain_center"], weight_before_norm=case["weight_before_norm"],
                hidden=case["hidden"])
        else:
            pw = case["post_weight"]
            got = oracle.beam_moe_finalize(
                np.array(case["expert_outputs"], dtype=np.uint16),
                np.array(case["weights"], dtype=np.uint32).view(np.float32),
                case["live_tokens"], routed_scale=case["routed_scale"],
                post_weight=None if pw is None else np.array(pw, dtype=np.uint16),
                post_eps=case["post_eps"])
        assert np.array_equal(got, want), case["op"]
