"""Writes directp_thresholds.json by calling only the oracle.

The thresholds T_k are the smallest FP32 x with RNE_E2M1(6*2^x) >= the k-th
non-negative E2M1 magnitude (Direct-P, "Direct Mapping" in the technical
summary of "Hardware-Aware FP4 FlashAttention-4").  The test suite re-derives
them from the closed form log2(midpoint/6) independently.
"""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402

T = oracle.directp_thresholds()
out = {
    "source": "oracle.directp_thresholds(); Direct-P map RNE_E2M1(6*2^x), c*(s-m) = x",
    "T_fp32": [float(t) for t in T],
    "T_hex": [t.tobytes()[::-1].hex() for t in T],
}
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "directp_thresholds.json"), "w") as f:
    json.dump(out, f, indent=1)
    f.write("\n")
