"""Miss rate of the gate shortcut against the FP32 gate on the rollback-stress
workload (B=1 H=8 S=32768 D=128, N(0,1) with 1% of the keys after position
16384 scaled by 8), computed with the oracle on a sample of query rows.

A miss is a (row, tile) where the FP32 gate fires and the shortcut does not,
counted at the first decision that differs in each row (after it the two
runs carry different references).  Prints one JSON line.

  python oracle/gate_shortcut_study.py [--rows N] [--theta T]
"""
import argparse
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import fsa_inputs  # noqa: E402
import oracle  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=1024)
    ap.add_argument("--theta", type=float, default=8.0)
    args = ap.parse_args()
    B, H, S, D = 1, 8, 32768, 128
    q, k, v = fsa_inputs.qkv(B, H, S, D, seed=0, stress_from=16384)
    rng = np.random.default_rng(2024)
    rows = np.sort(rng.choice(B * H * S, size=args.rows, replace=False)).astype(np.int64)
    exact = oracle.attention(q, k, v, fmt=None, mode="exact", rows=rows)["out"]
    res = {}
    for fmt in ("mxfp8", "mxfp6", "mxfp4"):
        f = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=args.theta, rows=rows,
                             want_bits=True, want_margins=True)
        s = oracle.attention(q, k, v, fmt=fmt, mode="fused", threshold=args.theta, rows=rows,
                             want_bits=True, gate="shortcut")
        misses, spurious, band = 0, 0, []
        for r in range(len(rows)):
            diff = np.nonzero(f["bits"][r] != s["bits"][r])[0]
            if len(diff) == 0:
                continue
            t = diff[0]
            if f["bits"][r, t]:
                misses += 1
                band.append(float(f["margins"][r, t] + args.theta))
            else:
                spurious += 1
        fires = int(f["bits"].sum())
        res[fmt] = {
            "fp32_gate_firings": fires,
            "shortcut_firings": int(s["bits"].sum()),
            "rows_with_a_miss": misses,
            "rows_with_a_spurious_firing": spurious,
            "miss_rate_per_fp32_firing": misses / fires if fires else 0.0,
            "missed_excess_range": [min(band), max(band)] if band else None,
            "rel_l2_shortcut_vs_fp32_gate": oracle.rel_l2(s["out"], f["out"]),
            "rel_l2_vs_exact_fp32_gate": oracle.rel_l2(f["out"], exact),
            "rel_l2_vs_exact_shortcut": oracle.rel_l2(s["out"], exact),
        }
    print(json.dumps({"workload": "rollback-stress B=1 H=8 S=32768 D=128", "theta": args.theta,
                      "sampled_rows": int(len(rows)), "formats": res}))


if __name__ == "__main__":
    main()
