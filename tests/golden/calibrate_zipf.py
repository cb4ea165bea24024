"""Derive the Zipf bias strength of the skewed chunk (writes tests/golden/zipf_alpha.json).

The skewed chunk adds bias_e = -alpha * 1.1 * ln(rank_e) to the router logits (rank_e a seeded permutation of
1..E) so that the 32 most-routed experts take about half of the routed pairs.  alpha is found by bisection on
[0, 4] with the ORACLE's routing only; the synthetic-input module then carries the figure as a constant.

    python tests/golden/calibrate_zipf.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from quantized_routed_expert_smoe_gb300 import synth  # noqa: E402


def top32_share(alpha: float) -> float:
    cfg = synth.CONFIGS["skew8192"]
    inp = synth.make_layer(cfg, zipf_alpha=alpha, with_weights=False)
    ids, _ = oracle.route(inp["logits"], cfg.K)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    return float(np.sort(counts)[::-1][:32].sum() / ids.size)


def main():
    lo, hi = 0.0, 4.0
    for _ in range(20):
        mid = 0.5 * (lo + hi)
        if top32_share(mid) < 0.5:
            lo = mid
        else:
            hi = mid
    alpha = 0.5 * (lo + hi)
    share = top32_share(alpha)
    out = dict(alpha=alpha, top32_share=share, target=0.5, config="skew8192", zipf_s=synth.ZIPF_S,
               script="tests/golden/calibrate_zipf.py")
    with open(os.path.join(ROOT, "tests", "golden", "zipf_alpha.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
