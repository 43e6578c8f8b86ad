"""Write tests/golden/zipf_beta.json: the scale beta of the Zipf expert bias of
the long-prefill workload.

bias[e] = beta * ln(rank_e ** -1.1), rank a seeded permutation of 1..E.  beta is
chosen by bisection so that, under the oracle's own routing of the workload's
seeded hidden states, the most popular expert receives 10x the mean number of
token copies (S / E): a literal Zipf(1.1) share for the top expert would exceed
the cap of one copy per token, so the skew is matched on the max/mean ratio.
Calls only the oracle and the input generator.
"""
import json
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def max_over_mean(logits, w, beta):
    bias = W.zipf_bias(w, beta)
    r = oracle.route_sigmoid(logits, bias, w.top_k, w.route_scale)
    counts, _ = oracle.histogram_offsets(r["idx"], w.E)
    return counts.max() / (w.S / w.E), int((counts == 0).sum())


def main():
    w = W.WORKLOADS["zipf"]
    hidden = W.normal_bf16(w.seed, W.TID_HIDDEN, (w.T, w.H), w.hidden_sigma)
    router_w = W.normal_f32(w.seed, W.TID_ROUTER_W, (w.E, w.H), w.router_sigma)
    logits = oracle.router_logits(hidden, router_w)
    lo, hi = 0.0, 2.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        ratio, _ = max_over_mean(logits, w, mid)
        if ratio < 10.0:
            lo = mid
        else:
            hi = mid
    beta = round(hi, 6)
    ratio, empty = max_over_mean(logits, w, beta)
    key = f"{w.name}:T{w.T}:E{w.E}:seed{w.seed}"
    out = {"note": __doc__.strip().splitlines()[0], "target_max_over_mean": 10.0,
           "beta": {key: beta}, "achieved": {key: {"max_over_mean": round(float(ratio), 4),
                                                    "experts_without_tokens": empty}}}
    path = Path(__file__).with_name("zipf_beta.json")
    path.write_text(json.dumps(out, indent=2) + "\n")
    print(path, out)


if __name__ == "__main__":
    main()
