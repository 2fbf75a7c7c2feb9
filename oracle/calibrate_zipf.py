"""Pick the strength of the routing-skew component of the V3-shaped inputs.

TEST INFRASTRUCTURE (runs the oracle only). For each candidate alpha it
draws the V3-shaped router weights and tokens (seed 0), routes them with the
oracle at bias 0, sorts the raw expert loads in descending order and fits a
line to log(load) against log(pair rank) over the top 16 ranks: the 16
experts the skew component is aligned with come in 8 pairs that share one
direction, so ranks 2j+1 and 2j+2 both have pair rank j+1. The smallest
alpha past which the slope stops steepening (it levels off above -1.1) is
the one stored as ZIPF_ALPHA in the input module.

    python -m oracle.calibrate_zipf [--tokens 4096]
"""
import argparse

import numpy as np

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om


def load_slope(counts, top=16):
    c = np.sort(np.asarray(counts, np.float64))[::-1][:top]
    r = (np.arange(top, dtype=np.float64) // 2) + 1
    return float(np.polyfit(np.log(r), np.log(np.maximum(c, 1.0)), 1)[0])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--alphas", type=str, default="1,2,3,4,5,6,8")
    args = ap.parse_args()
    p = synth.PRESETS["v3_t16384_d7168_e256_bf16"].replace(T=args.tokens)
    wr = synth._normal((p.E, p.d), synth.INIT_STD, p.seed, 1, "cpu", synth.torch_dtype(p.dtype))
    for a in [float(v) for v in args.alphas.split(",")]:
        x = synth.make_x(p, wr, alpha=a).float().numpy()
        s = om.router_scores(x, wr.float().numpy())
        idx, _ = om.select_experts(s, np.zeros(p.E, np.float32), p.G, p.K, p.M)
        c = om.expert_counts(idx, p.E)
        print(f"alpha={a:4.2f} slope={load_slope(c):+.3f} max/mean={om.load_max_over_mean(c, p.T, p.K):.2f}")


if __name__ == "__main__":
    main()
