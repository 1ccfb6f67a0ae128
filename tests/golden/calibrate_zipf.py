"""Recompute the router-bias strengths ``synth.ZIPF_KAPPA``.

For a Zipf exponent s, bisect kappa in b_e = -kappa * s * ln(rank_e + 1) so
that the log-log slope of "tokens that picked the expert of rank r" against r
(over ranks picked by fewer than half of the tokens, and at least once) is -s.
Workload: layer 0 of seed 0, H=2048, E=512, k=10, 4,096 tokens, router weights
N(0, 0.02) and activations N(0, 1) drawn from ``bit_expert_ffn_gb300.synth``.

The selection here is a plain numpy argpartition on fp64 logits: this script
shapes an input distribution and is not a parity reference.

Run:  python tests/golden/calibrate_zipf.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", ".."))
from bit_expert_ffn_gb300 import synth  # noqa: E402

H, E, K, T = 2048, 512, 10, 4096


def realised_slope(logits0, rank, kappa, s):
    b = -kappa * s * np.log(rank + 1.0)
    top = np.argpartition(-(logits0 + b), K, axis=1)[:, :K]
    cnt = np.bincount(top.ravel(), minlength=E)
    by_rank = cnt[np.argsort(rank)]
    r = np.arange(1, E + 1)
    m = (by_rank < 0.5 * T) & (by_rank > 0)
    return np.polyfit(np.log(r[m]), np.log(by_rank[m]), 1)[0]


def setup(seed=0, layer=0):
    w = synth.router_weights(seed, layer, E, H).astype(np.float64)
    x = synth.bf16_bits_to_f32(synth.activations(seed, T, H, step=1000)).astype(np.float64)
    return x @ w.T, synth.zipf_rank(seed, layer, E)


def calibrate(s, logits0, rank):
    lo, hi = 0.0, 5.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if realised_slope(logits0, rank, mid, s) > -s:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


if __name__ == "__main__":
    logits0, rank = setup()
    for s in (1.1, 1.4):
        k = calibrate(s, logits0, rank)
        print(f"s={s}: kappa={k:.4f} slope={realised_slope(logits0, rank, k, s):.4f}")
