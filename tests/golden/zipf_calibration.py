"""Calibration of the correction-bias strength beta of the Zipf(1.1) batched-decode
workload (test infrastructure; writes tests/golden/zipf_beta.json).

The workload asks for expert popularity following Zipf(s = 1.1) through the correction
bias, the page's own steering mechanism (the bias changes which experts are selected,
never their weights).  synth.zipf_bias sets bias_e = beta ln(p_e / p_max) + U(-0.1, 0.1)
with p_e ~ rank_e^-1.1 over a seeded ranking of the experts.  This script routes seeded
synthetic tokens through the oracle's router with that bias for a range of beta, fits the
slope of log(selection count) against log(rank) over ranks 17..256 (an expert is picked at
most once per token, so the 16 most popular saturate; the far tail is sparse), and keeps
the beta whose slope is -1.1 (linear interpolation between the bracketing grid points).

    python tests/golden/zipf_calibration.py     # about a minute on 16 cores
"""
import dataclasses
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402
import synth  # noqa: E402

TOKENS = 4096
RANK_LO, RANK_HI = 17, 256


def slope(cfg, beta, x, wr):
    c = dataclasses.replace(cfg, zipf_beta=beta)
    bias = synth.zipf_bias(c, 0, 0)
    idx, _, _, _ = oracle.router(x, wr, bias, cfg.topk, nthreads=oracle.num_threads())
    counts = np.bincount(idx.ravel(), minlength=cfg.n_experts).astype(np.float64)
    rank = synth.zipf_ranks(c, 0, 0)
    order = np.argsort(rank)[RANK_LO - 1:RANK_HI]
    keep = counts[order] > 0
    lr = np.log(rank[order][keep].astype(np.float64))
    lc = np.log(counts[order][keep])
    return float(np.polyfit(lr, lc, 1)[0]), int((counts > 0).sum())


def main():
    cfg = synth.config("decode64_zipf")
    wr = synth.layer_weights(cfg, 0)["wr"]
    x = synth.activations(cfg, 1000, TOKENS)
    grid = [0.05, 0.075, 0.1, 0.125, 0.15, 0.2, 0.25, 0.3]
    res = [(b,) + slope(cfg, b, x, wr) for b in grid]
    for b, s, u in res:
        print("beta %.4f  slope %+.3f  experts used %d" % (b, s, u))
    target = -cfg.zipf_s
    beta = None
    for (b0, s0, _), (b1, s1, _) in zip(res, res[1:]):
        if (s0 - target) * (s1 - target) <= 0:
            beta = b0 + (target - s0) * (b1 - b0) / (s1 - s0)
            break
    if beta is None:
        raise SystemExit("slope -1.1 not bracketed by the grid")
    beta = round(beta, 4)
    out = {"beta": beta, "zipf_s": cfg.zipf_s, "tokens": TOKENS, "token_seed": 1000,
           "fit_ranks": [RANK_LO, RANK_HI], "grid": [[b, s, u] for b, s, u in res]}
    json.dump(out, open(os.path.join(HERE, "zipf_beta.json"), "w"), indent=1)
    print("beta =", beta)


if __name__ == "__main__":
    main()
