"""Writes the stored per-expert router logit bias of the Mixtral-shaped workload (Zipf(1) expert load).

Run: python oracle/calibrate_zipf_bias.py    (writes moe_inputs/mixtral_zipf_router_bias.json)

Target assignment share of expert e: p_e = (1/(e+1)) / sum_j 1/(j+1). Start from b = ln p, then iterate
b <- b + ln(p / share(b)), where share(b) is the fraction of the k*T assignments that the oracle's router
gives each expert with the bias added to its logits, until every share is within 1% (relative) of p.
Only the oracle computes here; the result is an input of that workload, not an expected value.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import moe_inputs  # noqa: E402
from oracle import moe_oracle as O  # noqa: E402


def calibrate(cfg, seed=0, tol=0.01, max_iter=30):
    x = moe_inputs.to_f64(moe_inputs.make_x(cfg, seed), cfg.dtype)
    w_r, _ = moe_inputs.make_router(cfg, seed, bias=np.zeros(cfg.E, np.float32))
    L0 = x @ moe_inputs.to_f64(w_r, cfg.dtype)
    p = 1.0 / np.arange(1, cfg.E + 1)
    p /= p.sum()
    b = np.log(p)
    b -= b[0]
    for it in range(max_iter):
        b32 = b.astype(np.float32).astype(np.float64)        # the bias is stored in float32
        r = O.route(L0 + b32[None, :], cfg.k, cfg.gating)
        share = r["counts"] / float(cfg.k * cfg.T)
        err = np.max(np.abs(share / p - 1.0))
        print(f"iter {it}: max rel err {err:.4f} shares {np.round(share, 4).tolist()}")
        if err < tol:
            return b.astype(np.float32), share, err, it
        b = b + np.log(p / np.maximum(share, 1e-9))
        b -= b[0]
    raise RuntimeError("Zipf calibration did not converge")


def main():
    cfg = moe_inputs.get_config("mixtral_zipf")
    seed = 0
    b, share, err, it = calibrate(cfg, seed)
    path = moe_inputs.ZIPF_BIAS_FILE
    data = json.load(open(path)) if os.path.exists(path) else {}
    key = f"{cfg.name}/T{cfg.T}/h{cfg.h}/E{cfg.E}/k{cfg.k}/seed{seed}"
    data[key] = dict(bias=[float(v) for v in b], shares=[float(v) for v in share], max_rel_err=float(err),
                     iterations=it, script="oracle/calibrate_zipf_bias.py")
    with open(path, "w") as fh:
        json.dump(data, fh, indent=1)
    print("wrote", path, key, [round(float(v), 4) for v in b])


if __name__ == "__main__":
    main()
