"""Parity at the full workload sizes, in the launch configuration bench.py times (MoELayer, same calls).

All index outputs are compared in full (router ids and counts, dispatch offsets, permutation, drop mask, send
layout); router floats in full; the dispatched payload on sampled rows; y on sampled tokens that the oracle
computes one by one (every expert those tokens reach runs the oracle's float64 SwiGLU)."""
import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O
from tests import cases

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_SAMPLE = 48


def _expert_fn(cfg, seed=0, shared=False):
    cache = {}

    def f(e):
        if e not in cache:
            cache.clear()                          # keep at most one decoded expert in host memory
            wg, wu, wd = moe_inputs.expert_weights(cfg, e, seed, shared=shared)
            cache[e] = tuple(moe_inputs.to_f64(w, cfg.dtype) for w in (wg, wu, wd))
        return cache[e]
    return f


@pytest.mark.parametrize("name", moe_inputs.CONFIG_ORDER)
def test_full_size_layer(name):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    from top_routing_dispatch_moe_gb300.layer import MoELayer
    cfg = moe_inputs.get_config(name)
    inp = cases.router_inputs(cfg)
    assert inp["near_ties"] == 0
    r = inp["route"]
    C = O.capacity(cfg.cf, cfg.k, cfg.T, cfg.E)
    d = O.dispatch(r["ids"], cfg.E, C, cfg.R)

    dev = torch.device("cuda")
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    up = lambda a: cases.to_device(a, cfg, dev)   # noqa: E731
    shared = None
    if cfg.n_shared:
        shared = tuple(up(np.ascontiguousarray(a[0])[None]) for a in moe_inputs.all_expert_weights(cfg, shared=True))
    layer = MoELayer(T=cfg.T, h=cfg.h, E=cfg.E, k=cfg.k, F=cfg.F, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                     alpha=cfg.alpha, w_r=up(inp["w_r"]),
                     bias=torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None,
                     w_gate=up(wg), w_up=up(wu), w_down=up(wd), shared=shared, device=dev)
    del wg, wu, wd, shared
    x = up(inp["x"])
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()

    # router: indices exact, floats within 1e-5
    ro = {k: v.cpu().numpy() for k, v in layer.r_out.items()}
    np.testing.assert_array_equal(ro["topk_ids"], r["ids"])
    np.testing.assert_array_equal(ro["counts"], r["counts"])
    assert cases.rel_max(ro["logits"], r["logits"]) <= 1e-5
    assert cases.rel_max(ro["gates"], r["gates"]) <= 1e-5
    assert cases.rel_max(ro["P"], r["P"]) <= 1e-5
    assert abs(float(ro["aux"][0]) - r["aux"]) <= 1e-5 * abs(r["aux"])

    # dispatch: every index output exact
    do = {k: v.cpu().numpy() for k, v in layer.d_out.items() if k != "buf"}
    for key in ["offsets", "kept_counts", "dest_row", "src_token", "src_slot", "rank_counts", "rank_offsets"]:
        np.testing.assert_array_equal(do[key], d[key], err_msg=key)
    np.testing.assert_array_equal(do["drop_mask"].astype(bool), d["drop_mask"])

    rng = np.random.default_rng(123)
    # payload: sampled rows bit-exact (pad rows zero)
    rows = rng.choice(d["rows"], size=min(256, d["rows"]), replace=False)
    got_rows = cases.from_device(layer.d_out["buf"][torch.from_numpy(rows).to(dev)], cfg)
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    want = np.where((d["src_token"][rows] >= 0)[:, None], x64[np.maximum(d["src_token"][rows], 0)], 0.0)
    np.testing.assert_array_equal(got_rows, want)

    # y: sampled tokens through the oracle one by one
    toks = np.sort(rng.choice(cfg.T, size=N_SAMPLE, replace=False))
    sh = _expert_fn(cfg, shared=True) if cfg.n_shared else None
    y_ref = O.moe_layer_tokens(toks, x64, r, d, _expert_fn(cfg), shared=(lambda: sh(0)) if sh else None)
    y_got = cases.from_device(y[torch.from_numpy(toks).to(dev)], cfg)
    fn, tol = cases.y_tolerance(cfg)
    err = fn(y_got, y_ref)
    assert err <= tol, f"{name}: sampled y error {err:.3e} > {tol}"
    for i in range(N_SAMPLE):
        if np.linalg.norm(y_ref[i]) > 0:
            assert fn(y_got[i], y_ref[i]) <= 4 * tol, f"token {toks[i]}"
