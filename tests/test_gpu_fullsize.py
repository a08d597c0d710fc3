"""Parity at the full workload sizes, in the launch configuration bench.py times (MoELayer, same calls).

Everything is compared in full: the router's indices and floats, every dispatch index output, the dispatched
payload bit for bit (pad rows zero), and y of every token against the oracle's float64 layer, which runs one
expert at a time on that expert's tokens (one expert's decoded weights in host memory at a time): normwise within
the bf16 / fp32 tolerance, and every token's row within 4x it."""
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
    # the separate combine (the configuration bench.py times); the fused one is checked bitwise against it below
    fused = False
    layer = MoELayer(T=cfg.T, h=cfg.h, E=cfg.E, k=cfg.k, F=cfg.F, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                     alpha=cfg.alpha, w_r=up(inp["w_r"]),
                     bias=torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None,
                     w_gate=up(wg), w_up=up(wu), w_down=up(wd), shared=shared, device=dev, fuse_combine=fused)
    del wg, wu, wd, shared
    x = up(inp["x"])
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    if cfg.dtype == "bf16":   # the down GEMM with the combine in its epilogue: the same eout and y bits
        dd = layer.d_out
        arr = moe.moe_combine_arrivals(cfg.T, cfg.h, dev)
        sh = bool(cfg.n_shared)
        eout_f, sh_f, y_f = moe.moe_expert_down_combine(
            layer.act, dd["tile_sched"], layer.packed, cfg.E, cfg.h, dd["src_token"], dd["dest_row"],
            layer.r_out["gates"], arr, act_shared=layer.sh_act if sh else None,
            packed_shared=layer.shared_packed if sh else None)
        torch.cuda.synchronize()
        assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
        assert torch.equal(y_f.view(torch.int16), y.view(torch.int16)), f"{name}: fused combine differs"
        live = dd["src_token"] >= 0
        assert torch.equal(eout_f[live].view(torch.int16), layer.eout[live].view(torch.int16))
        if sh:
            assert torch.equal(sh_f.view(torch.int16), layer.sh_out.view(torch.int16))
        assert int(arr.abs().sum().item()) == 0
        del eout_f, sh_f, y_f, arr

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

    # payload: every row bit-exact (a kept row is its token's row of x, a pad row is zero)
    src = d["src_token"]
    if cfg.dtype == "bf16":
        got_bits = layer.d_out["buf"].view(torch.int16).cpu().numpy().view(np.uint16)
        want_bits = np.where((src >= 0)[:, None], np.asarray(inp["x"])[np.maximum(src, 0)], np.uint16(0))
    else:
        got_bits = layer.d_out["buf"].cpu().numpy().view(np.uint32)
        want_bits = np.where((src >= 0)[:, None], np.asarray(inp["x"], np.float32).view(np.uint32)[np.maximum(src, 0)],
                             np.uint32(0))
    np.testing.assert_array_equal(got_bits, want_bits)
    del got_bits, want_bits

    # y: every token through the oracle, one expert at a time
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    sh = _expert_fn(cfg, shared=True) if cfg.n_shared else None
    y_ref = O.moe_layer_tokens(np.arange(cfg.T), x64, r, d, _expert_fn(cfg), shared=(lambda: sh(0)) if sh else None)
    y_got = cases.from_device(y, cfg)
    assert np.isfinite(y_got).all()
    fn, tol = cases.y_tolerance(cfg)
    err = fn(y_got, y_ref)
    assert err <= tol, f"{name}: y error {err:.3e} > {tol}"
    norms = np.linalg.norm(y_ref, axis=1)
    row_err = np.linalg.norm(y_got - y_ref, axis=1) / np.where(norms > 0, norms, 1.0)
    if cfg.dtype == "f32":
        row_err = np.max(np.abs(y_got - y_ref), axis=1) / np.maximum(np.max(np.abs(y_ref), axis=1), 1e-300)
    live = norms > 0
    assert (row_err[live] <= 4 * tol).all(), f"{name}: worst token {int(np.argmax(np.where(live, row_err, 0)))}"
    assert not y_got[~live].any(), f"{name}: a token with every pair dropped has a non-zero y"


BWD_WORKLOADS = ["page3_cf1.25", "mixtral_zipf", "deepseek_v3", "qwen3_moe"]


@pytest.mark.parametrize("name", BWD_WORKLOADS)
def test_full_size_backward(name):
    """MoELayer.backward at the full workload size, from a forward that kept the pre-activations (the
    configuration bench.py times), each backward call against the oracle on the GPU's own inputs to it:
    combine backward (d_gates on sampled tokens), router backward (d_logits in full, d_bias), the router
    weight gradient on sampled entries, the expert backward of the active expert with the fewest rows in full
    (d_act, d_g / d_u, d_buf, fp32 weight gradients, oracle SwiGLU backward) and dx on sampled tokens."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    from top_routing_dispatch_moe_gb300.layer import MoELayer
    cfg = moe_inputs.get_config(name)
    bias = moe_inputs.load_zipf_bias(cfg) if cfg.bias == "zipf" else None
    inp = cases.router_inputs(cfg, bias=bias)
    assert inp["near_ties"] == 0
    dev = torch.device("cuda")
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    up = lambda a: cases.to_device(a, cfg, dev)   # noqa: E731
    shared = None
    if cfg.n_shared:
        shared = tuple(up(np.ascontiguousarray(a[0])[None]) for a in moe_inputs.all_expert_weights(cfg, shared=True))
    layer = MoELayer(T=cfg.T, h=cfg.h, E=cfg.E, k=cfg.k, F=cfg.F, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                     alpha=cfg.alpha, w_r=up(inp["w_r"]),
                     bias=torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None,
                     w_gate=up(wg), w_up=up(wu), w_down=up(wd), shared=shared, device=dev, backward=True)
    del wg, wu, wd, shared
    x = up(inp["x"])
    layer.forward(x, save=True)
    rng = np.random.default_rng(321)
    dy = torch.from_numpy(rng.normal(size=(cfg.T, cfg.h)).astype(np.float32)).to(dev).to(x.dtype)
    d_aux = 0.7
    g = layer.backward(x, dy, d_aux=d_aux)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    f64 = lambda t: t.detach().double().cpu().numpy()   # noqa: E731
    b, r, d = layer._bwd, layer.r_out, layer.d_out
    dest = d["dest_row"].cpu().numpy()
    toks = np.sort(rng.choice(cfg.T, size=N_SAMPLE, replace=False))

    # combine backward: d_gates of sampled tokens
    dst = dest[toks]                                          # [N, k], -1 for dropped pairs
    rows_t = torch.from_numpy(np.maximum(dst, 0).reshape(-1)).to(dev)
    eout_s = f64(layer.eout[rows_t]).reshape(len(toks), cfg.k, cfg.h)
    dy_s = f64(dy[torch.from_numpy(toks).to(dev)])
    want = np.where(dst >= 0, np.einsum("nkh,nh->nk", eout_s, dy_s), 0.0)
    assert cases.rel_max(f64(b["d_gates"])[toks], want) <= 1e-5

    # router backward in full
    rr = dict(ids=r["topk_ids"].cpu().numpy().astype(np.int64), gates=f64(r["gates"]), f=f64(r["f"]))
    dl_ref = O.route_backward(f64(r["logits"]), rr, f64(b["d_gates"]), cfg.gating, cfg.alpha, d_aux)
    assert cases.rel_max(f64(b["d_logits"]), dl_ref) <= 1e-5
    if g["d_bias"] is not None:
        assert cases.rel_max(f64(g["d_bias"]), dl_ref.sum(axis=0)) <= 1e-5

    # router weight gradient: 256 sampled entries of x^T d_logits
    x64, dl = moe_inputs.to_f64(inp["x"], cfg.dtype), f64(b["d_logits"])
    ii, ee = rng.integers(0, cfg.h, 256), rng.integers(0, cfg.E, 256)
    want = np.einsum("ts,ts->s", x64[:, ii], dl[:, ee])
    got = f64(g["dW_r"])[ii, ee]
    assert np.max(np.abs(got - want)) <= 1e-5 * np.max(np.abs(want))

    # the active expert with the fewest rows, in full
    off, kept = d["offsets"].cpu().numpy(), d["kept_counts"].cpu().numpy()
    e = int(np.argmin(np.where(kept > 0, kept, np.iinfo(np.int32).max)))
    a0, a1 = int(off[e]), int(off[e]) + int(kept[e])
    wge, wue, wde = (moe_inputs.to_f64(w, cfg.dtype) for w in moe_inputs.expert_weights(cfg, e, 0))
    ref = O.swiglu_ffn_backward(f64(d["buf"][a0:a1]), wge, wue, wde, f64(b["d_eout"][a0:a1]))
    Fp = (cfg.F + 127) // 128 * 128
    gu = f64(b["d_gu"][a0:a1]).reshape(a1 - a0, Fp // 128, 2, 128)
    checks = [("d_act", f64(b["d_act"][a0:a1]), ref["d_a"]),
              ("d_g", gu[:, :, 0, :].reshape(a1 - a0, Fp)[:, :cfg.F], ref["dG"]),
              ("d_u", gu[:, :, 1, :].reshape(a1 - a0, Fp)[:, :cfg.F], ref["dU"]),
              ("d_buf", f64(b["d_buf"][a0:a1]), ref["dX"]),
              ("dW_gate", f64(g["dW_gate"][e]), ref["dW_gate"]), ("dW_up", f64(g["dW_up"][e]), ref["dW_up"]),
              ("dW_down", f64(g["dW_down"][e]), ref["dW_down"])]
    for what, got, want in checks:
        assert cases.rel_l2(got, want) <= 2e-2, f"{name} expert {e} ({a1 - a0} rows): {what}"

    # dx on sampled tokens: extra (shared expert) + kept d_buf rows + d_logits W_r^T
    w_r64 = moe_inputs.to_f64(inp["w_r"], cfg.dtype)
    dbuf_s = f64(b["d_buf"][rows_t]).reshape(len(toks), cfg.k, cfg.h)
    want = dl[toks] @ w_r64.T + np.einsum("nkh,nk->nh", dbuf_s, (dst >= 0).astype(np.float64))
    if cfg.n_shared:
        want += f64(b["sh_dx"][torch.from_numpy(toks).to(dev)])
    got = f64(g["dx"][torch.from_numpy(toks).to(dev)])
    assert cases.rel_l2(got, want) <= 4e-3, name
