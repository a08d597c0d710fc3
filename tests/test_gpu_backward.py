"""GPU backward against the oracle's backward, element by element, on the same inputs.

The forward runs on the GPU (router, dispatch, experts, combine); each backward call is then given the GPU's
own forward results and checked against the oracle's backward function fed the same values (converted to
float64): combine (d_eout, d_gates), router (d_logits, d_bias, through every gating mode, with the aux term),
router weight (dW_r), dispatch (dx with the router term and an extra input gradient), and the expert FFN
(d_act, d_g / d_u, d_buf, fp32 weight gradients) per expert against the oracle's SwiGLU backward.

Tolerances: fp32 results max-rel 1e-5 (fp32 sums against float64); outputs rounded to bf16 within half a bf16
ulp of the reference's own value (rtol 2^-8) where they are one product, and normwise 4e-3 / max-rel 1e-2 where
they are sums rounded once; the expert backward, whose intermediates (act, d_act, d_g / d_u) are bf16, normwise
2e-2 like the layer output.
"""
import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O
from tests import cases

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_fp32": ("tiny_fp32", dict(T=300, cf=0.75), None),                       # softmax, capacity drops
    "page3_small": ("page3_cf1.25", dict(T=300, h=256, F=128), None),             # softmax, capacity
    "mixtral_small": ("mixtral_zipf", dict(T=400, h=256, F=128), "zipf"),         # renormalised, logit bias
    "deepseek_small": ("deepseek_v3", dict(T=200, h=256, F=128, E=64, k=6, n_shared=0), None),   # sigmoid + bias
    # E = 256: the router-weight products on the tensor cores with T = 1000 padded to 1024 and split over K
    "deepseek_wide": ("deepseek_v3", dict(T=1000, h=1024, F=128, E=256, k=8, n_shared=0), None),
}
_cache = {}


def _forward(name):
    if name in _cache:
        return _cache[name]
    import torch
    base, over, bias_kind = CASES[name]
    cfg = moe_inputs.get_config(base, **over)
    bias = moe_inputs.load_zipf_bias(moe_inputs.get_config("mixtral_zipf")) if bias_kind == "zipf" else None
    inp = cases.router_inputs(cfg, bias=bias)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    x = cases.to_device(inp["x"], cfg)
    layer.forward(x)
    rng = np.random.default_rng(11)
    dt = x.dtype
    dy = torch.from_numpy(rng.normal(size=(cfg.T, cfg.h)).astype(np.float32)).to("cuda").to(dt)
    torch.cuda.synchronize()
    _cache[name] = (cfg, inp, layer, x, dy)
    return _cache[name]


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _combine(name):
    from top_routing_dispatch_moe_gb300 import moe
    cfg, inp, layer, x, dy = _forward(name)
    r, d = layer.r_out, layer.d_out
    d_eout, d_gates = moe.moe_combine_backward(dy, layer.eout, d["src_token"], d["src_slot"], d["dest_row"], r["gates"])
    # pad rows of eout are never written by the GEMMs (and never read by combine): converted as zeros
    eout64 = cases.from_device_rows(layer.eout, d["src_token"] >= 0, cfg)
    ref_eout, ref_gates = O.combine_backward(_np(dy), eout64, d["dest_row"].cpu().numpy(), _np(r["gates"]),
                                             layer.rows)
    return cfg, d_eout, d_gates, ref_eout, ref_gates


@pytest.mark.parametrize("name", list(CASES))
def test_combine_backward(name):
    import torch
    cfg, d_eout, d_gates, ref_eout, ref_gates = _combine(name)
    torch.cuda.synchronize()
    rtol = 2.0 ** -8 if cfg.dtype == "bf16" else 1e-6
    np.testing.assert_allclose(_np(d_eout), ref_eout, rtol=rtol, atol=1e-30)
    assert cases.rel_max(_np(d_gates), ref_gates) <= 1e-5


@pytest.mark.parametrize("name", list(CASES))
def test_router_backward_and_weight_grad(name):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg, inp, layer, x, dy = _forward(name)
    _, _, d_gates, _, _ = _combine(name)
    r = layer.r_out
    alpha, d_aux = cfg.alpha, 0.7
    d_logits, d_bias = moe.moe_router_backward(r["logits"], r["topk_ids"], r["gates"], d_gates, r["f"], cfg.gating,
                                               alpha, d_aux)
    dW_r = moe.moe_router_weight_grad(x, d_logits)
    torch.cuda.synchronize()
    rr = dict(ids=r["topk_ids"].cpu().numpy().astype(np.int64), gates=_np(r["gates"]), f=_np(r["f"]))
    ref = O.route_backward(_np(r["logits"]), rr, _np(d_gates), cfg.gating, alpha, d_aux)
    assert cases.rel_max(_np(d_logits), ref) <= 1e-5
    assert cases.rel_max(_np(d_bias), ref.sum(axis=0)) <= 1e-5
    ref_w = moe_inputs.to_f64(inp["x"], cfg.dtype).T @ _np(d_logits)
    assert cases.rel_max(_np(dW_r), ref_w) <= 1e-5


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_backward(name):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg, inp, layer, x, dy = _forward(name)
    d = layer.d_out
    rng = np.random.default_rng(12)
    dt = x.dtype
    d_buf = torch.from_numpy(rng.normal(size=(layer.rows, cfg.h)).astype(np.float32)).to("cuda").to(dt)
    extra = torch.from_numpy(rng.normal(size=(cfg.T, cfg.h)).astype(np.float32)).to("cuda").to(dt)
    d_logits = torch.from_numpy(rng.normal(size=(cfg.T, cfg.E)).astype(np.float32)).to("cuda")
    dx = moe.moe_dispatch_backward(d_buf, d["dest_row"], d_logits, layer.w_r, dx_extra=extra)
    dx_plain = moe.moe_dispatch_backward(d_buf, d["dest_row"], None, layer.w_r)
    torch.cuda.synchronize()
    dest = d["dest_row"].cpu().numpy()
    db = _np(d_buf)
    plain = np.zeros((cfg.T, cfg.h))
    for j in range(cfg.k):
        kept = dest[:, j] >= 0
        plain[kept] += db[dest[kept, j]]
    ref = _np(extra) + plain + _np(d_logits) @ moe_inputs.to_f64(inp["w_r"], cfg.dtype).T
    if cfg.dtype == "bf16":
        assert cases.rel_l2(_np(dx), ref) <= 4e-3 and cases.rel_max(_np(dx), ref) <= 1e-2
        assert cases.rel_l2(_np(dx_plain), plain) <= 4e-3
    else:
        assert cases.rel_max(_np(dx), ref) <= 1e-5 and cases.rel_max(_np(dx_plain), plain) <= 1e-5


@pytest.mark.parametrize("saved", [False, True])
@pytest.mark.parametrize("sizes", [[0, 1, 127, 129, 300], [0, 257, 1900, 40]])
def test_expert_backward(sizes, saved):
    """Expert FFN backward per expert against the oracle's SwiGLU backward on the same bf16 operands: d_act,
    the packed d_g / d_u, d_buf and the fp32 weight gradients (zero for an expert without rows). F = 320 leaves a
    zero-padded part of the last 128-column block. The second size list has rows >= 512 E, so the dgrad GEMMs run
    on the 2-SM kernel; the weight gradients (M = 2 Fp = 768 and h = 256 output rows per expert) run on the
    2-SM kernel with its fp32 TMA-store epilogue. saved: the forward keeps g and u
    (moe_expert_up_gate_save: act bit-identical to moe_expert_up_gate, g and u within bf16 rounding of the
    float64 products) and the backward starts from them (moe_expert_up_gate_backward_saved)."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(7)
    dev = "cuda"
    E, h, F = len(sizes), 256, 320
    Fp = (F + 127) // 128 * 128
    ids = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(3).shuffle(ids)
    x = torch.randn(ids.size, h, device=dev).to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids[:, None]).to(dev), E, 0, 1)
    mk = lambda *s: (torch.randn(*s, device=dev) / s[-1] ** 0.5).to(torch.bfloat16)
    wg, wu, wd = mk(E, F, h), mk(E, F, h), mk(E, h, F)
    packed = moe.moe_pack_expert_weights(wg, wu, wd)
    packed_bwd = moe.moe_pack_expert_weights_backward(wg, wu, wd)
    buf, sched = d["buf"], d["tile_sched"]
    act = moe.moe_expert_up_gate(buf, sched, packed, E, F)
    d_eout = torch.randn(buf.shape[0], h, device=dev).to(torch.bfloat16)
    d_act = moe.moe_expert_down_backward(d_eout, sched, packed_bwd, E, F)
    if saved:
        act_s, gu_s, _, _ = moe.moe_expert_up_gate_save(buf, sched, packed, E, F)
        d_gu, d_buf = moe.moe_expert_up_gate_backward_saved(gu_s, d_act, sched, packed_bwd, E, h)
    else:
        d_gu, d_buf = moe.moe_expert_up_gate_backward(buf, d_act, sched, packed, packed_bwd, E)
    dWg, dWu, dWd = moe.moe_expert_weight_grads(buf, act, d_gu, d_eout, d["offsets"], d["kept_counts"], E)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    off = d["offsets"].cpu().tolist()
    f64 = lambda t: t.double().cpu().numpy()
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            assert not dWg[e].any() and not dWu[e].any() and not dWd[e].any()
            continue
        if saved:
            assert torch.equal(act_s[a:b], act[a:b])
            pre = f64(gu_s[a:b]).reshape(b - a, Fp // 128, 2, 128)
            for got, w in [(pre[:, :, 0, :].reshape(b - a, Fp), wg[e]), (pre[:, :, 1, :].reshape(b - a, Fp), wu[e])]:
                assert np.all(got[:, F:] == 0)
                assert cases.rel_l2(got[:, :F], f64(buf[a:b]) @ f64(w).T) <= 4e-3
        g = O.swiglu_ffn_backward(f64(buf[a:b]), f64(wg[e]), f64(wu[e]), f64(wd[e]), f64(d_eout[a:b]))
        gu = f64(d_gu[a:b]).reshape(b - a, Fp // 128, 2, 128)
        dG = gu[:, :, 0, :].reshape(b - a, Fp)
        dU = gu[:, :, 1, :].reshape(b - a, Fp)
        assert np.all(dG[:, F:] == 0) and np.all(dU[:, F:] == 0)
        for got, ref, what in [(f64(d_act[a:b]), g["d_a"], "d_act"), (dG[:, :F], g["dG"], "d_g"),
                               (dU[:, :F], g["dU"], "d_u"), (f64(d_buf[a:b]), g["dX"], "d_buf"),
                               (f64(dWg[e]), g["dW_gate"], "dW_gate"), (f64(dWu[e]), g["dW_up"], "dW_up"),
                               (f64(dWd[e]), g["dW_down"], "dW_down")]:
            assert cases.rel_l2(got, ref) <= 2e-2, f"expert {e} ({b - a} rows): {what} rel err {cases.rel_l2(got, ref):.3e}"


LAYER_CASES = {
    "page3_small": ("page3_cf1.25", dict(T=300, h=256, F=128), None),             # softmax, capacity drops
    "mixtral_small": ("mixtral_zipf", dict(T=400, h=256, F=128), "zipf"),         # renormalised, bias gradient
    "deepseek_small": ("deepseek_v3", dict(T=200, h=256, F=128, E=64, k=6), None),  # sigmoid + its shared expert
}


@pytest.mark.parametrize("save", [False, True])
@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_backward(name, save):
    """MoELayer.backward (every backward call in sequence) against the oracle's moe_layer_backward of its own
    float64 forward, for <dy, y> + d_aux * aux: dx, dW_r, d_bias, every expert's and the shared expert's weight
    gradients. The GPU's intermediates (eout, act, d_act, d_g / d_u, d_buf) are bf16: normwise 2e-2. save: the
    forward keeps the pre-activations and the backward starts from them (no up/gate recompute)."""
    import torch
    base, over, bias_kind = LAYER_CASES[name]
    cfg = moe_inputs.get_config(base, **over)
    bias = moe_inputs.load_zipf_bias(moe_inputs.get_config("mixtral_zipf")) if bias_kind == "zipf" else None
    inp = cases.router_inputs(cfg, bias=bias)
    assert inp["near_ties"] == 0
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    shared = tuple(a[0] for a in moe_inputs.all_expert_weights(cfg, shared=True)) if cfg.n_shared else None
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd, shared, backward=True)
    x = cases.to_device(inp["x"], cfg)
    layer.forward(x, save=save)
    rng = np.random.default_rng(13)
    dy = torch.from_numpy(rng.normal(size=(cfg.T, cfg.h)).astype(np.float32)).to("cuda").to(x.dtype)
    d_aux = 0.7
    g = layer.backward(x, dy, d_aux=d_aux)
    torch.cuda.synchronize()
    from top_routing_dispatch_moe_gb300 import moe
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()

    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    w_r64 = moe_inputs.to_f64(inp["w_r"], cfg.dtype)
    wfn = cases.weights_fn_from(cfg, wg, wu, wd)
    sfn = (lambda: tuple(moe_inputs.to_f64(w, cfg.dtype) for w in shared)) if shared else None
    fwd = O.moe_layer(x64, w_r64, inp["bias"], wfn, k=cfg.k, gating=cfg.gating, cf=cfg.cf, R=cfg.R, alpha=cfg.alpha,
                      shared=sfn)
    np.testing.assert_array_equal(layer.r_out["topk_ids"].cpu().numpy(), fwd["router"]["ids"])
    ref = O.moe_layer_backward(x64, w_r64, inp["bias"], wfn, fwd, _np(dy), gating=cfg.gating, alpha=cfg.alpha,
                               d_aux=d_aux, shared=sfn)
    checks = [("dx", _np(g["dx"]), ref["dx"]), ("dW_r", _np(g["dW_r"]), ref["dW_r"]),
              ("dW_gate", _np(g["dW_gate"]), np.stack([w[0] for w in ref["dW"]])),
              ("dW_up", _np(g["dW_up"]), np.stack([w[1] for w in ref["dW"]])),
              ("dW_down", _np(g["dW_down"]), np.stack([w[2] for w in ref["dW"]]))]
    if ref["d_bias"] is not None:
        checks.append(("d_bias", _np(g["d_bias"]), ref["d_bias"]))
    else:
        assert g["d_bias"] is None
    if shared:
        checks += [("shared_dW_gate", _np(g["shared_dW_gate"]), ref["shared"]["dW_gate"]),
                   ("shared_dW_up", _np(g["shared_dW_up"]), ref["shared"]["dW_up"]),
                   ("shared_dW_down", _np(g["shared_dW_down"]), ref["shared"]["dW_down"])]
    for what, got, want in checks:
        err = cases.rel_l2(got, want)
        assert err <= 2e-2, f"{what}: rel err {err:.3e}"


def test_layer_backward_sinkhorn():
    """Sinkhorn routing: the ids come from L + log c, the gates are softmax(L)[ids]; with the selection held
    constant the backward is the plain softmax one (the Zipf logit bias gets d_bias). Against the oracle's
    backward of its own Sinkhorn forward."""
    import torch
    cfg = moe_inputs.get_config("mixtral_sinkhorn", T=400, h=256, F=128)
    inp = cases.router_inputs(cfg, bias=moe_inputs.load_zipf_bias(moe_inputs.get_config("mixtral_zipf")))
    assert inp["near_ties"] == 0
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd, backward=True)
    x = cases.to_device(inp["x"], cfg)
    layer.forward(x)
    rng = np.random.default_rng(17)
    dy = torch.from_numpy(rng.normal(size=(cfg.T, cfg.h)).astype(np.float32)).to("cuda").to(x.dtype)
    g = layer.backward(x, dy, d_aux=0.7)
    torch.cuda.synchronize()
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    w_r64 = moe_inputs.to_f64(inp["w_r"], cfg.dtype)
    wfn = cases.weights_fn_from(cfg, wg, wu, wd)
    L = O.router_logits(x64, w_r64, inp["bias"], O.SOFTMAX)
    r = O.route_sinkhorn(L, cfg.k, alpha=cfg.alpha)
    np.testing.assert_array_equal(layer.r_out["topk_ids"].cpu().numpy(), r["ids"])
    d = O.dispatch(r["ids"], cfg.E, O.capacity(cfg.cf, cfg.k, cfg.T, cfg.E), cfg.R)
    buf = O.dispatch_payload(x64, d)
    eout = O.expert_outputs(buf, d, wfn)
    fwd = dict(router=r, dispatch=d, buf=buf, eout=eout)
    ref = O.moe_layer_backward(x64, w_r64, inp["bias"], wfn, fwd, _np(dy), gating=O.SOFTMAX_SELBIAS, alpha=cfg.alpha,
                               d_aux=0.7)
    for what, got, want in [("dx", _np(g["dx"]), ref["dx"]), ("dW_r", _np(g["dW_r"]), ref["dW_r"]),
                            ("d_bias", _np(g["d_bias"]), ref["d_bias"]),
                            ("dW_down", _np(g["dW_down"]), np.stack([w[2] for w in ref["dW"]]))]:
        err = cases.rel_l2(got, want)
        assert err <= 2e-2, f"{what}: rel err {err:.3e}"


@pytest.mark.parametrize("name", ["page3_small", "deepseek_small"])
def test_backward_deterministic(name):
    """Two backward passes over the same saved forward give bit-identical gradients (every reduction runs in a
    fixed order: no atomics in any accumulation, split-K parts and per-block partials added in order)."""
    import torch
    base, over, bias_kind = LAYER_CASES[name]
    cfg = moe_inputs.get_config(base, **over)
    inp = cases.router_inputs(cfg)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    shared = tuple(a[0] for a in moe_inputs.all_expert_weights(cfg, shared=True)) if cfg.n_shared else None
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd, shared, backward=True)
    x = cases.to_device(inp["x"], cfg)
    layer.forward(x, save=True)
    dy = torch.from_numpy(np.random.default_rng(17).normal(size=(cfg.T, cfg.h)).astype(np.float32)).cuda().to(x.dtype)
    first = {k: (v.clone() if v is not None else None) for k, v in layer.backward(x, dy, d_aux=0.3).items()}
    second = layer.backward(x, dy, d_aux=0.3)
    torch.cuda.synchronize()
    for k, v in first.items():
        if v is None:
            assert second[k] is None
            continue
        a, b = (v.view(torch.int16), second[k].view(torch.int16)) if v.dtype == torch.bfloat16 else (v, second[k])
        assert torch.equal(a, b), k
