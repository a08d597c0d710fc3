"""Sinkhorn routing on the GPU against the oracle: the Sinkhorn selection bias log c (1e-5), expert ids and
counts (bit-exact), gates (1e-5), the dispatch layout (bit-exact) and the layer output (tolerances of the
token-choice layer); reduced sizes and the Mixtral-shaped workload at full size on sampled tokens."""
import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O
from tests import cases

pytestmark = pytest.mark.gpu


def _zipf():
    return moe_inputs.load_zipf_bias(moe_inputs.get_config("mixtral_zipf"))


CASES = {
    "sk_mixtral_small": (dict(T=1500, h=256, F=512), True),
    "sk_many_experts": (dict(T=2000, h=256, F=128, E=128, k=8, bias="none"), False),
    "sk_ragged": (dict(T=777, h=264, F=136, E=16, k=3, bias="none"), False),
    "sk_tiny_fp32": (dict(dtype="f32", h=128, F=256, T=256, E=4, k=2, R=2, bias="none"), False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_sinkhorn_layer(name):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    over, zipf = CASES[name]
    cfg = moe_inputs.get_config("mixtral_sinkhorn", **over)
    inp = cases.router_inputs(cfg, bias=_zipf() if zipf else None)
    assert inp["near_ties"] == 0
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    ref = cases.oracle_layer(cfg, inp, cases.weights_fn_from(cfg, wg, wu, wd))
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    y = layer.forward(cases.to_device(inp["x"], cfg))
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    r = ref["route"]
    assert np.max(np.abs(layer.sk_bias.cpu().numpy() - r["sel_bias"])) <= 1e-5 * max(1.0, np.max(np.abs(r["sel_bias"])))
    np.testing.assert_array_equal(layer.r_out["topk_ids"].cpu().numpy(), r["ids"])
    np.testing.assert_array_equal(layer.r_out["counts"].cpu().numpy(), r["counts"])
    assert cases.rel_max(layer.r_out["gates"].cpu().numpy(), r["gates"]) <= 1e-5
    assert abs(float(layer.r_out["aux"].item()) - r["aux"]) <= 1e-5 * r["aux"]
    np.testing.assert_array_equal(layer.d_out["dest_row"].cpu().numpy(), ref["disp"]["dest_row"])
    fn, tol = cases.y_tolerance(cfg)
    assert fn(cases.from_device(y, cfg), ref["y"]) <= tol


def test_sinkhorn_undoes_the_zipf_skew():
    """The Zipf bias is a per-expert logit shift, which Sinkhorn balancing removes exactly: the Sinkhorn
    routing of the biased logits equals that of the unbiased ones, and its loads are near uniform."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config("mixtral_sinkhorn", T=4096, h=256, F=128)
    inp = cases.router_inputs(cfg, bias=_zipf())
    x = cases.to_device(inp["x"], cfg)
    w = cases.to_device(inp["w_r"], cfg)
    ids = []
    for b in (torch.from_numpy(inp["bias"]).cuda(), None):
        r = moe.moe_router(x, w, b, 2, "softmax")
        sb = moe.moe_sinkhorn_bias(r["logits"])
        out = moe.moe_router_from_logits(r["logits"], sb, 2, "softmax_selbias")
        torch.cuda.synchronize()
        ids.append(out["ids"].cpu().numpy())
        counts = out["counts"].cpu().numpy()
    assert np.mean(ids[0] == ids[1]) > 0.999          # identical up to fp32 near-ties
    assert counts.max() / counts.min() < 1.15


def test_sinkhorn_full_size_sampled():
    """Mixtral-shaped workload with Sinkhorn routing (T=8192, h=4096, E=8, k=2, F=14336) in the bench's
    launch configuration: all routing indices exact, y on 32 sampled tokens."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config("mixtral_sinkhorn")
    inp = cases.router_inputs(cfg)
    r = inp["route"]
    d = O.dispatch(r["ids"], cfg.E, 0, cfg.R)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    y = layer.forward(cases.to_device(inp["x"], cfg))
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    np.testing.assert_array_equal(layer.r_out["topk_ids"].cpu().numpy(), r["ids"])
    np.testing.assert_array_equal(layer.d_out["dest_row"].cpu().numpy(), d["dest_row"])
    toks = np.sort(np.random.default_rng(9).choice(cfg.T, 32, replace=False))
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    want = O.moe_layer_tokens(toks, x64, r, d, cases.weights_fn_from(cfg, wg, wu, wd))
    got = cases.from_device(y[torch.from_numpy(toks).cuda()], cfg)
    assert cases.rel_l2(got, want) <= 2e-2
