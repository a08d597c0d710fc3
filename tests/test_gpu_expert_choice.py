"""Expert-choice routing on the GPU against the oracle: every expert's chosen tokens (bit-exact), gates
(1e-5), the per-token slots (bit-exact), the gathered payload (bit-exact) and the layer output (1e-5 max-rel
in fp32, 2e-2 normwise in bf16); reduced sizes plus the page-3 shape at full size on sampled tokens."""
import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O
from tests import cases

pytestmark = pytest.mark.gpu

CASES = {
    "ec_small_bf16": dict(base="page3_expert_choice", T=1000, h=256, F=384),
    "ec_many_experts": dict(base="page3_expert_choice", T=700, h=512, E=64, k=8, F=256),
    "ec_full_capacity": dict(base="page3_expert_choice", T=333, h=128, E=4, k=4, F=128),
    "ec_tiny_fp32": dict(base="tiny_fp32", routing="expert_choice", cf=1.0),
    "ec_ragged": dict(base="page3_expert_choice", T=1111, h=264, E=16, k=3, F=136, cf=0.8),
}


def _run(name):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    over = dict(CASES[name])
    base = over.pop("base")
    cfg = moe_inputs.get_config(base, **over)
    inp = cases.ec_inputs(cfg)
    C = inp["C"]
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    wf = cases.weights_fn_from(cfg, wg, wu, wd)
    ref = O.expert_choice_layer(moe_inputs.to_f64(inp["x"], cfg.dtype), moe_inputs.to_f64(inp["w_r"], cfg.dtype), wf, C)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    y = layer.forward(cases.to_device(inp["x"], cfg))
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    return cfg, inp, ref, layer, cases.from_device(y, cfg)


@pytest.mark.parametrize("name", list(CASES))
def test_expert_choice_layer(name):
    cfg, inp, ref, layer, y = _run(name)
    assert inp["near_ties"] == 0
    ec = ref["ec"]
    np.testing.assert_array_equal(layer.ec["tokens"].cpu().numpy(), ec["tokens"])
    np.testing.assert_array_equal(layer.ec["slot"].cpu().numpy(), ec["slot"])
    assert cases.rel_max(layer.ec["gates"].cpu().numpy(), ec["gates"]) <= 1e-5
    np.testing.assert_array_equal(cases.from_device(layer.d_out["buf"], cfg), ref["buf"])
    fn, tol = cases.y_tolerance(cfg)
    assert fn(cases.from_device(layer.eout, cfg), ref["eout"]) <= tol
    assert fn(y, ref["y"]) <= tol
    chosen = (ec["slot"] >= 0).any(axis=1)
    assert np.all(y[~chosen] == 0)                       # tokens no expert chose


def test_expert_choice_full_size_sampled():
    """The page-3 shape with expert choice (T=4096, h=4096, E=8, C=1024, F=12288), bench launch
    configuration; all selections exact, y on 32 sampled tokens."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config("page3_expert_choice")
    inp = cases.ec_inputs(cfg)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    y = layer.forward(cases.to_device(inp["x"], cfg))
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    ec = inp["ec"]
    np.testing.assert_array_equal(layer.ec["tokens"].cpu().numpy(), ec["tokens"])
    np.testing.assert_array_equal(layer.ec["slot"].cpu().numpy(), ec["slot"])
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    toks = np.sort(np.random.default_rng(5).choice(cfg.T, 32, replace=False))
    wf = cases.weights_fn_from(cfg, wg, wu, wd)
    want = np.zeros((toks.size, cfg.h))
    for e in range(cfg.E):
        sel = [i for i, t in enumerate(toks) if ec["slot"][t, e] >= 0]
        if sel:
            out = O.swiglu_ffn(x64[toks[sel]], *wf(e))
            want[sel] += np.array([ec["gates"][e][ec["slot"][toks[i], e]] for i in sel])[:, None] * out
    got = cases.from_device(y[torch.from_numpy(toks).cuda()], cfg)
    assert cases.rel_l2(got, want) <= 2e-2
