"""MoELayer.capture_forward: the layer's forward replayed from a CUDA graph gives the same bits as the forward
launched from the host (router outputs, dispatch indices, y), on the 2-SM GEMM path (page-3 routing with
capacity) and on a large-E router (Qwen3-shaped, dropless, E = 128, k = 8)."""
import numpy as np
import pytest

import moe_inputs
from tests import cases

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over", [("page3_cf1.25", dict(T=2048, h=512, F=384)),
                                       ("qwen3_moe", dict(T=4096, h=256, F=128))])
def test_graph_replay_matches_eager(name, over):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    from top_routing_dispatch_moe_gb300.layer import MoELayer
    cfg = moe_inputs.get_config(name, **over)
    inp = cases.router_inputs(cfg)
    dev = torch.device("cuda")
    up = lambda a: cases.to_device(a, cfg, dev)   # noqa: E731
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    layer = MoELayer(T=cfg.T, h=cfg.h, E=cfg.E, k=cfg.k, F=cfg.F, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                     alpha=cfg.alpha, w_r=up(inp["w_r"]),
                     bias=torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None,
                     w_gate=up(wg), w_up=up(wu), w_down=up(wd), device=dev)
    x = up(inp["x"])
    layer.forward(x)
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in layer.r_out.items()}
    ref_d = {k: layer.d_out[k].clone() for k in ("dest_row", "src_token", "tile_sched")}
    y_ref = layer.y.clone()
    g = layer.capture_forward(x)
    for t in [layer.y, *layer.r_out.values(), layer.d_out["dest_row"]]:
        t.zero_()                                  # the replay must write them again
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    assert torch.equal(layer.y.view(torch.int16), y_ref.view(torch.int16))
    for k, v in ref.items():
        assert torch.equal(layer.r_out[k], v), k
    for k, v in ref_d.items():
        assert torch.equal(layer.d_out[k], v), k
