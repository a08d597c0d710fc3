"""moe_layer_forward / moe_layer_forward_host: the whole layer forward as one C-ABI call.

The chain is the launches of MoELayer.forward (router, dispatch, grouped up/gate and down GEMMs, combine), so y must
be bitwise the Python layer's, whose output the parity tests compare with the oracle; the router ids and aux read
back through moe_layer_views_of must be the layer's too. The host variant runs several batches from page-locked host
memory with the copies on its own streams: each batch's y must be bitwise a device forward of that batch. Cases:
capacity drops on the 2-SM GEMMs (page-3 routing), the one-SM GEMMs, sigmoid gating with a selection bias and the
shared expert inside the routed launches (DeepSeek-V3-shaped), fp32 on the CUDA cores, with and without a shared
expert (which fp32 runs as a dense group of its own), expert-choice routing, Sinkhorn-balanced routing and the FP8
send buffer."""
import numpy as np
import pytest

import moe_inputs
from tests import cases

pytestmark = pytest.mark.gpu

CASES = [("page3_cf1.25", dict(T=2048, h=512, F=384)),     # capacity drops, 2-SM GEMMs (rows >= 512 E)
         ("page3_cf1.25", dict(T=1024, h=512, F=256)),     # one-SM GEMMs
         ("deepseek_v3", dict(T=512, h=256, F=128)),       # sigmoid + selection bias, shared expert, E = 256, k = 8
         ("tiny_fp32", {}),
         ("tiny_fp32", dict(n_shared=1)),
         ("page3_expert_choice", dict(T=1024, h=512, F=256)),
         ("mixtral_sinkhorn", dict(T=1024, h=512, F=256, bias="none")),
         ("page3_fp8", dict(T=1024, h=512, F=256))]


def _layer(name, over):
    import torch
    from top_routing_dispatch_moe_gb300.layer import MoELayer
    cfg = moe_inputs.get_config(name, **over)
    inp = cases.router_inputs(cfg)
    dev = torch.device("cuda")
    up = lambda a: cases.to_device(a, cfg, dev)   # noqa: E731
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    sh = None
    if cfg.n_shared:
        sh = tuple(up(np.ascontiguousarray(a[0])[None]) for a in moe_inputs.all_expert_weights(cfg, shared=True))
    layer = MoELayer(T=cfg.T, h=cfg.h, E=cfg.E, k=cfg.k, F=cfg.F, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                     alpha=cfg.alpha, w_r=up(inp["w_r"]),
                     bias=torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None,
                     w_gate=up(wg), w_up=up(wu), w_down=up(wd), shared=sh, device=dev, routing=cfg.routing,
                     payload=cfg.payload)
    return cfg, layer, up(inp["x"])


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _view(ws, addr, n, dtype):
    import torch
    off = addr - ws.data_ptr()
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


@pytest.mark.parametrize("name,over", CASES)
def test_layer_forward_is_the_python_layer_bitwise(name, over):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg, layer, x = _layer(name, over)
    layer.forward(x)
    torch.cuda.synchronize()
    y_ref = layer.y.clone()
    desc = layer.native_desc()
    ws = moe._bytes_tensor(moe.moe_layer_workspace_size(desc), x.device)
    y = torch.empty_like(x)
    moe.moe_layer_forward(desc, x, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    assert torch.equal(_bits(y), _bits(y_ref))
    v = moe.moe_layer_views_of(desc, ws)
    assert v.rows == layer.rows
    ids = _view(ws, v.topk_ids, cfg.T * cfg.k, torch.int32).view(cfg.T, cfg.k)
    assert torch.equal(ids, layer.r_out["topk_ids"])
    assert torch.equal(_view(ws, v.aux, 1, torch.float32), layer.r_out["aux"])
    if cfg.routing == "expert_choice":
        assert v.dest_row is None
        slot = _view(ws, v.ec_slot, cfg.T * cfg.E, torch.int32).view(cfg.T, cfg.E)
        assert torch.equal(slot, layer.ec["slot"])
    else:
        dest = _view(ws, v.dest_row, cfg.T * cfg.k, torch.int32).view(cfg.T, cfg.k)
        assert torch.equal(dest, layer.d_out["dest_row"])
    if cfg.routing == "sinkhorn":
        assert torch.equal(_view(ws, v.sel_bias, cfg.E, torch.float32), layer.sk_bias)
    if cfg.payload == "fp8":
        assert torch.equal(_view(ws, v.buf8, layer.rows * cfg.h, torch.uint8).view(layer.rows, cfg.h),
                           layer.d_out["buf8"])


@pytest.mark.parametrize("name,over", [CASES[0], CASES[2], CASES[4], CASES[5], CASES[6], CASES[7]])
def test_layer_forward_host_batches(name, over):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg, layer, x = _layer(name, over)
    xs = [x, torch.flip(x, [0]), x * 2, x]               # x * 2 is exact; the scaled logits keep their order
    refs = []
    for xi in xs:
        layer.forward(xi)
        torch.cuda.synchronize()
        refs.append(layer.y.cpu())
    x_h = [xi.cpu().pin_memory() for xi in xs]
    y_h = [torch.empty_like(xi, device="cpu").pin_memory() for xi in xs]
    for t in y_h:
        t.zero_()
    desc = layer.native_desc()
    ws = moe._bytes_tensor(moe.moe_layer_host_workspace_size(desc), x.device)
    moe.moe_layer_forward_host(desc, x_h, y_h, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    for i, (got, ref) in enumerate(zip(y_h, refs)):
        assert torch.equal(_bits(got), _bits(ref)), f"batch {i}"
    # through the layer's helper as well (one call, then a synchronisation)
    y2 = [torch.empty_like(t).pin_memory() for t in y_h]
    layer.forward_host_native(x_h, y2, ws)
    for i, (got, ref) in enumerate(zip(y2, refs)):
        assert torch.equal(_bits(got), _bits(ref)), f"batch {i} (forward_host_native)"
    moe.moe_layer_forward_host(desc, [], [], ws)          # no batches: nothing to do


def test_layer_forward_host_rejects_pageable_buffers():
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg, layer, x = _layer("tiny_fp32", {})
    desc = layer.native_desc()
    ws = moe._bytes_tensor(moe.moe_layer_host_workspace_size(desc), x.device)
    x_pageable = x.cpu()
    y_pinned = torch.empty_like(x_pageable).pin_memory()
    with pytest.raises(moe.MoEError) as err:
        moe.moe_layer_forward_host(desc, [x_pageable], [y_pinned], ws)
    assert err.value.code == moe.MOE_ERR_INVALID_ARG
    assert "page-locked" in str(err.value)


@pytest.mark.parametrize("name,over", [CASES[0], CASES[2], CASES[6]])
def test_layer_forward_captures_into_a_cuda_graph(name, over):
    """moe_layer_forward only enqueues kernels on the caller's stream (no host synchronisation, no allocation), so
    it can be captured into a CUDA graph: replays give the eager call's bits."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg, layer, x = _layer(name, over)
    desc = layer.native_desc()
    ws = moe._bytes_tensor(moe.moe_layer_workspace_size(desc), x.device)
    y_ref = torch.empty_like(x)
    moe.moe_layer_forward(desc, x, y_ref, ws)           # eager (also sets the kernels' attributes up)
    torch.cuda.synchronize()
    y = torch.zeros_like(x)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_layer_forward(desc, x, y, ws, stream=s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    assert torch.equal(_bits(y), _bits(y_ref))
