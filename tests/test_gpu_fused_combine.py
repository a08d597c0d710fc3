"""The combine fused into the down GEMM's epilogue (moe_expert_down_combine) against the separate calls.

For every case the layer first runs with the separate down GEMM and moe_combine; the fused call then gets the
same act, tile schedule, weights and routing. eout (and the shared expert's output) must be bitwise the
separate down GEMM's, y bitwise moe_combine's (the same fused multiply-adds in the same order), the arrival
counters zero again after the call, and a second call must give the same bits. y is also checked against the
oracle. Cases cover the one-SM and the 2-SM kernels, capacity drops (including tokens with every choice
dropped), k = 2 and k = 8, and the shared expert in the same launch.
"""
import numpy as np
import pytest

from tests import cases
from tests.test_gpu_parity import run_case

pytestmark = pytest.mark.gpu

CASES = ["page3_small", "page3_small_cf0.5", "mixtral_small_cf1.25", "deepseek_small", "qwen3_small",
         "page3_pair", "mixtral_pair", "qwen3_pair", "deepseek_pair"]


def _fused(layer, stream=None, arrivals=None):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    d, r = layer.d_out, layer.r_out
    if arrivals is None:
        arrivals = moe.moe_combine_arrivals(layer.T, layer.h, layer.device)
    sh = layer.shared_packed is not None
    eout = torch.empty_like(layer.eout)
    eout[d["src_token"] < 0] = 0            # pad rows are never written: make them comparable
    out_sh = torch.empty_like(layer.sh_out) if sh else None
    y = torch.full_like(layer.y, float("nan"))
    moe.moe_expert_down_combine(layer.act, d["tile_sched"], layer.packed, layer.E, layer.h, d["src_token"],
                                d["dest_row"], r["gates"], arrivals, act_shared=layer.sh_act if sh else None,
                                packed_shared=layer.shared_packed, eout=eout, out_shared=out_sh, y=y,
                                stream=stream)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    return eout, out_sh, y, arrivals


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


@pytest.mark.parametrize("name", CASES)
def test_fused_combine_bit_identical(name):
    import torch
    cfg, inp, ref, got, layer, x = run_case(name)
    layer.forward(x)                               # the separate down GEMM and combine, as the reference
    torch.cuda.synchronize()
    live = layer.d_out["src_token"] >= 0
    y_sep = layer.y.clone()
    eout_sep = layer.eout.clone()
    eout_sep[~live] = 0
    e1, sh1, y1, arr = _fused(layer)
    assert torch.equal(_bits(e1), _bits(eout_sep))
    if sh1 is not None:
        assert torch.equal(_bits(sh1), _bits(layer.sh_out))
    assert torch.equal(_bits(y1), _bits(y_sep)), "fused combine differs from moe_combine"
    assert int(arr.abs().sum().item()) == 0, "arrival counters not reset"
    e2, sh2, y2, arr = _fused(layer, arrivals=arr)     # the counters left by the first call are reused
    assert torch.equal(_bits(y2), _bits(y1)) and torch.equal(_bits(e2), _bits(e1))
    assert int(arr.abs().sum().item()) == 0
    fn, tol = cases.y_tolerance(cfg)
    err = fn(cases.from_device(y1, cfg), ref["y"])
    assert err <= tol, f"{name}: fused y error {err:.3e} > {tol}"


def test_fully_dropped_tokens_are_zero():
    """With cf = 0.5 some tokens lose every choice: nothing arrives for them, and the fused call writes y = 0."""
    import torch
    cfg, inp, ref, got, layer, x = run_case("page3_small_cf0.5")
    dropped = np.nonzero(ref["disp"]["drop_mask"].all(axis=1))[0]
    assert dropped.size > 0
    _, _, y, _ = _fused(layer)
    idx = torch.from_numpy(dropped).to(y.device)
    assert not y[idx].float().abs().sum().item()


@pytest.mark.parametrize("name", ["page3_small", "deepseek_pair"])
def test_layer_with_fused_combine(name):
    """MoELayer(fuse_combine=True) gives the bits of the layer with the separate calls."""
    import torch
    from top_routing_dispatch_moe_gb300.layer import MoELayer  # noqa: F401
    cfg, inp, ref, got, layer, x = run_case(name)
    y_sep = layer.forward(x).clone()
    fused = cases.build_gpu_layer(cfg, inp, *_weights(cfg), shared=_shared(cfg), fuse_combine=True)
    y_f = fused.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(_bits(y_f), _bits(y_sep))
    y_f2 = fused.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y_f2), _bits(y_sep))


def _weights(cfg):
    import moe_inputs
    return moe_inputs.all_expert_weights(cfg)


def _shared(cfg):
    import moe_inputs
    return tuple(a[0] for a in moe_inputs.all_expert_weights(cfg, shared=True)) if cfg.n_shared else None
