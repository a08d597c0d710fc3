"""FP8 dispatch payload on the GPU against the oracle.

moe_dispatch_fp8: e4m3 codes and per-token, per-128-column scales bit-exact (the same fp32 division and
round-to-nearest-even on both sides), indices identical to moe_dispatch. moe_expert_up_gate_fp8: its prologue
turns the staged codes into the bf16 operand tile in shared memory; fed the oracle's dequantised rows as bf16,
the bf16 GEMM on the same (one-SM) kernel must give bit-identical act, which checks the converter's values and
its 128-byte swizzle exactly. moe_dequant_fp8 bit-exact against the oracle's dequantised rows. The layer with the
FP8 payload (dequantisation pass, then the bf16 GEMM) against the oracle's FP8 layer (normwise 2e-2).
"""
import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O
from tests import cases

pytestmark = pytest.mark.gpu


def _problem(T, h, E, k, seed):
    import torch
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = rng.normal(size=(T, h)).astype(np.float32)
    if h >= 256:
        x[::7, 128:256] = 0.0                 # all-zero blocks: scale 1, codes 0
        x[1::5, :128] *= 1e-4                 # small blocks: subnormal codes appear
        x[2::9, -128:] *= 300.0               # large blocks
    xb = torch.from_numpy(x).to("cuda").to(torch.bfloat16)
    x32 = xb.float().cpu().numpy()            # the bf16 values, exactly
    return ids, xb, x32


@pytest.mark.parametrize("T,h,E,k,C", [(300, 256, 4, 2, 0), (500, 384, 8, 2, 100), (1, 128, 2, 1, 0),
                                       (257, 1024, 8, 4, 150), (4000, 4096, 8, 2, 1250), (1500, 12288, 8, 2, 450),
                                       (5000, 128, 1024, 8, 0)])
def test_dispatch_fp8_bit_exact(T, h, E, k, C):
    """Small count tables take the fused launch (scan, scatter and quantised copy in one kernel; among them the
    page-3 width with 27 tokens per block, and 24 KB rows); the last case (E = 1024, T k = 40000) the separate
    count / scan / scatter / copy launches."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    ids, xb, x32 = _problem(T, h, E, k, seed=T + h)
    ids_d = torch.from_numpy(ids).to("cuda")
    d8 = moe.moe_dispatch_fp8(xb, ids_d, E, C, 1)
    d16 = moe.moe_dispatch(xb, ids_d, E, C, 1)
    torch.cuda.synchronize()
    for key in ["offsets", "kept_counts", "dest_row", "drop_mask", "src_token", "src_slot", "rank_counts",
                "rank_offsets"]:
        assert torch.equal(d8[key], d16[key]), key
    disp = O.dispatch(ids, E, C, 1)
    codes, scales = O.dispatch_payload_fp8(x32, disp)
    np.testing.assert_array_equal(d8["buf8"].cpu().numpy(), codes)
    np.testing.assert_array_equal(d8["scales"].cpu().numpy(), scales)


@pytest.mark.parametrize("T,h,E,k,C", [(300, 256, 4, 2, 0), (257, 1024, 8, 4, 150)])
def test_dequant_fp8_matches_oracle(T, h, E, k, C):
    """moe_dequant_fp8 (the receive side as a pass of its own): bf16(fp32(value) * scale) for every code,
    bit-identical to the oracle's dequantised rows (pad rows: codes 0, scale 0 -> 0)."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    ids, xb, x32 = _problem(T, h, E, k, seed=T + 2 * h)
    d8 = moe.moe_dispatch_fp8(xb, torch.from_numpy(ids).to("cuda"), E, C, 1)
    out = moe.moe_dequant_fp8(d8["buf8"], d8["scales"])
    torch.cuda.synchronize()
    deq = O.fp8_dequantize_rows(d8["buf8"].cpu().numpy(), d8["scales"].cpu().numpy())
    np.testing.assert_array_equal(out.float().cpu().numpy(), deq.astype(np.float32))


@pytest.mark.parametrize("sizes", [[0, 1, 127, 129, 300], [0, 257, 1900, 40]])
def test_up_gate_fp8_prologue(sizes):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(2)
    E, h, F = len(sizes), 384, 256
    ids = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])[:, None]
    np.random.default_rng(4).shuffle(ids)
    _, xb, x32 = _problem(ids.shape[0], h, E, 1, seed=9)
    ids_d = torch.from_numpy(ids).to("cuda")
    d8 = moe.moe_dispatch_fp8(xb, ids_d, E, 0, 1)
    mk = lambda *s: (torch.randn(*s, device="cuda") / s[-1] ** 0.5).to(torch.bfloat16)
    packed = moe.moe_pack_expert_weights(mk(E, F, h), mk(E, F, h), mk(E, h, F))
    act8 = moe.moe_expert_up_gate_fp8(d8["buf8"], d8["scales"], d8["tile_sched"], packed, E, F)
    deq = O.fp8_dequantize_rows(d8["buf8"].cpu().numpy(), d8["scales"].cpu().numpy())
    buf_deq = torch.from_numpy(deq.astype(np.float32)).to("cuda").to(torch.bfloat16)    # exact: already bf16 values
    act16 = moe.moe_expert_up_gate(buf_deq, d8["tile_sched"], packed, E, F)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    off = d8["offsets"].cpu().tolist()
    rows = sum(sizes)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if rows < 512 * E:                    # both on the one-SM kernel: the same operand tiles, bit for bit
            assert torch.equal(act8[a:b], act16[a:b]), f"expert {e}"
        else:                                 # the bf16 GEMM ran on the 2-SM kernel
            assert cases.rel_l2(act8[a:b].double().cpu().numpy(), act16[a:b].double().cpu().numpy()) <= 1e-2


def test_layer_fp8_payload():
    import torch
    cfg = moe_inputs.get_config("page3_fp8", T=600, h=384, F=256)
    inp = cases.router_inputs(cfg)
    assert inp["near_ties"] == 0
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    y = layer.forward(cases.to_device(inp["x"], cfg))
    torch.cuda.synchronize()
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    ref = O.moe_layer(x64, moe_inputs.to_f64(inp["w_r"], cfg.dtype), inp["bias"], cases.weights_fn_from(cfg, wg, wu, wd),
                      k=cfg.k, gating=cfg.gating, cf=cfg.cf, R=cfg.R, alpha=cfg.alpha, payload="fp8")
    np.testing.assert_array_equal(layer.r_out["topk_ids"].cpu().numpy(), ref["router"]["ids"])
    assert cases.rel_l2(cases.from_device(y, cfg), ref["y"]) <= 2e-2
    ref16 = O.moe_layer(x64, moe_inputs.to_f64(inp["w_r"], cfg.dtype), inp["bias"],
                        cases.weights_fn_from(cfg, wg, wu, wd), k=cfg.k, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                        alpha=cfg.alpha)
    # the FP8 payload moves y by about the e4m3 rounding (relative 2^-4 per element, averaging out)
    assert cases.rel_l2(ref["y"], ref16["y"]) <= 5e-2
