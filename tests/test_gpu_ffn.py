"""The grouped SwiGLU GEMMs alone, on one dense group, against the same products computed by torch in fp32
from the same bf16 operands (a localising check: on failure it reports which 128-row / 32-column blocks
disagree), plus the tile-schedule corner cases: empty experts, one-row experts, ragged tails.

The library runs the 2-SM kernel (pairs of 128-row tiles on a two-CTA cluster) when rows >= 512 * E and the
one-SM kernel otherwise; the cases below cover both, including odd tile counts (a phantom half tile) and
output widths that end inside the second CTA's half of a 256-column tile."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _ref_act(x, wg, wu):
    g = x.float() @ wg.float().T
    u = x.float() @ wu.float().T
    return g * torch_sigmoid(g) * u


def torch_sigmoid(t):
    import torch
    return torch.sigmoid(t)


def _blocks(err, rb=128, cb=32):
    bad = []
    for i in range(0, err.shape[0], rb):
        for j in range(0, err.shape[1], cb):
            blk = err[i:i + rb, j:j + cb]
            if blk.numel() and blk.max().item() > 0.05:
                bad.append((i, j, round(blk.max().item(), 3)))
    return bad[:12]


@pytest.mark.parametrize("rows,h,F", [(128, 128, 128), (300, 256, 384), (77, 512, 256), (1000, 1024, 640),
                                      (640, 384, 256), (1100, 512, 384), (512, 256, 128)])
def test_dense_group_up_gate_and_down(rows, h, F):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(rows + h + F)
    dev = "cuda"
    x = torch.randn(rows, h, device=dev).to(torch.bfloat16)
    wg = (torch.randn(1, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(1, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(1, h, F, device=dev) / F ** 0.5).to(torch.bfloat16)
    packed = moe.moe_pack_expert_weights(wg, wu, wd)
    sched = moe.moe_dense_tile_sched(rows)
    act = moe.moe_expert_up_gate(x, sched, packed, 1, F)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    ref = _ref_act(x, wg[0], wu[0])
    err = (act.float() - ref).abs() / (ref.abs().max() + 1e-30)
    rel = ((act.float() - ref).norm() / ref.norm()).item()
    assert rel < 1e-2, f"act rel err {rel:.3e}; bad blocks (row, col, err): {_blocks(err)}"
    eout = moe.moe_expert_down(act, sched, packed, 1, h)
    torch.cuda.synchronize()
    ref2 = act.float() @ wd[0].float().T
    err2 = (eout.float() - ref2).abs() / (ref2.abs().max() + 1e-30)
    rel2 = ((eout.float() - ref2).norm() / ref2.norm()).item()
    assert rel2 < 1e-2, f"eout rel err {rel2:.3e}; bad blocks: {_blocks(err2)}"


def test_grouped_schedule_with_empty_and_tiny_experts():
    """Experts with 0, 1, 127, 128, 129 and 300 rows in one grouped call (dropless dispatch of crafted ids)."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(0)
    dev = "cuda"
    sizes = [0, 1, 127, 128, 129, 300, 0, 5]
    E, h, F = len(sizes), 256, 256
    ids = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(0).shuffle(ids)
    T = ids.size
    x = torch.randn(T, h, device=dev).to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids[:, None]).to(dev), E, 0, 1)
    wg = (torch.randn(E, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, h, F, device=dev) / F ** 0.5).to(torch.bfloat16)
    packed = moe.moe_pack_expert_weights(wg, wu, wd)
    eout = moe.moe_expert_ffn(d["buf"], d["tile_sched"], packed, E, F)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    off = d["offsets"].cpu().tolist()
    assert off == list(np.concatenate([[0], np.cumsum(sizes)]))
    for e in range(E):
        if sizes[e] == 0:
            continue
        xb = d["buf"][off[e]:off[e + 1]]
        a = _ref_act(xb, wg[e], wu[e]).to(torch.bfloat16).float()
        ref = a @ wd[e].float().T
        got = eout[off[e]:off[e + 1]].float()
        rel = ((got - ref).norm() / ref.norm()).item()
        assert rel < 1e-2, f"expert {e} ({sizes[e]} rows): rel err {rel:.3e}"


def test_grouped_schedule_on_the_pair_kernel():
    """Experts with 0, 1, 257 and 1900 rows (0, 1, 3 and 15 tiles: three odd counts) with rows >= 512 * E, so the
    2-SM kernel runs, its phantom half tiles included."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(1)
    dev = "cuda"
    sizes = [0, 1, 257, 1900]
    E, h, F = len(sizes), 512, 384
    assert sum(sizes) >= 512 * E
    ids = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(1).shuffle(ids)
    T = ids.size
    x = torch.randn(T, h, device=dev).to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids[:, None]).to(dev), E, 0, 1)
    wg = (torch.randn(E, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, h, F, device=dev) / F ** 0.5).to(torch.bfloat16)
    packed = moe.moe_pack_expert_weights(wg, wu, wd)
    eout = moe.moe_expert_ffn(d["buf"], d["tile_sched"], packed, E, F)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    off = d["offsets"].cpu().tolist()
    for e in range(E):
        if sizes[e] == 0:
            continue
        xb = d["buf"][off[e]:off[e + 1]]
        a = _ref_act(xb, wg[e], wu[e]).to(torch.bfloat16).float()
        ref = a @ wd[e].float().T
        got = eout[off[e]:off[e + 1]].float()
        rel = ((got - ref).norm() / ref.norm()).item()
        assert rel < 1e-2, f"expert {e} ({sizes[e]} rows): rel err {rel:.3e}"


@pytest.mark.parametrize("h,F", [(512, 384), (1024, 200)])
def test_odd_last_tiles_on_the_pair_kernel(h, F):
    """Every expert ends on a pair whose second tile is absent (a phantom half), its last tile holding 1, 31, 32, 33,
    40, 100 or 128 valid rows, on the 2-SM kernel. Every act and eout element of every expert against torch in fp32
    from the same bf16 operands; F = 200 ends the act columns inside the first half of the last 256-column tile."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(2)
    dev = "cuda"
    sizes = [1, 256 + 31, 512 + 32, 256 + 33, 100, 128, 2560 + 40]
    E = len(sizes)
    assert sum(sizes) >= 512 * E and all(-(-n // 128) % 2 == 1 for n in sizes)
    ids = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)])
    np.random.default_rng(2).shuffle(ids)
    x = torch.randn(ids.size, h, device=dev).to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids[:, None]).to(dev), E, 0, 1)
    wg = (torch.randn(E, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(E, F, h, device=dev) / h ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(E, h, F, device=dev) / F ** 0.5).to(torch.bfloat16)
    packed = moe.moe_pack_expert_weights(wg, wu, wd)
    rows = d["buf"].shape[0]
    act = torch.empty(rows, F, dtype=torch.bfloat16, device=dev)
    eout = torch.empty(rows, h, dtype=torch.bfloat16, device=dev)
    moe.moe_expert_up_gate(d["buf"], d["tile_sched"], packed, E, F, act)
    moe.moe_expert_down(act, d["tile_sched"], packed, E, h, eout)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    off = d["offsets"].cpu().tolist()
    for e in range(E):
        xb = d["buf"][off[e]:off[e + 1]]
        a_ref = _ref_act(xb, wg[e], wu[e])
        a_got = act[off[e]:off[e + 1]].float()
        # act is bf16-rounded (relative 2^-9) from fp32 sums of the same products in another order
        err = (a_got - a_ref).abs() / (a_ref.abs() + 1e-2 * a_ref.abs().mean())
        assert err.max().item() < 2e-2, f"act, expert {e} ({sizes[e]} rows): {_blocks(err)}"
        o_ref = a_got @ wd[e].float().T
        o_got = eout[off[e]:off[e + 1]].float()
        err = (o_got - o_ref).abs() / (o_ref.abs() + 1e-2 * o_ref.abs().mean())
        assert err.max().item() < 2e-2, f"eout, expert {e} ({sizes[e]} rows): {_blocks(err)}"


@pytest.mark.parametrize("sizes,T", [
    ([0, 1, 257, 1900], 300),      # 2-SM kernel (rows >= 512 E); 3 shared tiles: a phantom pair half
    ([5, 130, 0, 77], 1000),       # one-SM kernel; ragged last shared tile
    ([0, 0, 0, 0], 640),           # no routed rows: the launch runs the shared expert alone
    ([40, 300, 2, 700], 0),        # no shared rows
])
def test_shared_expert_fused_into_routed_launch(sizes, T):
    """moe_expert_up_gate_shared / moe_expert_down_shared: the shared expert's dense tiles appended to the routed
    experts' work list of one launch per GEMM give bit-identical results to the separate calls (each tile's
    arithmetic is the same)."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(5)
    dev = "cuda"
    E, h, F = len(sizes), 256, 384
    ids = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(sizes)]) if sum(sizes) else np.zeros(0, np.int32)
    np.random.default_rng(2).shuffle(ids)
    xr = torch.randn(max(ids.size, 1), h, device=dev).to(torch.bfloat16)[:ids.size]
    d = moe.moe_dispatch(xr, torch.from_numpy(ids[:, None]).to(dev), E, 0, 1)
    mk = lambda *s: (torch.randn(*s, device=dev) / s[-1] ** 0.5).to(torch.bfloat16)
    packed = moe.moe_pack_expert_weights(mk(E, F, h), mk(E, F, h), mk(E, h, F))
    packed_sh = moe.moe_pack_expert_weights(mk(1, F, h), mk(1, F, h), mk(1, h, F))
    x = torch.randn(T, h, device=dev).to(torch.bfloat16)
    buf = d["buf"]
    act, act_sh = moe.moe_expert_up_gate_shared(buf, d["tile_sched"], packed, E, F, x, packed_sh)
    eout, out_sh = moe.moe_expert_down_shared(act, d["tile_sched"], packed, E, h, act_sh, packed_sh)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    off = d["offsets"].cpu().tolist()
    if buf.shape[0]:
        act_ref = moe.moe_expert_up_gate(buf, d["tile_sched"], packed, E, F)
        eout_ref = moe.moe_expert_down(act_ref, d["tile_sched"], packed, E, h)
        torch.cuda.synchronize()
        for e in range(E):
            a, b = off[e], off[e + 1]
            assert torch.equal(act[a:b], act_ref[a:b]), f"routed act, expert {e}"
            assert torch.equal(eout[a:b], eout_ref[a:b]), f"routed eout, expert {e}"
    if T:
        sched = moe.moe_dense_tile_sched(T)
        act_sh_ref = moe.moe_expert_up_gate(x, sched, packed_sh, 1, F)
        out_sh_ref = moe.moe_expert_down(act_sh_ref, sched, packed_sh, 1, h)
        torch.cuda.synchronize()
        assert torch.equal(act_sh, act_sh_ref)
        assert torch.equal(out_sh, out_sh_ref)
