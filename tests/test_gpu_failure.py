"""Failure detection on the GPU without a fault: the mbarrier waits of the tensor-core GEMMs, of the
dispatch's bulk row copy and of the router's weight staging are bounded. With the limit forced down to one poll the kernel gives up, latches
MOE_ERR_TIMEOUT in the library's device error word, drains its copies (and MMAs, freeing its tensor memory)
and returns; the context stays usable and the next call, at the default limit, is correct."""
import pytest

pytestmark = pytest.mark.gpu


def _problem(rows):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(3)
    h, F = 256, 256
    x = torch.randn(rows, h, device="cuda").to(torch.bfloat16)
    wg = (torch.randn(1, F, h, device="cuda") / h ** 0.5).to(torch.bfloat16)
    wu = (torch.randn(1, F, h, device="cuda") / h ** 0.5).to(torch.bfloat16)
    wd = (torch.randn(1, h, F, device="cuda") / F ** 0.5).to(torch.bfloat16)
    return x, wg, wu, moe.moe_pack_expert_weights(wg, wu, wd), moe.moe_dense_tile_sched(rows), F


@pytest.mark.parametrize("rows", [256, 512])      # the one-SM kernel (rows < 512 * E), the 2-SM kernel
def test_gemm_wait_timeout_reported_and_recoverable(rows):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    x, wg, wu, packed, sched, F = _problem(rows)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    try:
        moe.moe_set_wait_limit(1)
        moe.moe_expert_up_gate(x, sched, packed, 1, F)
        rc = moe.moe_check_device_error()
        msg = moe.moe_last_error_string()
    finally:
        moe.moe_set_wait_limit(0)
    assert rc == moe.MOE_ERR_TIMEOUT, (rc, msg)
    assert "wait ran out" in msg
    act = moe.moe_expert_up_gate(x, sched, packed, 1, F)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    g = x.float() @ wg[0].float().T
    ref = g * torch.sigmoid(g) * (x.float() @ wu[0].float().T)
    assert ((act.float() - ref).norm() / ref.norm()).item() < 1e-2


def test_dispatch_copy_wait_timeout_reported_and_recoverable():
    """The fused dispatch's row copy (bulk-copy unit, one issuing thread per block) waits on an mbarrier for
    each row piece; with the limit at one poll it gives up, waits for the loads already in flight, latches
    MOE_ERR_TIMEOUT and returns; the next call at the default limit copies every kept row exactly."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(5)
    # one 32 KB token row per block (two 16 KB pieces): each block polls its first piece right after issuing
    # the two loads, long before a 16 KB copy can have landed
    T, h, E, k, C = 152, 16384, 8, 2, 48
    x = torch.randn(T, h, device="cuda").to(torch.bfloat16)
    ids = torch.stack([torch.randperm(E, device="cuda")[:k] for _ in range(T)]).to(torch.int32)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    try:
        moe.moe_set_wait_limit(1)
        moe.moe_dispatch(x, ids, E, C, 1)
        rc = moe.moe_check_device_error()
        msg = moe.moe_last_error_string()
    finally:
        moe.moe_set_wait_limit(0)
    assert rc == moe.MOE_ERR_TIMEOUT, (rc, msg)
    assert "site 0x110" in msg
    o = moe.moe_dispatch(x, ids, E, C, 1)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    dest = o["dest_row"].long()
    kept = dest >= 0
    rows = dest[kept]
    toks = torch.arange(T, device="cuda")[:, None].expand(T, k)[kept]
    assert torch.equal(o["buf"][rows].view(torch.int16), x[toks].view(torch.int16))


def test_router_weight_wait_timeout_reported_and_recoverable():
    """The packed-weight router (bf16, E <= 32) has the bulk-copy unit bring the router weight into each block's
    shared memory and waits for it on an mbarrier; with the limit at one poll the wait gives up before a 128 KB
    copy can have landed, latches MOE_ERR_TIMEOUT (site 0x130), waits for the copy and returns; the next call at
    the default limit gives the same outputs as a call before the forced timeout."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    torch.manual_seed(7)
    T, h, E, k = 2048, 4096, 16, 2
    x = torch.randn(T, h, device="cuda").to(torch.bfloat16)
    w = (torch.randn(h, E, device="cuda") * 0.05).to(torch.bfloat16)
    wp = moe.moe_pack_router_weight(w)
    ref = moe.moe_router(x, w, None, k, "softmax", w_packed=wp)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    try:
        moe.moe_set_wait_limit(1)
        moe.moe_router(x, w, None, k, "softmax", w_packed=wp)
        rc = moe.moe_check_device_error()
        msg = moe.moe_last_error_string()
    finally:
        moe.moe_set_wait_limit(0)
    assert rc == moe.MOE_ERR_TIMEOUT, (rc, msg)
    assert "site 0x130" in msg
    again = moe.moe_router(x, w, None, k, "softmax", w_packed=wp)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    for key in ("ids", "gates", "logits", "counts", "P", "aux"):
        assert torch.equal(again[key], ref[key]), key

