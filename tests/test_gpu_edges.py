"""GPU edge cases of the C-ABI path against the oracle: empty input, single token, k = E, one expert,
empty experts, minimum and ragged hidden sizes, everything dropped but the first C, and the device-side
check of out-of-range expert ids."""
import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O
from tests import cases

pytestmark = pytest.mark.gpu


def _run(cfg, bias=None):
    import torch
    inp = cases.router_inputs(cfg, bias=bias)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    shared = tuple(a[0] for a in moe_inputs.all_expert_weights(cfg, shared=True)) if cfg.n_shared else None
    ref = cases.oracle_layer(cfg, inp, cases.weights_fn_from(cfg, wg, wu, wd),
                             (lambda: tuple(moe_inputs.to_f64(w, cfg.dtype) for w in shared)) if shared else None)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd, shared)
    y = layer.forward(cases.to_device(inp["x"], cfg))
    torch.cuda.synchronize()
    return inp, ref, layer, cases.from_device(y, cfg)


@pytest.mark.parametrize("over", [
    dict(T=1, E=4, k=4, R=2),                 # single token, k = E
    dict(T=3, E=1, k=1, R=1),                 # one expert: a dense SwiGLU layer
    dict(T=10, E=64, k=2, R=8),               # most experts empty
    dict(T=129, h=8, F=8),                    # minimum hidden size, F below one 128 block
    dict(T=257, h=264, F=136),                # ragged vector tails in h and F
])
@pytest.mark.parametrize("base", ["tiny_fp32", "page3_cf1.25"])
def test_small_shapes(base, over):
    cfg = moe_inputs.get_config(base, **dict(dict(h=128, F=256, T=64), **over))
    if cfg.E % cfg.R:
        cfg = moe_inputs.get_config(base, **dict(dict(h=128, F=256, T=64), **over, R=1))
    inp, ref, layer, y = _run(cfg)
    np.testing.assert_array_equal(layer.r_out["topk_ids"].cpu().numpy(), ref["route"]["ids"])
    np.testing.assert_array_equal(layer.d_out["dest_row"].cpu().numpy(), ref["disp"]["dest_row"])
    np.testing.assert_array_equal(layer.d_out["offsets"].cpu().numpy(), ref["disp"]["offsets"])
    fn, tol = cases.y_tolerance(cfg)
    assert fn(y, ref["y"]) <= tol


def test_empty_batch():
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    dev = "cuda"
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    w = torch.randn(64, 8, device=dev).to(torch.bfloat16)
    r = moe.moe_router(x, w, None, 2)
    torch.cuda.synchronize()
    assert r["counts"].sum().item() == 0 and r["aux"].item() == 0.0
    d = moe.moe_dispatch(x, r["ids"], 8, capacity=0, num_ranks=2)
    torch.cuda.synchronize()
    assert d["offsets"].cpu().tolist() == [0] * 9 and d["tile_sched"][0].item() == 0
    d2 = moe.moe_dispatch(x, r["ids"], 8, capacity=4, num_ranks=2)
    torch.cuda.synchronize()
    assert d2["offsets"].cpu().tolist() == [4 * e for e in range(9)]
    assert d2["src_token"].cpu().tolist() == [-1] * 32 and torch.count_nonzero(d2["buf"]).item() == 0
    y = moe.moe_combine(torch.empty((0, 64), dtype=torch.bfloat16, device=dev),
                        torch.empty((0, 2), dtype=torch.int32, device=dev),
                        torch.empty((0, 2), dtype=torch.float32, device=dev))
    assert y.shape == (0, 64)


def test_capacity_keeps_first_tokens():
    """Every token routed to experts (0, 1): with C = 5 only tokens 0..4 keep them; the rest are dropped and
    their rows in y are zero."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    T, h, E = 40, 64, 4
    ids = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    x = torch.randn(T, h, device="cuda").to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids).cuda(), E, capacity=5, num_ranks=2)
    torch.cuda.synchronize()
    ref = O.dispatch(ids, E, 5, 2)
    np.testing.assert_array_equal(d["dest_row"].cpu().numpy(), ref["dest_row"])
    np.testing.assert_array_equal(d["src_token"].cpu().numpy(), ref["src_token"])
    assert d["kept_counts"].cpu().tolist() == [5, 5, 0, 0]
    gates = torch.full((T, 2), 0.5, device="cuda")
    y = moe.moe_combine(d["buf"], d["dest_row"], gates)          # identity experts
    torch.cuda.synchronize()
    yn = y.float().cpu().numpy()
    xn = x.float().cpu().numpy()
    np.testing.assert_allclose(yn[:5], xn[:5], rtol=1e-2, atol=1e-2)
    assert np.all(yn[5:] == 0)


def test_out_of_range_id_is_flagged():
    """An expert id >= E is caught by the dispatch kernel's own bounds check: the pair is dropped, nothing is
    written out of bounds, and moe_check_device_error reports MOE_ERR_INVALID_ARG."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    T, h, E = 16, 32, 4
    ids = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    ids[3, 1] = E + 5
    x = torch.randn(T, h, device="cuda").to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids).cuda(), E, capacity=0, num_ranks=1)
    rc = moe.moe_check_device_error()
    assert rc == moe.MOE_ERR_INVALID_ARG and "out of range" in moe.moe_last_error_string()
    assert d["dest_row"][3, 1].item() == -1
    assert moe.moe_check_device_error() == moe.MOE_OK          # the flag was cleared


def test_identity_experts_end_to_end():
    """Dispatch then combine with identity experts (eout = buf): y = sum over kept j of gate * x, and with
    renormalised gates and no drops y = x up to bf16 rounding."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config("mixtral_zipf", T=512, h=256, F=128)
    inp = cases.router_inputs(cfg, bias=np.zeros(8, np.float32))
    x = cases.to_device(inp["x"], cfg)
    r = moe.moe_router(x, cases.to_device(inp["w_r"], cfg), torch.zeros(8, device="cuda"), cfg.k, cfg.gating)
    d = moe.moe_dispatch(x, r["ids"], cfg.E, 0, cfg.R)
    y = moe.moe_combine(d["buf"], d["dest_row"], r["gates"])
    torch.cuda.synchronize()
    assert cases.rel_l2(cases.from_device(y, cfg), moe_inputs.to_f64(inp["x"], cfg.dtype)) < 4e-3


def test_host_argument_errors():
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    x = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")      # h % 8 != 0
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_router(x, torch.zeros((12, 4), dtype=torch.bfloat16, device="cuda"), None, 2)
    assert ei.value.code == moe.MOE_ERR_INVALID_ARG
    x = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_router(x, torch.zeros((16, 4), dtype=torch.bfloat16, device="cuda"), None, 5)   # k > E
    assert ei.value.code == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_router(x, torch.zeros((16, 4), dtype=torch.bfloat16, device="cuda"), None, 2,
                       ws=torch.empty(1, dtype=torch.uint8, device="cuda"))
    assert ei.value.code == moe.MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_router(x.half(), torch.zeros((16, 4), dtype=torch.half, device="cuda"), None, 2)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("C", [0, 50])
def test_dispatch_large_count_table_path(C):
    """T=70000 tokens, E=1024 experts, k=1: the per-chunk count table (69 chunks x 1024 experts) is too large
    for the single-launch scan+scatter, so dispatch takes its three-launch path; both must agree with the
    oracle."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    T, h, E = 70000, 8, 1024
    rng = np.random.default_rng(C)
    ids = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    x = torch.randn(T, h, device="cuda").to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids).cuda(), E, capacity=C, num_ranks=8)
    torch.cuda.synchronize()
    ref = O.dispatch(ids, E, C, 8)
    for key in ["offsets", "kept_counts", "dest_row", "src_token", "src_slot", "rank_counts", "rank_offsets"]:
        np.testing.assert_array_equal(d[key].cpu().numpy(), ref[key], err_msg=key)
    live = ref["src_token"] >= 0
    got = d["buf"].view(torch.int16).cpu().numpy()
    want = x.view(torch.int16).cpu().numpy()[ref["src_token"][live]]
    np.testing.assert_array_equal(got[live], want)
    if C:
        assert np.all(got[~live] == 0)


def test_forward_host_batches_matches_device_forward():
    """Three different batches streamed from pinned host memory (copies overlapped with layer work on other
    streams) give bit-identical outputs to one device-resident forward per batch."""
    import torch
    cfg = moe_inputs.get_config("page3_cf1.25", T=512, h=256, F=256)
    inp = cases.router_inputs(cfg)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    xs = [moe_inputs.make_x(cfg, seed=s) for s in (0, 1, 2)]
    want = []
    for xb in xs:
        want.append(layer.forward(cases.to_device(xb, cfg)).clone())
    torch.cuda.synchronize()
    x_hosts = [torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).pin_memory() for xb in xs]
    y_hosts = [torch.empty(xb.shape, dtype=torch.int16).pin_memory() for xb in xs]
    layer.forward_host_batches(x_hosts, y_hosts)
    for yh, w in zip(y_hosts, want):
        assert torch.equal(yh, w.view(torch.int16).cpu())


@pytest.mark.parametrize("E,k", [(4, 2), (8, 2), (12, 3), (16, 4), (24, 2), (32, 8)])
@pytest.mark.parametrize("T,h", [(1, 1024), (17, 264), (1000, 1024), (300, 8)])
def test_router_small_expert_counts(E, k, T, h):
    """The fused bf16 router for E <= 32 (tensor-core logits, 16 tokens per block, h split over 8 warps):
    expert counts that fill 8-expert blocks partly or fully, a single token, a ragged last 16-token tile,
    h with a partial 32-column chunk (264) and h below one chunk (8), against the oracle's routing."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config("page3_cf1.25", T=T, h=h, E=E, k=k, F=128, R=1)
    inp = cases.router_inputs(cfg)
    assert inp["near_ties"] == 0
    x = cases.to_device(inp["x"], cfg)
    w = cases.to_device(inp["w_r"], cfg)
    r = moe.moe_router(x, w, None, k, cfg.gating, cfg.alpha)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    ref = inp["route"]
    np.testing.assert_array_equal(r["ids"].cpu().numpy(), ref["ids"])
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), ref["counts"])
    assert cases.rel_max(r["logits"].cpu().numpy(), ref["logits"]) <= 1e-5
    assert cases.rel_max(r["gates"].cpu().numpy(), ref["gates"]) <= 1e-5
    assert cases.rel_max(r["P"].cpu().numpy(), ref["P"]) <= 1e-5


@pytest.mark.parametrize("name,E,k", [("page3_cf1.25", 64, 2), ("deepseek_v3", 256, 8), ("qwen3_moe", 128, 8)])
@pytest.mark.parametrize("T,h", [(1, 256), (100, 1024), (700, 200), (2500, 2048)])
@pytest.mark.parametrize("want_logits", [True, False])
def test_router_large_expert_counts(name, E, k, T, h, want_logits):
    """The bf16 router for E > 32: logits on the tensor cores, split over K into up to 16 partial products
    when the 128 x 256 output tiles are fewer than the SMs (one token: 4 chunks of 64 columns for h=256;
    h=200 ends in an 8-column chunk), summed with the bias by the gating kernel. Each workload's gating
    (softmax for E=64 and 128, sigmoid with selection bias for E=256); the logits output requested or not."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config(name, T=T, h=h, E=E, k=k, F=128, R=1)
    inp = cases.router_inputs(cfg)
    assert inp["near_ties"] == 0
    x = cases.to_device(inp["x"], cfg)
    w = cases.to_device(inp["w_r"], cfg)
    b = None if inp["bias"] is None else torch.from_numpy(np.asarray(inp["bias"], np.float32)).cuda()
    r = moe.moe_router(x, w, b, k, cfg.gating, cfg.alpha, want_logits=want_logits)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    ref = inp["route"]
    np.testing.assert_array_equal(r["ids"].cpu().numpy(), ref["ids"])
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), ref["counts"])
    if want_logits:
        assert cases.rel_max(r["logits"].cpu().numpy(), ref["logits"]) <= 1e-5
    assert cases.rel_max(r["gates"].cpu().numpy(), ref["gates"]) <= 1e-5
    assert cases.rel_max(r["P"].cpu().numpy(), ref["P"]) <= 1e-5


def test_router_unsplit_logits_with_bias():
    """The bf16 tensor-core logits GEMM unsplit (T = 10000, E = 64: 79 output tiles, about one per SM) with the
    bias added in its fp32 epilogue, whose rows pass through TMA stores (the last tile 16 rows): logits, the
    indices and the gates against the oracle in the plain softmax mode."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config("page3_cf1.25", T=10000, h=256, E=64, k=4, F=128, R=1)
    bias = np.random.default_rng(5).normal(scale=0.1, size=cfg.E)
    inp = cases.router_inputs(cfg, bias=bias)
    assert inp["near_ties"] == 0
    x = cases.to_device(inp["x"], cfg)
    w = cases.to_device(inp["w_r"], cfg)
    b = torch.from_numpy(np.asarray(inp["bias"], np.float32)).cuda()
    r = moe.moe_router(x, w, b, cfg.k, cfg.gating, cfg.alpha)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    ref = inp["route"]
    np.testing.assert_array_equal(r["ids"].cpu().numpy(), ref["ids"])
    assert cases.rel_max(r["logits"].cpu().numpy(), ref["logits"]) <= 1e-5
    assert cases.rel_max(r["gates"].cpu().numpy(), ref["gates"]) <= 1e-5


def test_router_split_deterministic():
    """The E = 256 router (K split into partial logits, multi-block finalize with an arrival counter): two calls
    give bit-identical logits, gates, P and aux."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    cfg = moe_inputs.get_config("deepseek_v3", T=2000, h=2048, F=128, R=1)
    inp = cases.router_inputs(cfg)
    x = cases.to_device(inp["x"], cfg)
    w = cases.to_device(inp["w_r"], cfg)
    b = torch.from_numpy(np.asarray(inp["bias"], np.float32)).cuda()
    r1 = {k: v.clone() for k, v in moe.moe_router(x, w, b, cfg.k, cfg.gating, cfg.alpha).items()}
    r2 = moe.moe_router(x, w, b, cfg.k, cfg.gating, cfg.alpha)
    torch.cuda.synchronize()
    for key in ("logits", "ids", "gates", "counts", "f", "P", "aux"):
        assert torch.equal(r1[key], r2[key]), key


@pytest.mark.parametrize("T,h,E,k,C,dtype", [
    (1000, 16384, 8, 2, 230, "bf16"),       # 32 KB rows: two 16 KB pieces each, the ring wraps; drops and pads
    (700, 6008, 16, 4, 0, "f32"),           # fp32 rows of 24032 B: pieces of 16384 and 7648 bytes
    (2000, 4096, 1024, 1, 4, "bf16"),       # the largest count tables: the fewest ring stages, 63 rows a block
    (300, 8, 4, 2, 0, "f32"),               # 32-byte rows
])
def test_dispatch_copy_ring_shapes(T, h, E, k, C, dtype):
    """The fused dispatch's row copy (bulk-copy unit through a ring of shared stages) on rows split into
    pieces, uneven last pieces, the smallest ring and the smallest rows: index outputs against the oracle's
    dispatch, every kept row bitwise its token row, pad rows zero."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    rng = np.random.default_rng(T + h)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    torch.manual_seed(T)
    x = torch.randn(T, h, device="cuda")
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    d = moe.moe_dispatch(x, torch.from_numpy(ids).cuda(), E, capacity=C, num_ranks=1)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK
    ref = O.dispatch(ids, E, C, 1)
    for key in ["offsets", "kept_counts", "dest_row", "src_token", "src_slot", "rank_counts", "rank_offsets"]:
        np.testing.assert_array_equal(d[key].cpu().numpy(), ref[key], err_msg=key)
    iv = torch.int16 if dtype == "bf16" else torch.int32
    live = ref["src_token"] >= 0
    got = d["buf"].view(iv).cpu().numpy()
    want = x.view(iv).cpu().numpy()[ref["src_token"][live]]
    np.testing.assert_array_equal(got[live], want)
    if C:
        assert np.all(got[~live] == 0)
    from top_routing_dispatch_moe_gb300.checks import check_dispatch
    assert check_dispatch(d, ids, E, C, 1, x=x) == []
