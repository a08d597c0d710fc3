"""GPU parity of the CUDA path against the oracle, element by element, at sizes the oracle finishes in
seconds (several 128-row tiles, ragged tails, drop-forcing capacities, empty experts).

The "_pair" cases have at least 4 * 128 * E dispatched rows, the size from which the library runs the grouped
GEMMs on the 2-SM (cta_group::2) kernel, with experts of odd and even 128-row tile counts (an odd count leaves
the second CTA of the last pair a phantom tile); every element of their outputs is compared as well.

Indices (ids, counts, offsets, permutation, drop mask, send layout, tile schedule) must match bit-exactly;
the dispatched payload is a copy and must match bit-exactly too. Floats: router logits, gates, f, P and
aux within 1e-5 of max|ref| (fp32 arithmetic on both dtypes); expert outputs and y within 1e-5 max-rel
(fp32 layer) or 2e-2 normwise (bf16 with fp32 accumulation).
"""
import numpy as np
import pytest

import moe_inputs
from tests import cases

pytestmark = pytest.mark.gpu

_ZIPF = None


def _zipf_bias():
    global _ZIPF
    if _ZIPF is None:
        _ZIPF = moe_inputs.load_zipf_bias(moe_inputs.get_config("mixtral_zipf"))
    return _ZIPF


def _cfg(name):
    g = moe_inputs.get_config
    return {
        "tiny_fp32": (g("tiny_fp32"), None),
        "page3_small": (g("page3_cf1.25", T=1000, h=512, F=384), None),
        "page3_small_cf1.0": (g("page3_cf1.25", T=1000, h=512, F=384, cf=1.0), None),
        "page3_small_cf0.5": (g("page3_cf1.25", T=777, h=256, F=256, cf=0.5), None),
        "mixtral_small": (g("mixtral_zipf", T=1500, h=256, F=512), "zipf"),
        "mixtral_small_cf1.25": (g("mixtral_zipf", T=1500, h=256, F=512, cf=1.25), "zipf"),
        "deepseek_small": (g("deepseek_v3", T=700, h=512, F=256), None),
        "qwen3_small": (g("qwen3_moe", T=2000, h=256, F=128), None),
        "tiny_fp32_cf": (g("tiny_fp32", T=300, cf=0.75), None),
        # 2-SM GEMM path: page-3 routing with capacity (C = 813, rows = 6504), the Zipf-skewed renormalised
        # routing dropless (rows = 4600; the largest expert has 13 tiles), Qwen3-shaped uniform routing
        # (rows = 65536 = 4 * 128 * E) and a sigmoid-routed layer with its shared expert in the same launches
        "page3_pair": (g("page3_cf1.25", T=2600, h=512, F=384), None),
        "mixtral_pair": (g("mixtral_zipf", T=2300, h=256, F=512), "zipf"),
        "qwen3_pair": (g("qwen3_moe", T=8192, h=256, F=128), None),
        "deepseek_pair": (g("deepseek_v3", T=2100, h=512, F=256, E=16, k=4), None),
    }[name]


CASE_NAMES = ["tiny_fp32", "page3_small", "page3_small_cf1.0", "page3_small_cf0.5", "mixtral_small",
              "mixtral_small_cf1.25", "deepseek_small", "qwen3_small", "tiny_fp32_cf",
              "page3_pair", "mixtral_pair", "qwen3_pair", "deepseek_pair"]
PAIR_CASES = [n for n in CASE_NAMES if n.endswith("_pair")]
PAIR_MIN_ROWS_PER_EXPERT = 4 * 128     # the library's switch to the 2-SM grouped GEMM

_cache = {}


def run_case(name):
    if name in _cache:
        return _cache[name]
    import torch
    cfg, bias_kind = _cfg(name)
    inp = cases.router_inputs(cfg, bias=_zipf_bias() if bias_kind == "zipf" else None)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    shared = tuple(a[0] for a in moe_inputs.all_expert_weights(cfg, shared=True)) if cfg.n_shared else None
    ref = cases.oracle_layer(cfg, inp, cases.weights_fn_from(cfg, wg, wu, wd),
                             (lambda: tuple(moe_inputs.to_f64(w, cfg.dtype) for w in shared)) if shared else None)
    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd, shared)
    x = cases.to_device(inp["x"], cfg)
    y = layer.forward(x)
    torch.cuda.synchronize()
    from top_routing_dispatch_moe_gb300 import moe
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    got = {k: v.cpu().numpy() for k, v in layer.r_out.items()}
    got.update({k: v.cpu().numpy() for k, v in layer.d_out.items() if k != "buf"})
    got["buf"] = cases.from_device(layer.d_out["buf"], cfg)
    # pad rows of eout are never written by the GEMMs: only the dispatched rows are read back
    got["eout"] = cases.from_device_rows(layer.eout, layer.d_out["src_token"] >= 0, cfg)
    got["act_dtype"] = str(layer.act.dtype)
    got["y"] = cases.from_device(y, cfg)
    got["y_bits"] = y.clone()
    _cache[name] = (cfg, inp, ref, got, layer, x)
    return _cache[name]


@pytest.mark.parametrize("name", CASE_NAMES)
def test_router_indices_exact(name):
    cfg, inp, ref, got, *_ = run_case(name)
    assert inp["near_ties"] == 0
    r = ref["route"]
    np.testing.assert_array_equal(got["topk_ids"], r["ids"])
    np.testing.assert_array_equal(got["counts"], r["counts"])
    assert got["counts"].sum() == cfg.k * cfg.T


@pytest.mark.parametrize("name", CASE_NAMES)
def test_router_floats(name):
    cfg, inp, ref, got, *_ = run_case(name)
    r = ref["route"]
    assert cases.rel_max(got["logits"], r["logits"]) <= 1e-5
    assert cases.rel_max(got["gates"], r["gates"]) <= 1e-5
    assert cases.rel_max(got["f"], r["f"]) <= 1e-6
    assert cases.rel_max(got["P"], r["P"]) <= 1e-5
    assert abs(float(got["aux"][0]) - r["aux"]) <= 1e-5 * abs(r["aux"])


@pytest.mark.parametrize("name", CASE_NAMES)
def test_dispatch_indices_exact(name):
    cfg, inp, ref, got, *_ = run_case(name)
    d = ref["disp"]
    for key in ["offsets", "kept_counts", "dest_row", "src_token", "src_slot", "rank_counts", "rank_offsets"]:
        np.testing.assert_array_equal(got[key], d[key], err_msg=key)
    np.testing.assert_array_equal(got["drop_mask"].astype(bool), d["drop_mask"])
    if cfg.cf > 0 and name.endswith(("cf1.0", "cf0.5", "cf1.25", "_cf")):
        assert d["drop_mask"].any(), "drop-forcing case dropped nothing"


@pytest.mark.parametrize("name", CASE_NAMES)
def test_dispatch_payload_exact(name):
    cfg, inp, ref, got, *_ = run_case(name)
    np.testing.assert_array_equal(got["buf"], ref["buf"])


@pytest.mark.parametrize("name", CASE_NAMES)
def test_tile_schedule(name):
    cfg, inp, ref, got, *_ = run_case(name)
    d = ref["disp"]
    s = got["tile_sched"]
    E = cfg.E
    kept = d["kept_counts"]
    ntiles = [(int(c) + 127) // 128 for c in kept]
    assert s[0] == sum(ntiles) and s[1] == E
    np.testing.assert_array_equal(s[2:2 + E + 1], np.concatenate([[0], np.cumsum(ntiles)]))
    off = (2 + E + 1 + 3) & ~3
    tiles = s[off:off + 4 * s[0]].reshape(-1, 4)
    want = [(e, d["offsets"][e] + 128 * m, min(d["offsets"][e] + 128 * (m + 1), d["offsets"][e] + kept[e]), 0)
            for e in range(E) for m in range(ntiles[e])]
    np.testing.assert_array_equal(tiles, np.array(want, dtype=np.int64).reshape(-1, 4))


@pytest.mark.parametrize("name", CASE_NAMES)
def test_expert_outputs(name):
    cfg, inp, ref, got, *_ = run_case(name)
    d = ref["disp"]
    live = d["src_token"] >= 0
    assert np.isfinite(got["eout"][live]).all()
    fn, tol = cases.y_tolerance(cfg)
    err = fn(got["eout"][live], ref["eout"][live])
    assert err <= tol, f"expert outputs err {err:.3e} > {tol}"


@pytest.mark.parametrize("name", PAIR_CASES)
def test_pair_cases_reach_the_2sm_gemm(name):
    """The reduced cases meant for the 2-SM kernel are above its row threshold, and their experts' 128-row
    tile counts include odd ones (phantom second tiles) as well as even ones."""
    cfg, inp, ref, got, layer, _ = run_case(name)
    assert layer.rows >= PAIR_MIN_ROWS_PER_EXPERT * cfg.E
    tiles = (ref["disp"]["kept_counts"] + 127) // 128
    assert (tiles % 2 == 1).any() and (tiles[tiles > 0] % 2 == 0).any(), tiles


@pytest.mark.parametrize("name", PAIR_CASES)
def test_pair_cases_every_element(name):
    """Every dispatched row of eout and every token's y, one row at a time against the oracle: normwise within
    the bf16 tolerance and no row above 4x it (a wrong tile, a swapped pair half or a phantom tile stored over
    real rows shows up as whole rows far off)."""
    cfg, inp, ref, got, *_ = run_case(name)
    fn, tol = cases.y_tolerance(cfg)
    live = np.nonzero(ref["disp"]["src_token"] >= 0)[0]
    for r in live:
        assert fn(got["eout"][r], ref["eout"][r]) <= 4 * tol, f"eout row {r}"
    for t in range(cfg.T):
        if np.linalg.norm(ref["y"][t]) > 0:
            assert fn(got["y"][t], ref["y"][t]) <= 4 * tol, f"y token {t}"
        else:
            assert not got["y"][t].any(), f"y token {t} (every pair dropped) not zero"


@pytest.mark.parametrize("name", CASE_NAMES)
def test_layer_output(name):
    cfg, inp, ref, got, *_ = run_case(name)
    fn, tol = cases.y_tolerance(cfg)
    err = fn(got["y"], ref["y"])
    assert err <= tol, f"y err {err:.3e} > {tol}"
    # every token's row individually within 4x the tolerance (no silently wrong token)
    for t in range(0, cfg.T, max(1, cfg.T // 97)):
        if np.linalg.norm(ref["y"][t]) > 0:
            assert fn(got["y"][t], ref["y"][t]) <= 4 * tol, t


@pytest.mark.parametrize("name", ["page3_small", "deepseek_small", "tiny_fp32"])
def test_deterministic(name):
    import torch
    cfg, inp, ref, got, layer, x = run_case(name)
    y2 = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int16) if y2.dtype == torch.bfloat16 else y2,
                       got["y_bits"].view(torch.int16) if y2.dtype == torch.bfloat16 else got["y_bits"])
