"""Host logic of bench.py on the CPU: the parity report of the cpu_baseline leg (its verdict on an exact
output, on a perturbed one and on an index mismatch outside the near ties) and the roofline's choice of bound."""
import types

import numpy as np
import pytest
import torch

import bench
import moe_inputs
from oracle import moe_oracle as O


@pytest.fixture(scope="module")
def oracle_run():
    cfg = moe_inputs.get_config("tiny_fp32")
    inp = bench.host_inputs(cfg)
    w64 = bench.decode_weights(cfg, inp)
    keep = {}
    bench.oracle_step(cfg, inp, w64, np.arange(0, cfg.T, 7), keep)
    return cfg, keep


def _layer(cfg, keep, y_rows):
    y = torch.zeros((cfg.T, cfg.h), dtype=torch.float32)
    y[torch.as_tensor(keep["tokens"])] = torch.as_tensor(y_rows, dtype=torch.float32)
    return types.SimpleNamespace(y=y, r_out={"topk_ids": torch.as_tensor(keep["route"]["ids"].astype(np.int32))})


def test_parity_report_verdicts(oracle_run):
    cfg, keep = oracle_run
    exact = bench.parity_report(cfg, _layer(cfg, keep, keep["y"]), keep)
    assert exact["pass"] and exact["ids_mismatched_tokens"] == 0 and exact["y_err"] < 1e-6
    assert exact["tokens_checked"] == len(keep["tokens"])
    off = bench.parity_report(cfg, _layer(cfg, keep, keep["y"] * 1.01), keep)
    assert not off["pass"] and off["y_err"] > 1e-3
    lay = _layer(cfg, keep, keep["y"])
    ids = lay.r_out["topk_ids"].clone()
    t = int(np.setdiff1d(np.arange(cfg.T), O.near_tie_rows(keep["route"]["gaps"], 1e-6))[0])
    ids[t] = ids[t].flip(0)                 # a swapped pair of ids on a token that is not a near tie
    lay.r_out["topk_ids"] = ids
    swapped = bench.parity_report(cfg, lay, keep)
    assert swapped["ids_mismatched_tokens"] == 1 and not swapped["pass"]


def test_parity_report_skips_other_routings():
    cfg = moe_inputs.get_config("page3_expert_choice")
    assert "skipped" in bench.parity_report(cfg, None, {})


def test_reference_arm_json_line_on_cpu():
    """`bench.py --impl reference` times the oracle on the host cores and prints one JSON line with the bench's
    keys (impl, metric, value, unit, cpu_baseline of kind oracle, e2e without host-device bytes); a rank other
    than 0 prints nothing and exits 0."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3", "--workload",
           "tiny_fp32"]
    env = dict(os.environ, RANK="0")
    out = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("tiny_fp32")
    env["RANK"] = "1"
    out = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_lazy_weights_decode_one_expert_at_a_time():
    """The further workloads' parity decodes expert weights on demand (the DeepSeek-V3-shaped workload's would
    not fit in host memory as float64 all at once): the same values as the eager decode, one expert held."""
    cfg = moe_inputs.get_config("deepseek_v3", T=64, h=64, F=32, E=16, k=4)
    inp = bench.host_inputs(cfg)
    eager = bench.decode_weights(cfg, inp)
    lazy = bench.decode_weights(cfg, inp, lazy=True)
    for e in [3, 0, 15, 3]:
        for a, b in zip(lazy[e], eager[e]):
            np.testing.assert_array_equal(a, b)
        assert sorted(k for k in lazy if k != "shared") == [e]
    for a, b in zip(lazy["shared"](), eager["shared"]()):
        np.testing.assert_array_equal(a, b)


def test_stage_metrics_bounds_and_bandwidths():
    """Per-stage GB/s are the algorithmic bytes over the stage's mean time; the up/gate GEMM's bound is the
    tensor peak for the page-3 shape and the HBM copy bandwidth for the DeepSeek-V3 shape (about one 128-row tile
    per expert: fewer flops per weight byte than the ridge point)."""
    st = {s: [0.01, 0.01] for s in ("router", "dispatch", "up_gate", "down", "combine")}
    cfg = moe_inputs.get_config("page3_cf1.25")
    m = bench.stage_metrics(cfg, st, kept=8192, active=8)
    assert m["roofline"]["bound"] == "tensor" and m["roofline"]["unit"] == "TFLOP/s"
    assert m["router_gbs"] == pytest.approx((cfg.T * cfg.h + cfg.h * cfg.E) * 2 / 1e-5 / 1e9)
    assert m["dispatch_gbs"] == pytest.approx((cfg.T + 8192) * cfg.h * 2 / 1e-5 / 1e9)
    assert m["combine_gbs"] == pytest.approx((8192 + cfg.T) * cfg.h * 2 / 1e-5 / 1e9)
    ds = moe_inputs.get_config("deepseek_v3")
    m = bench.stage_metrics(ds, st, kept=ds.k * ds.T, active=148)
    assert m["roofline"]["bound"] == "hbm" and m["roofline"]["unit"] == "GB/s"
    assert m["combine_gbs"] == pytest.approx((ds.k * ds.T + 2 * ds.T) * ds.h * 2 / 1e-5 / 1e9)
