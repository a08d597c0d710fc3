"""A C program as the library's user (tests/c_client/layer_forward.c): compiled with gcc against include/moe.h and the
in-tree libmoe_gb300.so, it packs the weights and runs moe_layer_forward_host on batches in page-locked host memory,
with no Python between it and the library. Its outputs must be bitwise MoELayer.forward's for the same inputs (the
2-SM GEMM path, capacity drops)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import moe_inputs
from tests import cases

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _compile(tmp_path):
    from top_routing_dispatch_moe_gb300 import build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.path.dirname(os.path.dirname(build.nvcc()))
    pkg = os.path.dirname(build.LIB)
    exe = str(tmp_path / "layer_forward")
    libdirs = [pkg] + [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d)]
    cmd = [cc, "-O2", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_client", "layer_forward.c"), "-o", exe]
    for d in libdirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lmoe_gb300", "-lcudart"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_matches_the_python_layer(tmp_path):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    from top_routing_dispatch_moe_gb300.layer import capacity_slots
    exe = _compile(tmp_path)
    cfg = moe_inputs.get_config("page3_cf1.25", T=2048, h=512, F=384)
    inp = cases.router_inputs(cfg)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg)
    bits = lambda a: np.ascontiguousarray(a).view(np.uint16)   # noqa: E731
    x0 = bits(inp["x"])
    xs = [x0, np.ascontiguousarray(x0[::-1])]
    C = capacity_slots(cfg.cf, cfg.k, cfg.T, cfg.E)
    src = tmp_path / "in.bin"
    with open(src, "wb") as f:
        np.array([cfg.T, cfg.h, cfg.E, cfg.k, cfg.F, moe.GATING[cfg.gating], C, cfg.R, len(xs)], np.int32).tofile(f)
        np.array([cfg.alpha], np.float32).tofile(f)
        for x in xs:
            x.tofile(f)
        for a in (inp["w_r"], wg, wu, wd):
            bits(a).tofile(f)
    dst = tmp_path / "out.bin"
    r = subprocess.run([exe, str(src), str(dst)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    y_c = np.fromfile(dst, dtype=np.uint16).reshape(len(xs), cfg.T, cfg.h)

    layer = cases.build_gpu_layer(cfg, inp, wg, wu, wd)
    assert layer.rows >= 512 * cfg.E                       # the 2-SM GEMMs
    for i, x in enumerate(xs):
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        y = layer.forward(xd)
        torch.cuda.synchronize()
        assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
        np.testing.assert_array_equal(y_c[i], y.view(torch.int16).cpu().numpy().view(np.uint16), err_msg=f"batch {i}")
