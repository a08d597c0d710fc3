"""CPU checks of the C-ABI library: it loads, exports every entry point include/moe.h declares, and its
size functions and host-side argument checks behave as documented (no compute calls without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from top_routing_dispatch_moe_gb300 import build
    build.build()
    from top_routing_dispatch_moe_gb300 import moe
    return moe


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 18
    raw = lib.raw_lib()
    for n in names:
        assert hasattr(raw, n), n
    assert sorted(lib.EXPORTED) == names
    assert "sm_103a" in lib.moe_version()


def test_size_functions(lib):
    assert lib.moe_dispatch_rows(4096, 8, 2, 1280) == 8 * 1280
    assert lib.moe_dispatch_rows(4096, 8, 2, 0) == 8192
    # tile schedule: header + prefix (aligned to 4 words) + 4 words per tile, at most rows/128 + E tiles
    E = 8
    words = ((2 + E + 1 + 3) & ~3) + 4 * ((8 * 1280 + 127) // 128 + E)
    assert lib.moe_tile_sched_bytes(4096, 8, 2, 1280) == 4 * words
    Fp = 12288
    assert lib.moe_packed_weights_bytes(8, 4096, 12288, lib.MOE_BF16) == 8 * 2 * Fp * 4096 * 2 + 8 * 4096 * 12288 * 2
    assert lib.moe_packed_weights_bytes(1, 8, 8, lib.MOE_F32) == 2 * 128 * 8 * 4 + 8 * 8 * 4
    assert lib.moe_expert_ffn_workspace_size(10240, 12288, lib.MOE_BF16) == 10240 * 12288 * 2
    assert lib.moe_router_workspace_size(4096, 4096, 8, 2, lib.MOE_BF16) > 0
    assert lib.moe_dispatch_workspace_size(4096, 8, 2, 0) >= 8 * 4 * (4096 // 512)


def test_host_checks_reject_before_any_cuda_call(lib):
    raw = lib.raw_lib()
    P = ctypes.c_void_p
    n = None
    # bad dtype
    assert raw.moe_router(n, n, n, 4, 16, 4, 2, 7, 0, 0.0, n, n, n, n, n, n, n, n, 0, n) == lib.MOE_ERR_UNSUPPORTED
    assert "dtype" in lib.moe_last_error_string()
    # bad gating
    assert raw.moe_router(n, n, n, 4, 16, 4, 2, 1, 9, 0.0, n, n, n, n, n, n, n, n, 0, n) == lib.MOE_ERR_UNSUPPORTED
    # h not a multiple of 8
    assert raw.moe_router(n, n, n, 4, 12, 4, 2, 1, 0, 0.0, n, n, n, n, n, n, n, n, 0, n) == lib.MOE_ERR_INVALID_ARG
    # k > E
    assert raw.moe_router(n, n, n, 4, 16, 4, 5, 1, 0, 0.0, n, n, n, n, n, n, n, n, 0, n) == lib.MOE_ERR_INVALID_ARG
    # null outputs
    assert raw.moe_router(n, n, n, 4, 16, 4, 2, 1, 0, 0.0, n, n, n, n, n, n, n, n, 0, n) == lib.MOE_ERR_INVALID_ARG
    # misaligned pointer
    bad = P(0x1003)
    ok = P(0x1000)
    assert raw.moe_router(bad, ok, n, 4, 16, 4, 2, 1, 0, 0.0, n, ok, ok, ok, ok, ok, ok, n, 0,
                          n) == lib.MOE_ERR_INVALID_ARG
    # workspace too small (checked before launching)
    assert raw.moe_router(ok, ok, n, 4, 16, 4, 2, 1, 0, 0.0, n, ok, ok, ok, ok, ok, ok, ok, 1,
                          n) == lib.MOE_ERR_WORKSPACE
    # dispatch: ranks must divide E; capacity >= 0
    args = [ok, ok, 4, 16, 8, 2, 0, 3, 1] + [ok] * 10 + [ok, 1 << 20, n]
    assert raw.moe_dispatch(*args) == lib.MOE_ERR_INVALID_ARG
    args[6], args[7] = -1, 2
    assert raw.moe_dispatch(*args) == lib.MOE_ERR_INVALID_ARG
    # FFN: F % 8
    assert raw.moe_expert_ffn(ok, ok, ok, 8, 16, 12, 4, 1, ok, ok, 1 << 20, n) == lib.MOE_ERR_INVALID_ARG
    # FFN workspace
    assert raw.moe_expert_ffn(ok, ok, ok, 8, 16, 16, 4, 1, ok, ok, 8, n) == lib.MOE_ERR_WORKSPACE
    # combine: dtype
    assert raw.moe_combine(ok, ok, ok, n, 4, 16, 2, 5, ok, n) == lib.MOE_ERR_UNSUPPORTED
    # pack: F % 8
    assert raw.moe_pack_expert_weights(ok, ok, ok, 2, 16, 12, 1, ok, n) == lib.MOE_ERR_INVALID_ARG
    # dispatch: E out of range, misaligned x, workspace too small
    args = [ok, ok, 4, 16, 8, 2, 0, 1, 1] + [ok] * 10 + [ok, 1 << 20, n]
    args[4] = 0
    assert raw.moe_dispatch(*args) == lib.MOE_ERR_INVALID_ARG
    args[4], args[0] = 8, bad
    assert raw.moe_dispatch(*args) == lib.MOE_ERR_INVALID_ARG
    assert "aligned" in lib.moe_last_error_string()
    args[0], args[20] = ok, 1
    assert raw.moe_dispatch(*args) == lib.MOE_ERR_WORKSPACE
    # combine: k out of range, null eout, misaligned y
    assert raw.moe_combine(ok, ok, ok, n, 4, 16, 17, 1, ok, n) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_combine(n, ok, ok, n, 4, 16, 2, 1, ok, n) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_combine(ok, ok, ok, n, 4, 16, 2, 1, bad, n) == lib.MOE_ERR_INVALID_ARG
    # expert up/gate: dtype, misaligned act
    assert raw.moe_expert_up_gate(ok, ok, ok, 8, 16, 16, 4, 5, ok, n) == lib.MOE_ERR_UNSUPPORTED
    assert raw.moe_expert_up_gate(ok, ok, ok, 8, 16, 16, 4, 1, bad, n) == lib.MOE_ERR_INVALID_ARG


def test_host_checks_of_the_backward_and_fp8_entry_points(lib):
    raw = lib.raw_lib()
    P = ctypes.c_void_p
    n = None
    ok, bad = P(0x1000), P(0x1003)
    # dequantisation pass: h % 128, alignment, nulls; zero rows is a no-op
    assert raw.moe_dequant_fp8(ok, ok, 4, 100, ok, n) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_dequant_fp8(bad, ok, 4, 128, ok, n) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_dequant_fp8(n, n, 4, 128, n, n) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_dequant_fp8(n, n, 0, 128, n, n) == lib.MOE_OK
    # the pre-activation-saving forward and the backward from it: bf16 only, pointers checked
    assert raw.moe_expert_up_gate_save(ok, ok, ok, 4, 16, 16, 8, n, 0, n, n, n, lib.MOE_F32, ok, ok,
                                       n) == lib.MOE_ERR_UNSUPPORTED
    assert raw.moe_expert_up_gate_save(ok, ok, ok, 4, 16, 16, 8, n, 0, n, n, n, lib.MOE_BF16, ok, n,
                                       n) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_expert_up_gate_backward_saved(ok, ok, ok, ok, 4, 16, 16, 8, lib.MOE_F32, ok, ok,
                                                 n) == lib.MOE_ERR_UNSUPPORTED
    assert raw.moe_expert_up_gate_backward_saved(n, ok, ok, ok, 4, 16, 16, 8, lib.MOE_BF16, ok, ok,
                                                 n) == lib.MOE_ERR_INVALID_ARG
    # weight gradients: every operand 16-byte aligned (vector transposes), checked before any launch
    ws = lib.raw_lib().moe_expert_weight_grads_workspace_size(4, 16, 16, 8, lib.MOE_BF16)
    assert ws > 0
    assert raw.moe_expert_weight_grads(bad, ok, ok, ok, ok, ok, 4, 16, 16, 8, lib.MOE_BF16, ok, ok, ok, ok, ws,
                                       n) == lib.MOE_ERR_INVALID_ARG
    # dispatch backward: the tensor-core path's workspace holds the d_logits pieces and the fp32 router term
    T, h, E = 1000, 1024, 256
    need = lib.raw_lib().moe_dispatch_backward_workspace_size(T, h, E, lib.MOE_BF16)
    assert need >= T * 3 * E * 2 + T * h * 4
    assert lib.raw_lib().moe_dispatch_backward_workspace_size(T, h, 8, lib.MOE_BF16) < need
    # router weight gradient: room for either path
    assert lib.raw_lib().moe_router_weight_grad_workspace_size(T, h, E) >= h * 1024 * 2 + E * 3 * 1024 * 2


def _c_kind(t):
    """Kind of a C type of the header: ptr, void, f32, f64, or i/u plus the width in bits (LP64)."""
    t = " ".join(t.replace("const", " ").split())
    if "*" in t:
        return "ptr"
    return {"int": "i32", "unsigned": "u32", "size_t": "u64", "long long": "i64", "unsigned long long": "u64",
            "float": "f32", "double": "f64", "void": "void"}[t]


def _ct_kind(c):
    """The same kind for a ctypes type (ctypes aliases types of equal width, so compare by width and sign)."""
    if c is None:
        return "void"
    if c in (ctypes.c_void_p, ctypes.c_char_p):
        return "ptr"
    if c in (ctypes.c_float, ctypes.c_double):
        return "f%d" % (8 * ctypes.sizeof(c))
    return ("i" if c(-1).value < 0 else "u") + str(8 * ctypes.sizeof(c))


def test_binding_signatures_match_the_header(lib):
    """Every prototype of include/moe.h against the ctypes signature the binding gives it: the same return
    kind and the same parameter kinds in the same order (a pointer, int, size_t, float, ...), so that no
    argument is marshalled with the wrong width."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    decls = re.findall(r"([A-Za-z_][A-Za-z0-9_ \*]*?)\b(moe_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src)
    assert sorted(n for _, n, _ in decls) == _declared()
    sigs = {}
    for name, (res, args) in lib._SIGS.items():
        sigs[name] = (_ct_kind(res), [_ct_kind(a) for a in args])
    checked = 0
    for ret, name, params in decls:
        ps = [p.strip() for p in params.split(",") if p.strip() and p.strip() != "void"]
        want = (_c_kind(ret), [_c_kind(re.sub(r"\b[A-Za-z_][A-Za-z0-9_]*$", "", p)) for p in ps])
        if name in sigs:
            assert sigs[name] == want, (name, sigs[name], want)
            checked += 1
        else:   # declared but bound by hand in the binding: must at least be exported
            assert hasattr(lib.raw_lib(), name), name
    assert checked >= 40


def test_host_checks_of_the_fused_combine(lib):
    """moe_expert_down_combine: bf16 only, the shared expert's three pointers all or none, k in range, y aligned;
    the arrival counters cover every (token, 256-column block)."""
    raw = lib.raw_lib()
    P = ctypes.c_void_p
    n = None
    ok, bad = P(0x1000), P(0x1003)
    assert raw.moe_combine_arrivals_bytes(4096, 4096) == 4096 * 16 * 4
    assert raw.moe_combine_arrivals_bytes(3, 264) % 256 == 0 and raw.moe_combine_arrivals_bytes(3, 264) >= 3 * 2 * 4
    args = [ok, ok, ok, 8, 256, 128, 64, ok, ok, ok, 32, 2, n, n, lib.MOE_BF16, ok, n, ok, ok, n]
    bf = list(args)
    bf[14] = lib.MOE_F32
    assert raw.moe_expert_down_combine(*bf) == lib.MOE_ERR_UNSUPPORTED
    half = list(args)
    half[12] = ok                                    # act_shared without packed_shared / out_shared
    assert raw.moe_expert_down_combine(*half) == lib.MOE_ERR_INVALID_ARG
    assert "all NULL or all set" in lib.moe_last_error_string()
    kk = list(args)
    kk[11] = 17
    assert raw.moe_expert_down_combine(*kk) == lib.MOE_ERR_INVALID_ARG
    yy = list(args)
    yy[17] = bad
    assert raw.moe_expert_down_combine(*yy) == lib.MOE_ERR_INVALID_ARG
    nul = list(args)
    nul[18] = n                                      # no arrival counters
    assert raw.moe_expert_down_combine(*nul) == lib.MOE_ERR_INVALID_ARG
    none = list(args)
    none[10] = 0                                     # T = 0: nothing to do, nothing launched
    assert raw.moe_expert_down_combine(*none) == lib.MOE_OK


def test_layer_structs_match_the_header(lib, tmp_path):
    """The ctypes mirrors of moe_layer_desc / moe_layer_views have the sizes and field offsets a C compiler gives
    the header's structs."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    desc_f = [f[0] for f in lib.MoELayerDesc._fields_]
    view_f = [f[0] for f in lib.MoELayerViews._fields_]
    body = ['printf("%zu %zu\\n", sizeof(moe_layer_desc), sizeof(moe_layer_views));']
    body += [f'printf("%zu\\n", offsetof(moe_layer_desc, {f}));' for f in desc_f]
    body += [f'printf("%zu\\n", offsetof(moe_layer_views, {f}));' for f in view_f]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"moe.h\"\nint main(void) {\n    "
                   + "\n    ".join(body) + "\n    return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[:2] == [ctypes.sizeof(lib.MoELayerDesc), ctypes.sizeof(lib.MoELayerViews)]
    got = out[2:]
    want = [getattr(lib.MoELayerDesc, f).offset for f in desc_f] + [getattr(lib.MoELayerViews, f).offset for f in view_f]
    assert got == want


def test_layer_forward_host_checks(lib):
    """moe_layer_forward / moe_layer_forward_host reject a bad descriptor, null buffers and a short workspace before
    anything is enqueued (the fake parameter addresses below are never dereferenced)."""
    raw = lib.raw_lib()
    P = ctypes.c_void_p
    ok = 0x1000
    d = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 0, 0.01, 0, 1, ok, None, ok, None)
    assert raw.moe_layer_workspace_size(None) == 0
    need = raw.moe_layer_workspace_size(ctypes.byref(d))
    need_host = raw.moe_layer_host_workspace_size(ctypes.byref(d))
    assert need > 0 and need_host == need + 4 * ((64 * 64 * 2 + 255) // 256 * 256)
    assert raw.moe_layer_forward(None, P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_layer_forward(ctypes.byref(d), None, P(ok), P(ok), need, None) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_layer_forward(ctypes.byref(d), P(ok), P(ok), P(ok), need - 1, None) == lib.MOE_ERR_WORKSPACE
    assert raw.moe_layer_forward(ctypes.byref(d), P(ok), P(ok), P(ok + 8), need, None) == lib.MOE_ERR_INVALID_ARG
    bad = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 3, 0.01, 0, 1, ok, None, ok, None)   # selection-bias mode
    assert raw.moe_layer_forward(ctypes.byref(bad), P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_UNSUPPORTED
    bad = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 0, 0.01, 0, 3, ok, None, ok, None)   # 3 ranks, E = 4
    assert raw.moe_layer_forward(ctypes.byref(bad), P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_INVALID_ARG
    bad = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 0, 0.01, 0, 1, None, None, ok, None)  # no router weight
    assert raw.moe_layer_forward(ctypes.byref(bad), P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_INVALID_ARG
    bad = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 0, 0.01, 0, 1, ok, None, ok, None, 5, 0, 0)  # routing 5
    assert raw.moe_layer_forward(ctypes.byref(bad), P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_UNSUPPORTED
    bad = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_F32, 0, 0.01, 0, 1, ok, None, ok, None, 0, 1, 0)    # fp32 + FP8
    assert raw.moe_layer_forward(ctypes.byref(bad), P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_UNSUPPORTED
    bad = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 0, 0.01, 0, 1, ok, None, ok, None, 0, 1, 0)   # h % 128
    assert raw.moe_layer_forward(ctypes.byref(bad), P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_INVALID_ARG
    bad = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 0, 0.01, 0, 1, ok, None, ok, None, 1, 0, 0)   # EC, C = 0
    assert raw.moe_layer_forward(ctypes.byref(bad), P(ok), P(ok), P(ok), need, None) == lib.MOE_ERR_INVALID_ARG
    ec = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 0, 0.01, 16, 1, ok, None, ok, None, 1, 0, 0)   # EC, C = 16
    sk = lib.MoELayerDesc(64, 64, 4, 2, 64, lib.MOE_BF16, 3, 0.01, 0, 1, ok, None, ok, None, 2, 0, 0)    # Sinkhorn
    for dd in (ec, sk):
        n_dd = raw.moe_layer_workspace_size(ctypes.byref(dd))
        assert n_dd > 0
        assert raw.moe_layer_forward(ctypes.byref(dd), P(ok), P(ok), P(ok), n_dd - 1, None) == lib.MOE_ERR_WORKSPACE
    arr = (P * 1)(ok)
    assert raw.moe_layer_forward_host(ctypes.byref(d), -1, arr, arr, P(ok), need_host, None) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_layer_forward_host(ctypes.byref(d), 1, arr, arr, P(ok), need_host - 1, None) == lib.MOE_ERR_WORKSPACE
    assert raw.moe_layer_forward_host(ctypes.byref(d), 1, None, arr, P(ok), need_host, None) == lib.MOE_ERR_INVALID_ARG
