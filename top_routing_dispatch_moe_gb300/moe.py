"""Python binding of the C-ABI library libmoe_gb300.so (argument marshalling only).

Every function has the name of the C entry point it calls and takes torch tensors for the device buffers;
all computation happens in the library's CUDA kernels. Torch provides device memory and the stream.
Importing this module fails loudly if the library has not been built (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_gb300.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it first (python -m top_routing_dispatch_moe_gb300.build)")
_lib = ctypes.CDLL(_LIB_PATH)

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(6)
MOE_F32, MOE_BF16 = 0, 1
GATING = {"softmax": 0, "softmax_renorm": 1, "sigmoid_bias_renorm": 2, "softmax_selbias": 3}
TILE_M = 128

_P, _I, _Z, _F, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_longlong
_SIGS = {
    "moe_router_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "moe_router": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_router_packed_bytes": (_Z, [_I, _I, _I]),
    "moe_pack_router_weight": (_I, [_P, _I, _I, _I, _P, _P]),
    "moe_router_packed": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_router_from_logits_workspace_size": (_Z, [_I, _I]),
    "moe_router_from_logits": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_sinkhorn_workspace_size": (_Z, [_I, _I]),
    "moe_sinkhorn_bias": (_I, [_P, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_dispatch_rows": (_Z, [_I, _I, _I, _I]),
    "moe_tile_sched_bytes": (_Z, [_I, _I, _I, _I]),
    "moe_dispatch_workspace_size": (_Z, [_I, _I, _I, _I]),
    "moe_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_dispatch_static": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dense_tile_sched": (_I, [_I, _P, _P]),
    "moe_expert_choice_workspace_size": (_Z, [_I, _I]),
    "moe_expert_choice_route": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_choice_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_expert_choice_combine": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_packed_weights_bytes": (_Z, [_I, _I, _I, _I]),
    "moe_pack_expert_weights": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_expert_up_gate": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_expert_down": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_expert_up_gate_shared": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _I, _P, _P]),
    "moe_dispatch_fp8": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_up_gate_fp8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_dequant_fp8": (_I, [_P, _P, _I, _I, _P, _P]),
    "moe_combine_backward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_router_backward_workspace_size": (_Z, [_I, _I]),
    "moe_router_backward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _F, _P, _P, _P, _Z, _P]),
    "moe_router_weight_grad_workspace_size": (_Z, [_I, _I, _I]),
    "moe_router_weight_grad": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_dispatch_backward_workspace_size": (_Z, [_I, _I, _I, _I]),
    "moe_dispatch_backward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_packed_weights_backward_bytes": (_Z, [_I, _I, _I, _I]),
    "moe_pack_expert_weights_backward": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_expert_down_backward": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_expert_up_gate_backward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_expert_up_gate_save": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _P, _P, _P]),
    "moe_expert_up_gate_backward_saved": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_expert_weight_grads_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "moe_expert_weight_grads": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_down_shared": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _I, _P, _P]),
    "moe_expert_ffn_workspace_size": (_Z, [_I, _I, _I]),
    "moe_expert_ffn": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_combine_arrivals_bytes": (_Z, [_I, _I]),
    "moe_expert_down_combine": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P]),
    "moe_layer_workspace_size": (_Z, [_P]),
    "moe_layer_host_workspace_size": (_Z, [_P]),
    "moe_layer_views_of": (_I, [_P, _P, _P]),
    "moe_layer_forward": (_I, [_P, _P, _P, _P, _Z, _P]),
    "moe_layer_forward_host": (_I, [_P, _I, _P, _P, _P, _Z, _P]),
    "moe_last_error_string": (ctypes.c_char_p, []),
    "moe_check_device_error": (_I, [_P]),
    "moe_set_wait_limit": (None, [_LL]),
    "moe_version": (ctypes.c_char_p, []),
    "moe_launch_count": (ctypes.c_ulonglong, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = sorted(_SIGS)
LIB_PATH = _LIB_PATH


class MoEError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[moe status {code}] {msg}")
        self.code = code


def _check(rc: int):
    if rc != MOE_OK:
        raise MoEError(rc, _lib.moe_last_error_string().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return MOE_F32
    if dt == torch.bfloat16:
        return MOE_BF16
    raise MoEError(MOE_ERR_UNSUPPORTED, f"dtype {dt}")


def _bytes_tensor(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------------------------------------ router

def moe_router_workspace_size(T, h, E, k, dtype) -> int:
    return _lib.moe_router_workspace_size(T, h, E, k, dtype)


def moe_pack_router_weight(w_r, packed=None, stream=None):
    """The router weight repacked once for moe_router_packed (bf16: W_r^T [E, h]; fp32: a copy of w_r)."""
    h, E = w_r.shape
    dt = dtype_code(w_r.dtype)
    if packed is None:
        packed = _bytes_tensor(_lib.moe_router_packed_bytes(h, E, dt), w_r.device)
    _check(_lib.moe_pack_router_weight(_ptr(w_r), h, E, dt, _ptr(packed), _stream(stream)))
    return packed


def moe_router(x, w_r, bias, k: int, gating: str | int = "softmax", alpha: float = 0.01, *, logits=None,
               topk_ids=None, gates=None, counts=None, f=None, P=None, aux=None, ws=None, stream=None,
               want_logits=True, w_packed=None):
    """moe_router, or moe_router_packed when `w_packed` (moe_pack_router_weight of w_r) is given; w_r then only
    supplies the shape."""
    T, h = x.shape
    E = w_r.shape[1]
    dev = x.device
    dt = dtype_code(x.dtype)
    g = GATING[gating] if isinstance(gating, str) else int(gating)
    if logits is None and want_logits:
        logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    gates = torch.empty((T, k), dtype=torch.float32, device=dev) if gates is None else gates
    counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None else counts
    f = torch.empty(E, dtype=torch.float32, device=dev) if f is None else f
    P = torch.empty(E, dtype=torch.float32, device=dev) if P is None else P
    aux = torch.empty(1, dtype=torch.float32, device=dev) if aux is None else aux
    need = moe_router_workspace_size(T, h, E, k, dt)
    ws = _bytes_tensor(need, dev) if ws is None else ws
    fn = _lib.moe_router if w_packed is None else _lib.moe_router_packed
    _check(fn(_ptr(x), _ptr(w_r if w_packed is None else w_packed), _ptr(bias), T, h, E, k, dt, g, alpha, _ptr(logits),
              _ptr(topk_ids), _ptr(gates), _ptr(counts), _ptr(f), _ptr(P), _ptr(aux), _ptr(ws), ws.numel(),
              _stream(stream)))
    return dict(logits=logits, ids=topk_ids, gates=gates, counts=counts, f=f, P=P, aux=aux)


def moe_router_from_logits(logits, bias, k: int, gating: str | int = "softmax", alpha: float = 0.01, *,
                           topk_ids=None, gates=None, counts=None, f=None, P=None, aux=None, ws=None, stream=None):
    T, E = logits.shape
    dev = logits.device
    g = GATING[gating] if isinstance(gating, str) else int(gating)
    topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    gates = torch.empty((T, k), dtype=torch.float32, device=dev) if gates is None else gates
    counts = torch.empty(E, dtype=torch.int32, device=dev) if counts is None else counts
    f = torch.empty(E, dtype=torch.float32, device=dev) if f is None else f
    P = torch.empty(E, dtype=torch.float32, device=dev) if P is None else P
    aux = torch.empty(1, dtype=torch.float32, device=dev) if aux is None else aux
    ws = _bytes_tensor(_lib.moe_router_from_logits_workspace_size(T, E), dev) if ws is None else ws
    _check(_lib.moe_router_from_logits(_ptr(logits), _ptr(bias), T, E, k, g, alpha, _ptr(topk_ids), _ptr(gates),
                                       _ptr(counts), _ptr(f), _ptr(P), _ptr(aux), _ptr(ws), ws.numel(),
                                       _stream(stream)))
    return dict(ids=topk_ids, gates=gates, counts=counts, f=f, P=P, aux=aux)


def moe_sinkhorn_bias(logits, n_iter: int = 16, *, sel_bias=None, ws=None, stream=None):
    T, E = logits.shape
    dev = logits.device
    sel_bias = torch.empty(E, dtype=torch.float32, device=dev) if sel_bias is None else sel_bias
    ws = _bytes_tensor(_lib.moe_sinkhorn_workspace_size(T, E), dev) if ws is None else ws
    _check(_lib.moe_sinkhorn_bias(_ptr(logits), T, E, n_iter, _ptr(sel_bias), _ptr(ws), ws.numel(), _stream(stream)))
    return sel_bias


# ---------------------------------------------------------------------------------------------- dispatch

def moe_dispatch_rows(T, E, k, capacity) -> int:
    return _lib.moe_dispatch_rows(T, E, k, capacity)


def moe_tile_sched_bytes(T, E, k, capacity) -> int:
    return _lib.moe_tile_sched_bytes(T, E, k, capacity)


def moe_dispatch_workspace_size(T, E, k, capacity) -> int:
    return _lib.moe_dispatch_workspace_size(T, E, k, capacity)


def moe_dispatch(x, topk_ids, E: int, capacity: int = 0, num_ranks: int = 1, *, out=None, ws=None, stream=None):
    """Returns dict(buf, offsets, kept_counts, dest_row, drop_mask, src_token, src_slot, rank_counts,
    rank_offsets, tile_sched). `out` may hold preallocated tensors under those names."""
    T, h = x.shape
    k = topk_ids.shape[1]
    dev = x.device
    dt = dtype_code(x.dtype)
    rows = moe_dispatch_rows(T, E, k, capacity)
    o = dict(out or {})
    o.setdefault("buf", torch.empty((rows, h), dtype=x.dtype, device=dev))
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("kept_counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("dest_row", torch.empty((T, k), dtype=torch.int32, device=dev))
    o.setdefault("drop_mask", torch.empty((T, k), dtype=torch.uint8, device=dev))
    o.setdefault("src_token", torch.empty(rows, dtype=torch.int32, device=dev))
    o.setdefault("src_slot", torch.empty(rows, dtype=torch.int32, device=dev))
    o.setdefault("rank_counts", torch.empty(num_ranks, dtype=torch.int32, device=dev))
    o.setdefault("rank_offsets", torch.empty(num_ranks + 1, dtype=torch.int32, device=dev))
    o.setdefault("tile_sched", torch.empty(moe_tile_sched_bytes(T, E, k, capacity) // 4, dtype=torch.int32,
                                           device=dev))
    need = moe_dispatch_workspace_size(T, E, k, capacity)
    ws = _bytes_tensor(need, dev) if ws is None else ws
    _check(_lib.moe_dispatch(_ptr(x), _ptr(topk_ids), T, h, E, k, capacity, num_ranks, dt, _ptr(o["buf"]),
                             _ptr(o["offsets"]), _ptr(o["kept_counts"]), _ptr(o["dest_row"]), _ptr(o["drop_mask"]),
                             _ptr(o["src_token"]), _ptr(o["src_slot"]), _ptr(o["rank_counts"]),
                             _ptr(o["rank_offsets"]), _ptr(o["tile_sched"]), _ptr(ws), ws.numel(), _stream(stream)))
    o["rows"] = rows
    return o


def moe_dispatch_fp8(x, topk_ids, E: int, capacity: int = 0, num_ranks: int = 1, *, out=None, ws=None, stream=None):
    """moe_dispatch with the send buffer in FP8: returns dict(buf8 [rows, h] uint8 e4m3 codes, scales [rows, h/128]
    fp32, and every index output of moe_dispatch). `out` may hold preallocated tensors under those names."""
    T, h = x.shape
    k = topk_ids.shape[1]
    dev = x.device
    rows = moe_dispatch_rows(T, E, k, capacity)
    o = dict(out or {})
    o.setdefault("buf8", torch.empty((rows, h), dtype=torch.uint8, device=dev))
    o.setdefault("scales", torch.empty((rows, h // 128), dtype=torch.float32, device=dev))
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("kept_counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("dest_row", torch.empty((T, k), dtype=torch.int32, device=dev))
    o.setdefault("drop_mask", torch.empty((T, k), dtype=torch.uint8, device=dev))
    o.setdefault("src_token", torch.empty(rows, dtype=torch.int32, device=dev))
    o.setdefault("src_slot", torch.empty(rows, dtype=torch.int32, device=dev))
    o.setdefault("rank_counts", torch.empty(num_ranks, dtype=torch.int32, device=dev))
    o.setdefault("rank_offsets", torch.empty(num_ranks + 1, dtype=torch.int32, device=dev))
    o.setdefault("tile_sched", torch.empty(moe_tile_sched_bytes(T, E, k, capacity) // 4, dtype=torch.int32,
                                           device=dev))
    ws = _bytes_tensor(moe_dispatch_workspace_size(T, E, k, capacity), dev) if ws is None else ws
    _check(_lib.moe_dispatch_fp8(_ptr(x), _ptr(topk_ids), T, h, E, k, capacity, num_ranks, _ptr(o["buf8"]),
                                 _ptr(o["scales"]), _ptr(o["offsets"]), _ptr(o["kept_counts"]), _ptr(o["dest_row"]),
                                 _ptr(o["drop_mask"]), _ptr(o["src_token"]), _ptr(o["src_slot"]), _ptr(o["rank_counts"]),
                                 _ptr(o["rank_offsets"]), _ptr(o["tile_sched"]), _ptr(ws), ws.numel(), _stream(stream)))
    o["rows"] = rows
    return o


def moe_expert_up_gate_fp8(buf8, scales, tile_sched, packed_w, E: int, F: int, act=None, stream=None):
    rows, h = buf8.shape
    if act is None:
        act = torch.empty((rows, F), dtype=torch.bfloat16, device=buf8.device)
    _check(_lib.moe_expert_up_gate_fp8(_ptr(buf8), _ptr(scales), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows,
                                       _ptr(act), _stream(stream)))
    return act


def moe_dequant_fp8(buf8, scales, out=None, stream=None):
    rows, h = buf8.shape
    out = torch.empty((rows, h), dtype=torch.bfloat16, device=buf8.device) if out is None else out
    _check(_lib.moe_dequant_fp8(_ptr(buf8), _ptr(scales), rows, h, _ptr(out), _stream(stream)))
    return out


def moe_dispatch_static(x, topk_ids, E: int, capacity: int = 0, num_ranks: int = 1, *, out=None, stream=None):
    """moe_dispatch without a workspace: the library's fixed device scratch is used (for callers that cannot
    allocate device memory). Outputs as moe_dispatch; `out` may hold preallocated output tensors."""
    T, h = x.shape
    k = topk_ids.shape[1]
    dev = x.device
    rows = moe_dispatch_rows(T, E, k, capacity)
    o = dict(out or {})
    o.setdefault("buf", torch.empty((rows, h), dtype=x.dtype, device=dev))
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("kept_counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("dest_row", torch.empty((T, k), dtype=torch.int32, device=dev))
    o.setdefault("drop_mask", torch.empty((T, k), dtype=torch.uint8, device=dev))
    o.setdefault("src_token", torch.empty(rows, dtype=torch.int32, device=dev))
    o.setdefault("src_slot", torch.empty(rows, dtype=torch.int32, device=dev))
    o.setdefault("rank_counts", torch.empty(num_ranks, dtype=torch.int32, device=dev))
    o.setdefault("rank_offsets", torch.empty(num_ranks + 1, dtype=torch.int32, device=dev))
    o.setdefault("tile_sched", torch.empty(moe_tile_sched_bytes(T, E, k, capacity) // 4, dtype=torch.int32,
                                           device=dev))
    _check(_lib.moe_dispatch_static(_ptr(x), _ptr(topk_ids), T, h, E, k, capacity, num_ranks, dtype_code(x.dtype),
                                    _ptr(o["buf"]), _ptr(o["offsets"]), _ptr(o["kept_counts"]), _ptr(o["dest_row"]),
                                    _ptr(o["drop_mask"]), _ptr(o["src_token"]), _ptr(o["src_slot"]),
                                    _ptr(o["rank_counts"]), _ptr(o["rank_offsets"]), _ptr(o["tile_sched"]),
                                    _stream(stream)))
    o["rows"] = rows
    return o


def moe_dense_tile_sched(rows: int, tile_sched=None, device="cuda", stream=None):
    if tile_sched is None:
        tile_sched = torch.empty(moe_tile_sched_bytes(rows, 1, 1, 0) // 4, dtype=torch.int32, device=device)
    _check(_lib.moe_dense_tile_sched(rows, _ptr(tile_sched), _stream(stream)))
    return tile_sched


# ---------------------------------------------------------------------------------------- expert choice

def moe_expert_choice_workspace_size(T, E) -> int:
    return _lib.moe_expert_choice_workspace_size(T, E)


def moe_expert_choice_route(logits, C: int, *, tokens=None, gates=None, slot=None, ws=None, stream=None):
    T, E = logits.shape
    dev = logits.device
    tokens = torch.empty((E, C), dtype=torch.int32, device=dev) if tokens is None else tokens
    gates = torch.empty((E, C), dtype=torch.float32, device=dev) if gates is None else gates
    slot = torch.empty((T, E), dtype=torch.int32, device=dev) if slot is None else slot
    ws = _bytes_tensor(moe_expert_choice_workspace_size(T, E), dev) if ws is None else ws
    _check(_lib.moe_expert_choice_route(_ptr(logits), T, E, C, _ptr(tokens), _ptr(gates), _ptr(slot), _ptr(ws),
                                        ws.numel(), _stream(stream)))
    return dict(tokens=tokens, gates=gates, slot=slot)


def moe_expert_choice_dispatch(x, tokens, *, buf=None, tile_sched=None, stream=None):
    T, h = x.shape
    E, C = tokens.shape
    if buf is None:
        buf = torch.empty((E * C, h), dtype=x.dtype, device=x.device)
    if tile_sched is None:
        tile_sched = torch.empty(moe_tile_sched_bytes(T, E, 1, C) // 4, dtype=torch.int32, device=x.device)
    _check(_lib.moe_expert_choice_dispatch(_ptr(x), _ptr(tokens), T, h, E, C, dtype_code(x.dtype), _ptr(buf),
                                           _ptr(tile_sched), _stream(stream)))
    return dict(buf=buf, tile_sched=tile_sched)


def moe_expert_choice_combine(eout, slot, gates, shared_out=None, y=None, stream=None):
    T, E = slot.shape
    C = gates.shape[1]
    h = eout.shape[1]
    if y is None:
        y = torch.empty((T, h), dtype=eout.dtype, device=eout.device)
    _check(_lib.moe_expert_choice_combine(_ptr(eout), _ptr(slot), _ptr(gates), _ptr(shared_out), T, h, E, C,
                                          dtype_code(eout.dtype), _ptr(y), _stream(stream)))
    return y


# ------------------------------------------------------------------------------------------------ experts

def moe_packed_weights_bytes(E, h, F, dtype) -> int:
    return _lib.moe_packed_weights_bytes(E, h, F, dtype)


def moe_pack_expert_weights(w_gate, w_up, w_down, packed=None, stream=None):
    E, F, h = w_gate.shape
    dt = dtype_code(w_gate.dtype)
    if packed is None:
        packed = _bytes_tensor(moe_packed_weights_bytes(E, h, F, dt), w_gate.device)
    _check(_lib.moe_pack_expert_weights(_ptr(w_gate), _ptr(w_up), _ptr(w_down), E, h, F, dt, _ptr(packed),
                                        _stream(stream)))
    return packed


def moe_expert_up_gate(buf, tile_sched, packed_w, E: int, F: int, act=None, stream=None):
    rows, h = buf.shape
    if act is None:
        act = torch.empty((rows, F), dtype=buf.dtype, device=buf.device)
    _check(_lib.moe_expert_up_gate(_ptr(buf), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows, dtype_code(buf.dtype),
                                   _ptr(act), _stream(stream)))
    return act


def moe_expert_up_gate_shared(buf, tile_sched, packed_w, E: int, F: int, x, packed_shared, act=None, act_shared=None,
                              stream=None):
    """Routed up/gate GEMM and the shared expert's (x -> act_shared) in one launch (bf16)."""
    rows, h = buf.shape
    T = x.shape[0]
    if act is None:
        act = torch.empty((rows, F), dtype=buf.dtype, device=buf.device)
    if act_shared is None:
        act_shared = torch.empty((T, F), dtype=buf.dtype, device=buf.device)
    _check(_lib.moe_expert_up_gate_shared(_ptr(buf), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows, _ptr(x), T,
                                          _ptr(packed_shared), _ptr(act_shared), dtype_code(buf.dtype), _ptr(act),
                                          _stream(stream)))
    return act, act_shared


def moe_expert_down_shared(act, tile_sched, packed_w, E: int, h: int, act_shared, packed_shared, eout=None,
                           out_shared=None, stream=None):
    """Routed down GEMM and the shared expert's (act_shared -> out_shared) in one launch (bf16)."""
    rows, F = act.shape
    T = act_shared.shape[0]
    if eout is None:
        eout = torch.empty((rows, h), dtype=act.dtype, device=act.device)
    if out_shared is None:
        out_shared = torch.empty((T, h), dtype=act.dtype, device=act.device)
    _check(_lib.moe_expert_down_shared(_ptr(act), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows, _ptr(act_shared),
                                       T, _ptr(packed_shared), _ptr(out_shared), dtype_code(act.dtype), _ptr(eout),
                                       _stream(stream)))
    return eout, out_shared


def moe_expert_down(act, tile_sched, packed_w, E: int, h: int, eout=None, stream=None):
    rows, F = act.shape
    if eout is None:
        eout = torch.empty((rows, h), dtype=act.dtype, device=act.device)
    _check(_lib.moe_expert_down(_ptr(act), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows, dtype_code(act.dtype),
                                _ptr(eout), _stream(stream)))
    return eout


def moe_expert_ffn_workspace_size(rows, F, dtype) -> int:
    return _lib.moe_expert_ffn_workspace_size(rows, F, dtype)


def moe_expert_ffn(buf, tile_sched, packed_w, E: int, F: int, eout=None, ws=None, stream=None):
    rows, h = buf.shape
    dt = dtype_code(buf.dtype)
    if eout is None:
        eout = torch.empty((rows, h), dtype=buf.dtype, device=buf.device)
    need = moe_expert_ffn_workspace_size(rows, F, dt)
    ws = _bytes_tensor(need, buf.device) if ws is None else ws
    _check(_lib.moe_expert_ffn(_ptr(buf), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows, dt, _ptr(eout), _ptr(ws),
                               ws.numel(), _stream(stream)))
    return eout


# ------------------------------------------------------------------------------------------------ combine

def moe_combine(eout, dest_row, gates, shared_out=None, y=None, stream=None):
    T, k = dest_row.shape
    h = eout.shape[1]
    if y is None:
        y = torch.empty((T, h), dtype=eout.dtype, device=eout.device)
    _check(_lib.moe_combine(_ptr(eout), _ptr(dest_row), _ptr(gates), _ptr(shared_out), T, h, k,
                            dtype_code(eout.dtype), _ptr(y), _stream(stream)))
    return y


def moe_combine_arrivals(T: int, h: int, device) -> torch.Tensor:
    """Zeroed arrival counters of moe_expert_down_combine (int32, moe_combine_arrivals_bytes of them)."""
    return torch.zeros(max(1, _lib.moe_combine_arrivals_bytes(T, h) // 4), dtype=torch.int32, device=device)


def moe_expert_down_combine(act, tile_sched, packed_w, E: int, h: int, src_token, dest_row, gates, arrivals,
                            act_shared=None, packed_shared=None, eout=None, out_shared=None, y=None, stream=None):
    """Down GEMM (routed and, with act_shared, the shared expert's rows) with the combine in its epilogue (bf16):
    returns (eout, out_shared or None, y), y bit-identical to moe_combine on those eout / out_shared."""
    rows, F = act.shape
    T, k = dest_row.shape
    dev = act.device
    if eout is None:
        eout = torch.empty((rows, h), dtype=act.dtype, device=dev)
    if act_shared is not None and out_shared is None:
        out_shared = torch.empty((T, h), dtype=act.dtype, device=dev)
    if y is None:
        y = torch.empty((T, h), dtype=act.dtype, device=dev)
    _check(_lib.moe_expert_down_combine(_ptr(act), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows, _ptr(src_token),
                                        _ptr(dest_row), _ptr(gates), T, k, _ptr(act_shared), _ptr(packed_shared),
                                        dtype_code(act.dtype), _ptr(eout), _ptr(out_shared), _ptr(y), _ptr(arrivals),
                                        _stream(stream)))
    return eout, out_shared, y


# ------------------------------------------------------------------------------------------------ layer

class MoELayerDesc(ctypes.Structure):
    """struct moe_layer_desc: the layer's sizes, modes and device-resident parameters."""
    _fields_ = [("T", _I), ("h", _I), ("E", _I), ("k", _I), ("F", _I), ("dtype", _I), ("gating", _I),
                ("alpha", _F), ("capacity", _I), ("num_ranks", _I), ("w_r_packed", _P), ("bias", _P),
                ("packed_w", _P), ("packed_shared", _P), ("routing", _I), ("payload", _I), ("sinkhorn_iters", _I)]


class MoELayerViews(ctypes.Structure):
    """struct moe_layer_views: device addresses of the intermediates inside a layer workspace."""
    _fields_ = [(n, _P) for n in ("logits", "topk_ids", "gates", "counts", "f", "P", "aux", "buf", "offsets",
                                  "kept_counts", "dest_row", "drop_mask", "src_token", "src_slot", "rank_counts",
                                  "rank_offsets", "tile_sched", "act", "eout", "act_shared", "out_shared")] + \
              [("rows", _LL)] + [(n, _P) for n in ("ec_tokens", "ec_gates", "ec_slot", "sel_bias", "buf8", "scales")]


ROUTING = {"token": 0, "expert_choice": 1, "sinkhorn": 2}
PAYLOAD = {"dtype": 0, "bf16": 0, "f32": 0, "fp8": 1}


def moe_layer_desc(*, T, h, E, k, F, dtype, gating, alpha, capacity, num_ranks, w_r_packed, bias, packed_w,
                   packed_shared=None, routing="token", payload="dtype", sinkhorn_iters=0) -> MoELayerDesc:
    """The descriptor of a layer whose parameters are the given device tensors (kept alive by the caller)."""
    g = GATING[gating] if isinstance(gating, str) else int(gating)
    d = MoELayerDesc(T, h, E, k, F, dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype), g,
                     float(alpha), capacity, num_ranks, _ptr(w_r_packed), _ptr(bias), _ptr(packed_w),
                     _ptr(packed_shared), ROUTING[routing] if isinstance(routing, str) else int(routing),
                     PAYLOAD[payload] if isinstance(payload, str) else int(payload), int(sinkhorn_iters))
    return d


def moe_layer_workspace_size(desc: MoELayerDesc) -> int:
    return _lib.moe_layer_workspace_size(ctypes.byref(desc))


def moe_layer_host_workspace_size(desc: MoELayerDesc) -> int:
    return _lib.moe_layer_host_workspace_size(ctypes.byref(desc))


def moe_layer_views_of(desc: MoELayerDesc, ws) -> MoELayerViews:
    v = MoELayerViews()
    _check(_lib.moe_layer_views_of(ctypes.byref(desc), _ptr(ws), ctypes.byref(v)))
    return v


def moe_layer_forward(desc: MoELayerDesc, x, y, ws, stream=None):
    _check(_lib.moe_layer_forward(ctypes.byref(desc), _ptr(x), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)))
    return y


def moe_layer_forward_host(desc: MoELayerDesc, x_hosts, y_hosts, ws, stream=None):
    """x_hosts[i] -> y_hosts[i]: page-locked host tensors of the layer's shape (any dtype of the same bytes).
    Enqueues everything on the stream and returns; synchronise the stream before reading y_hosts."""
    n = len(x_hosts)
    if len(y_hosts) != n:
        raise MoEError(MOE_ERR_INVALID_ARG, "x_hosts and y_hosts differ in length")
    xs = (_P * max(n, 1))(*[t.data_ptr() for t in x_hosts])
    ys = (_P * max(n, 1))(*[t.data_ptr() for t in y_hosts])
    _check(_lib.moe_layer_forward_host(ctypes.byref(desc), n, xs, ys, _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)))
    return y_hosts


# ------------------------------------------------------------------------------------------------ errors

def moe_last_error_string() -> str:
    return _lib.moe_last_error_string().decode(errors="replace")


def moe_check_device_error(stream=None) -> int:
    return _lib.moe_check_device_error(_stream(stream))


def moe_set_wait_limit(spins: int):
    _lib.moe_set_wait_limit(int(spins))


def moe_launch_count() -> int:
    return int(_lib.moe_launch_count())


def moe_version() -> str:
    return _lib.moe_version().decode()


def raw_lib():
    """The ctypes handle (tests call entry points with raw pointers through it)."""
    return _lib


# ------------------------------------------------------------------------------------------------ backward

def moe_combine_backward(dy, eout, src_token, src_slot, dest_row, gates, d_eout=None, d_gates=None, stream=None):
    T, h = dy.shape
    rows = eout.shape[0]
    k = dest_row.shape[1]
    if d_eout is None:
        d_eout = torch.empty((rows, h), dtype=dy.dtype, device=dy.device)
    if d_gates is None:
        d_gates = torch.empty((T, k), dtype=torch.float32, device=dy.device)
    _check(_lib.moe_combine_backward(_ptr(dy), _ptr(eout), _ptr(src_token), _ptr(src_slot), _ptr(dest_row),
                                     _ptr(gates), T, h, k, rows, dtype_code(dy.dtype), _ptr(d_eout), _ptr(d_gates),
                                     _stream(stream)))
    return d_eout, d_gates


def moe_router_backward(logits, topk_ids, gates, d_gates, f, gating, alpha: float = 0.01, d_aux: float = 1.0, *,
                        d_logits=None, want_bias_grad=True, ws=None, stream=None):
    T, E = logits.shape
    k = topk_ids.shape[1]
    g = GATING[gating] if isinstance(gating, str) else int(gating)
    if d_logits is None:
        d_logits = torch.empty((T, E), dtype=torch.float32, device=logits.device)
    d_bias = torch.empty(E, dtype=torch.float32, device=logits.device) if want_bias_grad else None
    if ws is None:
        ws = _bytes_tensor(_lib.moe_router_backward_workspace_size(T, E), logits.device)
    _check(_lib.moe_router_backward(_ptr(logits), _ptr(topk_ids), _ptr(gates), _ptr(d_gates), _ptr(f), T, E, k, g,
                                    alpha, d_aux, _ptr(d_logits), _ptr(d_bias), _ptr(ws), ws.numel(),
                                    _stream(stream)))
    return d_logits, d_bias


def moe_router_weight_grad(x, d_logits, dW_r=None, ws=None, stream=None):
    T, h = x.shape
    E = d_logits.shape[1]
    if dW_r is None:
        dW_r = torch.empty((h, E), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _bytes_tensor(_lib.moe_router_weight_grad_workspace_size(T, h, E), x.device)
    _check(_lib.moe_router_weight_grad(_ptr(x), _ptr(d_logits), T, h, E, dtype_code(x.dtype), _ptr(dW_r), _ptr(ws),
                                       ws.numel(), _stream(stream)))
    return dW_r


def moe_dispatch_backward(d_buf, dest_row, d_logits, w_r, dx_extra=None, dx=None, ws=None, stream=None):
    T, k = dest_row.shape
    h = d_buf.shape[1]
    E = w_r.shape[1]
    if dx is None:
        dx = torch.empty((T, h), dtype=d_buf.dtype, device=d_buf.device)
    if ws is None and d_logits is not None:
        ws = _bytes_tensor(_lib.moe_dispatch_backward_workspace_size(T, h, E, dtype_code(d_buf.dtype)), d_buf.device)
    _check(_lib.moe_dispatch_backward(_ptr(d_buf), _ptr(dest_row), _ptr(d_logits), _ptr(w_r), _ptr(dx_extra), T, h, k,
                                      E, dtype_code(d_buf.dtype), _ptr(dx), _ptr(ws),
                                      ws.numel() if ws is not None else 0, _stream(stream)))
    return dx


def moe_pack_expert_weights_backward(w_gate, w_up, w_down, packed_bwd=None, stream=None):
    E, F, h = w_gate.shape
    dt = dtype_code(w_gate.dtype)
    if packed_bwd is None:
        packed_bwd = _bytes_tensor(_lib.moe_packed_weights_backward_bytes(E, h, F, dt), w_gate.device)
    _check(_lib.moe_pack_expert_weights_backward(_ptr(w_gate), _ptr(w_up), _ptr(w_down), E, h, F, dt, _ptr(packed_bwd),
                                                 _stream(stream)))
    return packed_bwd


def gu_cols(F: int) -> int:
    """Columns of d_gu: 2 * (F rounded up to 128)."""
    return 2 * ((F + 127) // 128 * 128)


def moe_expert_down_backward(d_eout, tile_sched, packed_bwd, E: int, F: int, d_act=None, stream=None):
    rows, h = d_eout.shape
    if d_act is None:
        d_act = torch.empty((rows, F), dtype=d_eout.dtype, device=d_eout.device)
    _check(_lib.moe_expert_down_backward(_ptr(d_eout), _ptr(tile_sched), _ptr(packed_bwd), E, h, F, rows,
                                         dtype_code(d_eout.dtype), _ptr(d_act), _stream(stream)))
    return d_act


def moe_expert_up_gate_backward(buf, d_act, tile_sched, packed_w, packed_bwd, E: int, d_gu=None, d_buf=None,
                                stream=None):
    rows, h = buf.shape
    F = d_act.shape[1]
    if d_gu is None:
        d_gu = torch.empty((rows, gu_cols(F)), dtype=buf.dtype, device=buf.device)
    if d_buf is None:
        d_buf = torch.empty((rows, h), dtype=buf.dtype, device=buf.device)
    _check(_lib.moe_expert_up_gate_backward(_ptr(buf), _ptr(d_act), _ptr(tile_sched), _ptr(packed_w), _ptr(packed_bwd),
                                            E, h, F, rows, dtype_code(buf.dtype), _ptr(d_gu), _ptr(d_buf),
                                            _stream(stream)))
    return d_gu, d_buf


def moe_expert_up_gate_save(buf, tile_sched, packed_w, E: int, F: int, *, x=None, packed_shared=None, act=None,
                            gu=None, act_shared=None, gu_shared=None, stream=None):
    """act and the saved pre-activations gu [rows, gu_cols(F)] (and the shared expert's with packed_shared)."""
    rows, h = buf.shape
    dev = buf.device
    T = x.shape[0] if (x is not None and packed_shared is not None) else 0
    act = torch.empty((rows, F), dtype=buf.dtype, device=dev) if act is None else act
    gu = torch.empty((rows, gu_cols(F)), dtype=buf.dtype, device=dev) if gu is None else gu
    if T:
        act_shared = torch.empty((T, F), dtype=buf.dtype, device=dev) if act_shared is None else act_shared
        gu_shared = torch.empty((T, gu_cols(F)), dtype=buf.dtype, device=dev) if gu_shared is None else gu_shared
    _check(_lib.moe_expert_up_gate_save(_ptr(buf), _ptr(tile_sched), _ptr(packed_w), E, h, F, rows,
                                        _ptr(x) if T else None, T, _ptr(packed_shared) if T else None,
                                        _ptr(act_shared) if T else None, _ptr(gu_shared) if T else None,
                                        dtype_code(buf.dtype), _ptr(act), _ptr(gu), _stream(stream)))
    return act, gu, act_shared, gu_shared


def moe_expert_up_gate_backward_saved(gu, d_act, tile_sched, packed_bwd, E: int, h: int, d_gu=None, d_buf=None,
                                      stream=None):
    rows, F = d_act.shape
    dev = d_act.device
    d_gu = torch.empty((rows, gu_cols(F)), dtype=d_act.dtype, device=dev) if d_gu is None else d_gu
    d_buf = torch.empty((rows, h), dtype=d_act.dtype, device=dev) if d_buf is None else d_buf
    _check(_lib.moe_expert_up_gate_backward_saved(_ptr(gu), _ptr(d_act), _ptr(tile_sched), _ptr(packed_bwd), E, h, F,
                                                  rows, dtype_code(d_act.dtype), _ptr(d_gu), _ptr(d_buf),
                                                  _stream(stream)))
    return d_gu, d_buf


def moe_expert_weight_grads(buf, act, d_gu, d_eout, offsets, kept_counts, E: int, dW_gate=None, dW_up=None,
                            dW_down=None, ws=None, stream=None):
    rows, h = buf.shape
    F = act.shape[1]
    dev = buf.device
    f32 = torch.float32
    dW_gate = torch.empty((E, F, h), dtype=f32, device=dev) if dW_gate is None else dW_gate
    dW_up = torch.empty((E, F, h), dtype=f32, device=dev) if dW_up is None else dW_up
    dW_down = torch.empty((E, h, F), dtype=f32, device=dev) if dW_down is None else dW_down
    if ws is None:
        ws = _bytes_tensor(_lib.moe_expert_weight_grads_workspace_size(E, h, F, rows, dtype_code(buf.dtype)), dev)
    _check(_lib.moe_expert_weight_grads(_ptr(buf), _ptr(act), _ptr(d_gu), _ptr(d_eout), _ptr(offsets),
                                        _ptr(kept_counts), E, h, F, rows, dtype_code(buf.dtype), _ptr(dW_gate),
                                        _ptr(dW_up), _ptr(dW_down), _ptr(ws), ws.numel(), _stream(stream)))
    return dW_gate, dW_up, dW_down

