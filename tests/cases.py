"""Shared test helpers: seeded inputs for a workload, the oracle's answer, and (on a GPU) the CUDA path's.

Inputs come from moe_inputs; the expected values come from oracle/ only. Rows of x whose top-k selection
has an oracle score gap below 1e-5 are redrawn from their own substream until none is left, so that the
fp32 GPU router and the fp64 oracle must agree on every index (gaps below 1e-6 are counted and reported).
"""
from __future__ import annotations

import numpy as np

import moe_inputs
from oracle import moe_oracle as O

REDRAW_GAP = 1e-5
REPORT_GAP = 1e-6


def router_inputs(cfg, seed=0, bias=None):
    """x (with near-tie rows redrawn), w_r, bias, the oracle's routing, and the redraw record.

    Sinkhorn routing couples all tokens through the column scalings (redrawing one row moves every score by
    ~1e-4), so for it the whole input is redrawn instead: the first seed >= `seed` whose balanced scores have
    no gap below 1e-5."""
    if cfg.routing == "sinkhorn":
        w_r, b = moe_inputs.make_router(cfg, seed, bias=bias)
        w64 = moe_inputs.to_f64(w_r, cfg.dtype)
        for s in range(seed, seed + 200):
            x = moe_inputs.make_x(cfg, s)
            L = O.router_logits(moe_inputs.to_f64(x, cfg.dtype), w64, b, O.SOFTMAX)
            r = O.route_sinkhorn(L, cfg.k, alpha=cfg.alpha)
            if O.near_tie_rows(r["gaps"], REDRAW_GAP).size == 0:
                return dict(x=x, w_r=w_r, bias=b, route=r, redrawn=0, x_seed=s,
                            near_ties=int((r["gaps"] < REPORT_GAP).sum()))
        raise RuntimeError("no near-tie-free input among 200 seeds")
    w_r, b = moe_inputs.make_router(cfg, seed, bias=bias)
    w64 = moe_inputs.to_f64(w_r, cfg.dtype)
    redraw: dict[int, int] = {}
    x = moe_inputs.make_x(cfg, seed)
    for _ in range(8):
        if cfg.routing == "sinkhorn":           # logits with the bias added, then Sinkhorn-balanced top-k
            L = O.router_logits(moe_inputs.to_f64(x, cfg.dtype), w64, b, O.SOFTMAX)
            r = O.route_sinkhorn(L, cfg.k, alpha=cfg.alpha)
        else:
            L = O.router_logits(moe_inputs.to_f64(x, cfg.dtype), w64, b, cfg.gating)
            r = O.route(L, cfg.k, cfg.gating, b, cfg.alpha)
        close = O.near_tie_rows(r["gaps"], REDRAW_GAP)
        if close.size == 0:
            break
        for t in close.tolist():
            redraw[t] = redraw.get(t, 0) + 1
        x = moe_inputs.make_x(cfg, seed, redraw=redraw)
    else:
        raise RuntimeError("near ties persist after 8 redraw rounds")
    near = int((r["gaps"] < REPORT_GAP).sum())
    return dict(x=x, w_r=w_r, bias=b, route=r, redrawn=len(redraw), near_ties=near)


def oracle_layer(cfg, inp, weights_fn, shared_fn=None, full_ffn=True):
    """Router, dispatch and (when full_ffn) the whole layer from the oracle."""
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    r = inp["route"]
    C = O.capacity(cfg.cf, cfg.k, cfg.T, cfg.E)
    d = O.dispatch(r["ids"], cfg.E, C, cfg.R)
    out = dict(route=r, disp=d, C=C)
    if full_ffn:
        buf = O.dispatch_payload(x64, d)
        eout = O.expert_outputs(buf, d, weights_fn)
        sh = O.swiglu_ffn(x64, *shared_fn()) if shared_fn else None
        out.update(buf=buf, eout=eout, shared_out=sh, y=O.combine(eout, d["dest_row"], r["gates"], sh))
    return out


def weights_fn_from(cfg, wg, wu, wd):
    def f(e):
        return (moe_inputs.to_f64(wg[e], cfg.dtype), moe_inputs.to_f64(wu[e], cfg.dtype),
                moe_inputs.to_f64(wd[e], cfg.dtype))
    return f


def torch_dtype(cfg):
    import torch
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def to_device(a, cfg, device="cuda"):
    """Upload a stored tensor (float32 or bf16 bit patterns) as a torch tensor of the working dtype."""
    import torch
    if cfg.dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def from_device(t, cfg):
    """Download a working-dtype tensor to float64 numpy."""
    import torch
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return moe_inputs.to_f64(bits, "bf16")
    return t.detach().cpu().numpy().astype(np.float64)


def from_device_rows(t, mask, cfg):
    """Download the rows of a working-dtype tensor where `mask` (a device bool tensor) is set, as float64 numpy of
    the full shape with every other row zero (rows a kernel never writes hold whatever the allocator left, and
    are not converted)."""
    import torch
    out = torch.zeros_like(t)
    out[mask] = t[mask]
    return from_device(out, cfg)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def rel_max(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    m = np.max(np.abs(b)) if b.size else 0.0
    return float(np.max(np.abs(a - b)) / (m if m > 0 else 1.0)) if b.size else 0.0


def y_tolerance(cfg):
    """fp32: max|y - y_ref| / max|y_ref| <= 1e-5; bf16 with fp32 accumulation: ||y - y_ref|| / ||y_ref|| <= 2e-2."""
    return (rel_max, 1e-5) if cfg.dtype == "f32" else (rel_l2, 2e-2)


def build_gpu_layer(cfg, inp, wg, wu, wd, shared=None, device="cuda", backward=False, fuse_combine=False):
    import torch
    from top_routing_dispatch_moe_gb300.layer import MoELayer
    dev = torch.device(device)
    b = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
    sh = None
    if shared is not None:
        sh = tuple(to_device(np.ascontiguousarray(w)[None], cfg, dev) for w in shared)   # one expert: [1, ...]
    layer = MoELayer(T=cfg.T, h=cfg.h, E=cfg.E, k=cfg.k, F=cfg.F, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                     alpha=cfg.alpha, w_r=to_device(inp["w_r"], cfg, dev), bias=b, w_gate=to_device(wg, cfg, dev),
                     w_up=to_device(wu, cfg, dev), w_down=to_device(wd, cfg, dev), shared=sh, device=dev,
                     routing=cfg.routing, backward=backward, payload=cfg.payload, fuse_combine=fuse_combine)
    return layer


def ec_inputs(cfg, seed=0):
    """Inputs of an expert-choice workload. For every expert whose C-th and (C+1)-th best scores differ by
    less than 1e-5 (the oracle's float64 scores), the two boundary tokens are redrawn from their own
    substreams, until no expert's choice is that close."""
    w_r, _ = moe_inputs.make_router(cfg, seed)
    w64 = moe_inputs.to_f64(w_r, cfg.dtype)
    C = O.capacity(cfg.cf, cfg.k, cfg.T, cfg.E)
    redraw: dict[int, int] = {}
    x = moe_inputs.make_x(cfg, seed)
    for _ in range(8):
        L = O.router_logits(moe_inputs.to_f64(x, cfg.dtype), w64, None, O.SOFTMAX)
        ec = O.expert_choice(L, C)
        close = np.nonzero(ec["gaps"] < REDRAW_GAP)[0]
        if close.size == 0:
            break
        for e in close.tolist():
            order = np.argsort(-ec["prob"][:, e], kind="stable")
            for t in (int(order[C - 1]), int(order[C])):
                redraw[t] = redraw.get(t, 0) + 1
        x = moe_inputs.make_x(cfg, seed, redraw=redraw)
    else:
        raise RuntimeError("expert-choice near ties persist after 8 redraw rounds")
    return dict(x=x, w_r=w_r, bias=None, C=C, logits=L, ec=ec, redrawn=len(redraw),
                near_ties=int((ec["gaps"] < REPORT_GAP).sum()))
