"""One MoE layer forward over preallocated device buffers, chaining the four C-ABI calls.

router ("Megatron-LM 分布式训练（六）", section "Router") -> dispatch ("v6 长序列和 MoE", table row
"dispatch") -> grouped SwiGLU expert FFN (table row "expert"; shared expert per the data flow of the
Megatron page) -> combine (table row "combine"). All work is enqueued on one stream with no host sync.
"""
from __future__ import annotations

import math

import torch

from . import moe


def capacity_slots(cf: float, k: int, T: int, E: int) -> int:
    """Per-expert capacity C = cf * k * T / E rounded up ("v6 长序列和 MoE", "Capacity" bullet); 0 = dropless."""
    if cf <= 0:
        return 0
    return int(math.ceil(cf * k * T / E - 1e-9))


class MoELayer:
    """Holds the packed expert weights, the router weight and every intermediate buffer of one layer.

    Stages (in order): "router", "dispatch", "up_gate", "down", ["shared_up_gate", "shared_down"], "combine". With
    bf16 the shared expert runs inside the "up_gate" and "down" launches; the two shared stages exist for fp32.
    forward(x, events=...) records one CUDA event before the first stage and after each stage when given
    a dict of lists, so callers can time the stages on the launching stream. forward(x, save=True) (a layer built
    with backward=True, bf16 token-choice or Sinkhorn routing, bf16 payload) also keeps the experts'
    pre-activations g and u, so that the next backward() needs no recompute of the up/gate GEMM."""

    STAGES = ("router", "dispatch", "up_gate", "down", "shared_up_gate", "shared_down", "combine")

    def __init__(self, *, T, h, E, k, F, gating, cf, R, alpha, w_r, bias, w_gate, w_up, w_down,
                 shared=None, device="cuda", routing="token", backward=False, payload="bf16", fuse_combine=False):
        self.T, self.h, self.E, self.k, self.F = T, h, E, k, F
        self.gating, self.R, self.alpha = gating, R, alpha
        self.C = capacity_slots(cf, k, T, E)
        self.dtype = w_r.dtype
        dt = self.dtype
        dev = torch.device(device)
        self.device = dev
        self.w_r = w_r
        self.w_r_packed = moe.moe_pack_router_weight(w_r)    # the router's operand layout, packed once
        self.bias = bias
        self.packed = moe.moe_pack_expert_weights(w_gate, w_up, w_down)
        self.shared_packed = moe.moe_pack_expert_weights(*shared) if shared is not None else None
        # the dgrad GEMMs' weight operands (only when the layer will run backward: twice the weight memory)
        self.packed_bwd = moe.moe_pack_expert_weights_backward(w_gate, w_up, w_down) if backward else None
        self.shared_packed_bwd = (moe.moe_pack_expert_weights_backward(*shared)
                                  if backward and shared is not None else None)
        self._bwd = None
        i32, f32 = torch.int32, torch.float32
        code = moe.dtype_code(dt)
        self.routing = routing
        if payload not in ("bf16", "fp8") or (payload == "fp8" and (routing != "token" or dt != torch.bfloat16)):
            raise ValueError("payload: 'bf16', or 'fp8' with token-choice routing in bf16")
        self.payload = payload
        if routing == "expert_choice":
            # every expert takes C = cf * k * T / E tokens (k: the average number of experts per token)
            self.rows = E * self.C
            self.ec = dict(tokens=torch.empty((E, self.C), dtype=i32, device=dev),
                           gates=torch.empty((E, self.C), dtype=f32, device=dev),
                           slot=torch.empty((T, E), dtype=i32, device=dev))
            self.ec_ws = moe._bytes_tensor(moe.moe_expert_choice_workspace_size(T, E), dev)
        else:
            self.rows = moe.moe_dispatch_rows(T, E, k, self.C)
        if routing == "sinkhorn":
            self.sk_bias = torch.empty(E, dtype=f32, device=dev)
            self.sk_ws = moe._bytes_tensor(moe._lib.moe_sinkhorn_workspace_size(T, E), dev)
            self.rl_ws = moe._bytes_tensor(moe._lib.moe_router_from_logits_workspace_size(T, E), dev)
        self.r_out = dict(logits=torch.empty((T, E), dtype=f32, device=dev),
                          topk_ids=torch.empty((T, k), dtype=i32, device=dev),
                          gates=torch.empty((T, k), dtype=f32, device=dev),
                          counts=torch.empty(E, dtype=i32, device=dev), f=torch.empty(E, dtype=f32, device=dev),
                          P=torch.empty(E, dtype=f32, device=dev), aux=torch.empty(1, dtype=f32, device=dev))
        self.r_ws = moe._bytes_tensor(moe.moe_router_workspace_size(T, h, E, k, code), dev)
        self.d_out = dict(buf=torch.empty((self.rows, h), dtype=dt, device=dev),
                          offsets=torch.empty(E + 1, dtype=i32, device=dev),
                          kept_counts=torch.empty(E, dtype=i32, device=dev),
                          dest_row=torch.empty((T, k), dtype=i32, device=dev),
                          drop_mask=torch.empty((T, k), dtype=torch.uint8, device=dev),
                          src_token=torch.empty(self.rows, dtype=i32, device=dev),
                          src_slot=torch.empty(self.rows, dtype=i32, device=dev),
                          rank_counts=torch.empty(R, dtype=i32, device=dev),
                          rank_offsets=torch.empty(R + 1, dtype=i32, device=dev),
                          tile_sched=torch.empty(moe.moe_tile_sched_bytes(T, E, k, self.C) // 4, dtype=i32,
                                                 device=dev))
        self.d_ws = moe._bytes_tensor(moe.moe_dispatch_workspace_size(T, E, k, self.C), dev)
        if payload == "fp8":                         # the FP8 send buffer replaces the bf16 one
            self.d_out.pop("buf")
            self.d_out["buf8"] = torch.empty((self.rows, h), dtype=torch.uint8, device=dev)
            self.d_out["scales"] = torch.empty((self.rows, h // 128), dtype=f32, device=dev)
            self.buf_deq = torch.empty((self.rows, h), dtype=dt, device=dev)   # the receive side, dequantised
        self.act = torch.empty((self.rows, F), dtype=dt, device=dev)
        self.eout = torch.empty((self.rows, h), dtype=dt, device=dev)
        if self.shared_packed is not None:
            self.sh_sched = moe.moe_dense_tile_sched(T, device=dev)
            self.sh_act = torch.empty((T, F), dtype=dt, device=dev)
            self.sh_out = torch.empty((T, h), dtype=dt, device=dev)
        self.y = torch.empty((T, h), dtype=dt, device=dev)
        # combine fused into the down GEMM's epilogue (bf16, token-choice or Sinkhorn routing): one launch fewer,
        # y bit-identical to the separate combine; its arrival counters start at zero and every call leaves them so
        if fuse_combine and (dt != torch.bfloat16 or routing == "expert_choice"
                             or (payload == "fp8" and shared is not None)):
            raise ValueError("fuse_combine: bf16 with token-choice or Sinkhorn routing (and no shared expert with the "
                             "FP8 payload)")
        self.fuse_combine = bool(fuse_combine)
        self.arrivals = moe.moe_combine_arrivals(T, h, dev) if self.fuse_combine else None
        self._saved = False
        if backward:                                 # pre-activations kept by forward(save=True)
            self.gu = torch.empty((self.rows, moe.gu_cols(F)), dtype=dt, device=dev)
            self.sh_gu = (torch.empty((T, moe.gu_cols(F)), dtype=dt, device=dev)
                          if self.shared_packed is not None else None)

    def forward(self, x, stream=None, events=None, y=None, save=False):
        if save and (self.packed_bwd is None or self.routing not in ("token", "sinkhorn")
                     or self.dtype != torch.bfloat16 or self.payload != "bf16"):
            raise NotImplementedError("MoELayer.forward(save=True): a layer built with backward=True, token-choice or "
                                      "Sinkhorn routing in bf16 with the bf16 send buffer")

        def mark(stage):
            if events is not None:
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(stream if stream is not None else torch.cuda.current_stream())
                events.setdefault(stage, []).append(ev)

        mark("start")
        r = self.r_out
        moe.moe_router(x, self.w_r, self.bias, self.k, "softmax" if self.routing == "sinkhorn" else self.gating,
                       self.alpha, logits=r["logits"],
                       topk_ids=r["topk_ids"], gates=r["gates"], counts=r["counts"], f=r["f"], P=r["P"], aux=r["aux"],
                       ws=self.r_ws, stream=stream, w_packed=self.w_r_packed)
        if self.routing == "expert_choice":
            moe.moe_expert_choice_route(r["logits"], self.C, tokens=self.ec["tokens"], gates=self.ec["gates"],
                                        slot=self.ec["slot"], ws=self.ec_ws, stream=stream)
        elif self.routing == "sinkhorn":
            # balanced selection: Sinkhorn column scalings as a selection-only bias, softmax gates
            moe.moe_sinkhorn_bias(r["logits"], sel_bias=self.sk_bias, ws=self.sk_ws, stream=stream)
            moe.moe_router_from_logits(r["logits"], self.sk_bias, self.k, "softmax_selbias", self.alpha,
                                       topk_ids=r["topk_ids"], gates=r["gates"], counts=r["counts"], f=r["f"],
                                       P=r["P"], aux=r["aux"], ws=self.rl_ws, stream=stream)
        mark("router")
        if self.routing == "expert_choice":
            moe.moe_expert_choice_dispatch(x, self.ec["tokens"], buf=self.d_out["buf"],
                                           tile_sched=self.d_out["tile_sched"], stream=stream)
        elif self.payload == "fp8":
            moe.moe_dispatch_fp8(x, r["topk_ids"], self.E, self.C, self.R, out=self.d_out, ws=self.d_ws, stream=stream)
        else:
            moe.moe_dispatch(x, r["topk_ids"], self.E, self.C, self.R, out=self.d_out, ws=self.d_ws, stream=stream)
        mark("dispatch")
        sched = self.d_out["tile_sched"]
        shared_out = None
        out = self.y if y is None else y
        if self.payload == "fp8":
            # dequantise the e4m3 send buffer in a pass of its own, then the bf16 GEMM (on GB300 faster than
            # moe_expert_up_gate_fp8's dequantisation inside the GEMM, with the same act)
            moe.moe_dequant_fp8(self.d_out["buf8"], self.d_out["scales"], out=self.buf_deq, stream=stream)
            moe.moe_expert_up_gate(self.buf_deq, sched, self.packed, self.E, self.F, act=self.act, stream=stream)
            mark("up_gate")
            self._down(sched, out, stream)
            mark("down")
        elif self.shared_packed is not None and self.dtype == torch.bfloat16:
            # the shared expert's tiles run inside the routed experts' launches
            if save:
                moe.moe_expert_up_gate_save(self.d_out["buf"], sched, self.packed, self.E, self.F, x=x,
                                            packed_shared=self.shared_packed, act=self.act, gu=self.gu,
                                            act_shared=self.sh_act, gu_shared=self.sh_gu, stream=stream)
            else:
                moe.moe_expert_up_gate_shared(self.d_out["buf"], sched, self.packed, self.E, self.F, x,
                                              self.shared_packed, act=self.act, act_shared=self.sh_act, stream=stream)
            mark("up_gate")
            self._down(sched, out, stream, shared=True)
            mark("down")
            shared_out = self.sh_out
        else:
            if save:
                moe.moe_expert_up_gate_save(self.d_out["buf"], sched, self.packed, self.E, self.F, act=self.act,
                                            gu=self.gu, stream=stream)
            else:
                moe.moe_expert_up_gate(self.d_out["buf"], sched, self.packed, self.E, self.F, act=self.act,
                                       stream=stream)
            mark("up_gate")
            self._down(sched, out, stream)
            mark("down")
        if self.shared_packed is not None and shared_out is None:
            moe.moe_expert_up_gate(x, self.sh_sched, self.shared_packed, 1, self.F, act=self.sh_act, stream=stream)
            mark("shared_up_gate")
            moe.moe_expert_down(self.sh_act, self.sh_sched, self.shared_packed, 1, self.h, eout=self.sh_out,
                                stream=stream)
            mark("shared_down")
            shared_out = self.sh_out
        if self.routing == "expert_choice":
            moe.moe_expert_choice_combine(self.eout, self.ec["slot"], self.ec["gates"], shared_out, y=out,
                                          stream=stream)
        elif not self.fuse_combine:
            moe.moe_combine(self.eout, self.d_out["dest_row"], r["gates"], shared_out, y=out, stream=stream)
        mark("combine")
        self._saved = bool(save)
        return out

    def _down(self, sched, y, stream, shared=False):
        """The down GEMM (with the shared expert's tiles in the same launch when `shared`), and with the combine
        in its epilogue when the layer fuses it (y is then written here)."""
        if self.fuse_combine:
            d = self.d_out
            moe.moe_expert_down_combine(self.act, sched, self.packed, self.E, self.h, d["src_token"], d["dest_row"],
                                        self.r_out["gates"], self.arrivals,
                                        act_shared=self.sh_act if shared else None,
                                        packed_shared=self.shared_packed if shared else None, eout=self.eout,
                                        out_shared=self.sh_out if shared else None, y=y, stream=stream)
        elif shared:
            moe.moe_expert_down_shared(self.act, sched, self.packed, self.E, self.h, self.sh_act, self.shared_packed,
                                       eout=self.eout, out_shared=self.sh_out, stream=stream)
        else:
            moe.moe_expert_down(self.act, sched, self.packed, self.E, self.h, eout=self.eout, stream=stream)

    def backward(self, x, dy, d_aux=1.0, stream=None, events=None):
        """Gradients of <dy, y> + d_aux * aux for the last forward(x): returns dict(dx, dW_r, d_bias, dW_gate,
        dW_up, dW_down[, shared_dW_gate, shared_dW_up, shared_dW_down]); weight gradients fp32, dx in the
        layer's dtype. Token-choice or Sinkhorn routing, bf16, and a layer built with backward=True. Order of the calls:
        combine, expert down / up-gate dgrad, expert weight gradients, [shared expert], router, router weight,
        dispatch (+ the router and shared terms of dx). `events` as in forward (stages "combine_bwd",
        "expert_dgrad", "expert_wgrad", ["shared_bwd"], "router_bwd", "dispatch_bwd")."""
        if self.packed_bwd is None:
            raise RuntimeError("MoELayer.backward: build the layer with backward=True")
        if self.routing not in ("token", "sinkhorn") or self.dtype != torch.bfloat16 or self.payload != "bf16":
            raise NotImplementedError("MoELayer.backward: token-choice or Sinkhorn routing in bf16 with the bf16 "
                                      "send buffer")

        def mark(stage):
            if events is not None:
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(stream if stream is not None else torch.cuda.current_stream())
                events.setdefault(stage, []).append(ev)

        dev, dt, f32 = self.device, self.dtype, torch.float32
        T, h, E, k, F, rows = self.T, self.h, self.E, self.k, self.F, self.rows
        if self._bwd is None:
            b = dict(d_eout=torch.empty((rows, h), dtype=dt, device=dev),
                     d_gates=torch.empty((T, k), dtype=f32, device=dev),
                     d_act=torch.empty((rows, F), dtype=dt, device=dev),
                     d_gu=torch.empty((rows, moe.gu_cols(F)), dtype=dt, device=dev),
                     d_buf=torch.empty((rows, h), dtype=dt, device=dev),
                     d_logits=torch.empty((T, E), dtype=f32, device=dev),
                     dx=torch.empty((T, h), dtype=dt, device=dev),
                     dW_r=torch.empty((h, E), dtype=f32, device=dev),
                     dW_gate=torch.empty((E, F, h), dtype=f32, device=dev),
                     dW_up=torch.empty((E, F, h), dtype=f32, device=dev),
                     dW_down=torch.empty((E, h, F), dtype=f32, device=dev),
                     ws_wg=moe._bytes_tensor(moe._lib.moe_expert_weight_grads_workspace_size(
                         E, h, F, rows, moe.dtype_code(dt)), dev),
                     ws_rb=moe._bytes_tensor(moe._lib.moe_router_backward_workspace_size(T, E), dev),
                     ws_rw=moe._bytes_tensor(moe._lib.moe_router_weight_grad_workspace_size(T, h, E), dev),
                     ws_db=moe._bytes_tensor(moe._lib.moe_dispatch_backward_workspace_size(T, h, E,
                                                                                           moe.dtype_code(dt)), dev))
            if self.shared_packed is not None:
                b.update(sh_d_act=torch.empty((T, F), dtype=dt, device=dev),
                         sh_d_gu=torch.empty((T, moe.gu_cols(F)), dtype=dt, device=dev),
                         sh_dx=torch.empty((T, h), dtype=dt, device=dev),
                         sh_dW_gate=torch.empty((1, F, h), dtype=f32, device=dev),
                         sh_dW_up=torch.empty((1, F, h), dtype=f32, device=dev),
                         sh_dW_down=torch.empty((1, h, F), dtype=f32, device=dev),
                         sh_off=torch.tensor([0, T], dtype=torch.int32, device=dev),
                         sh_kept=torch.tensor([T], dtype=torch.int32, device=dev),
                         ws_sh=moe._bytes_tensor(moe._lib.moe_expert_weight_grads_workspace_size(
                             1, h, F, T, moe.dtype_code(dt)), dev))
            self._bwd = b
        b = self._bwd
        r, d = self.r_out, self.d_out
        sched = d["tile_sched"]
        mark("start")
        moe.moe_combine_backward(dy, self.eout, d["src_token"], d["src_slot"], d["dest_row"], r["gates"],
                                 d_eout=b["d_eout"], d_gates=b["d_gates"], stream=stream)
        mark("combine_bwd")
        moe.moe_expert_down_backward(b["d_eout"], sched, self.packed_bwd, E, F, d_act=b["d_act"], stream=stream)
        if self._saved:                  # g and u kept by forward(save=True)
            moe.moe_expert_up_gate_backward_saved(self.gu, b["d_act"], sched, self.packed_bwd, E, h, d_gu=b["d_gu"],
                                                  d_buf=b["d_buf"], stream=stream)
        else:
            moe.moe_expert_up_gate_backward(d["buf"], b["d_act"], sched, self.packed, self.packed_bwd, E,
                                            d_gu=b["d_gu"], d_buf=b["d_buf"], stream=stream)
        mark("expert_dgrad")
        moe.moe_expert_weight_grads(d["buf"], self.act, b["d_gu"], b["d_eout"], d["offsets"], d["kept_counts"], E,
                                    dW_gate=b["dW_gate"], dW_up=b["dW_up"], dW_down=b["dW_down"], ws=b["ws_wg"],
                                    stream=stream)
        mark("expert_wgrad")
        sh_dx = None
        if self.shared_packed is not None:
            moe.moe_expert_down_backward(dy, self.sh_sched, self.shared_packed_bwd, 1, F, d_act=b["sh_d_act"],
                                         stream=stream)
            if self._saved:
                moe.moe_expert_up_gate_backward_saved(self.sh_gu, b["sh_d_act"], self.sh_sched, self.shared_packed_bwd,
                                                      1, h, d_gu=b["sh_d_gu"], d_buf=b["sh_dx"], stream=stream)
            else:
                moe.moe_expert_up_gate_backward(x, b["sh_d_act"], self.sh_sched, self.shared_packed,
                                                self.shared_packed_bwd, 1, d_gu=b["sh_d_gu"], d_buf=b["sh_dx"],
                                                stream=stream)
            moe.moe_expert_weight_grads(x, self.sh_act, b["sh_d_gu"], dy, b["sh_off"], b["sh_kept"], 1,
                                        dW_gate=b["sh_dW_gate"], dW_up=b["sh_dW_up"], dW_down=b["sh_dW_down"],
                                        ws=b["ws_sh"], stream=stream)
            sh_dx = b["sh_dx"]
            mark("shared_bwd")
        # the bias is part of the logits in the plain softmax modes and under Sinkhorn routing (whose router runs
        # in the plain softmax mode); the sigmoid mode's bias only selects
        want_bias = self.bias is not None and (self.gating in ("softmax", "softmax_renorm") or self.routing == "sinkhorn")
        d_logits, d_bias = moe.moe_router_backward(r["logits"], r["topk_ids"], r["gates"], b["d_gates"], r["f"],
                                                   self.gating, self.alpha, d_aux, d_logits=b["d_logits"],
                                                   want_bias_grad=want_bias, ws=b["ws_rb"], stream=stream)
        moe.moe_router_weight_grad(x, d_logits, dW_r=b["dW_r"], ws=b["ws_rw"], stream=stream)
        mark("router_bwd")
        moe.moe_dispatch_backward(b["d_buf"], d["dest_row"], d_logits, self.w_r, dx_extra=sh_dx,
                                  dx=b["dx"], ws=b["ws_db"], stream=stream)
        mark("dispatch_bwd")
        out = dict(dx=b["dx"], dW_r=b["dW_r"], d_bias=d_bias, dW_gate=b["dW_gate"], dW_up=b["dW_up"],
                   dW_down=b["dW_down"])
        if self.shared_packed is not None:
            out.update(shared_dW_gate=b["sh_dW_gate"][0], shared_dW_up=b["sh_dW_up"][0],
                       shared_dW_down=b["sh_dW_down"][0])
        return out

    def capture_forward(self, x, stream=None):
        """The forward of x (device-resident, kept at this address) captured once into a CUDA graph; each
        `replay()` then runs the layer's launches from the graph instead of from the host, into the same output
        buffers (`self.y`, `self.r_out`, `self.d_out`, ...). Call `forward` once before (it sets up the kernels'
        attributes); the graph holds the layer's buffers and x by address, so neither may be freed or moved while
        it is in use."""
        import torch
        s = stream if stream is not None else torch.cuda.Stream(device=self.device)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(self.device)
        with torch.cuda.graph(g, stream=s):
            self.forward(x, stream=s)
        return g

    def native_desc(self):
        """The moe_layer_desc of this layer for the one-call C entry points moe_layer_forward and
        moe_layer_forward_host (every routing mode and send buffer of `forward`, with the separate combine: the
        same launches): it points at this layer's packed parameters, which must outlive its use."""
        if self.fuse_combine:
            raise NotImplementedError("moe_layer_forward runs the separate combine (MoELayer(fuse_combine=False))")
        return moe.moe_layer_desc(T=self.T, h=self.h, E=self.E, k=self.k, F=self.F, dtype=self.dtype,
                                  gating="softmax" if self.routing == "sinkhorn" else self.gating, alpha=self.alpha,
                                  capacity=self.C, num_ranks=self.R, w_r_packed=self.w_r_packed, bias=self.bias,
                                  packed_w=self.packed, packed_shared=self.shared_packed, routing=self.routing,
                                  payload="fp8" if self.payload == "fp8" else "dtype")

    def forward_host_native(self, x_hosts, y_hosts, ws=None):
        """forward_host_batches through the C ABI: one moe_layer_forward_host call (the copies and the overlap are
        the library's). ws: a device byte tensor of moe_layer_host_workspace_size bytes, kept across calls (one is
        made when None). Returns after the last output has reached host memory."""
        desc = self.native_desc()
        if ws is None:
            ws = moe._bytes_tensor(moe.moe_layer_host_workspace_size(desc), self.device)
        moe.moe_layer_forward_host(desc, x_hosts, y_hosts, ws)
        torch.cuda.synchronize(self.device)
        return y_hosts

    def forward_host_batches(self, x_hosts, y_hosts):
        """Runs the layer over a sequence of batches that live in pinned host memory: x_hosts[i] -> y_hosts[i].

        Every batch's tokens are copied host -> device and its output device -> host, on two copy streams,
        while the layer works on another batch on the current stream (two device buffers for x and for y,
        each reused only after the copy or the layer that last used it has finished). Returns after the last
        output has reached host memory. The host tensors must be pinned and have the layer's dtype and
        shape (bf16 may be given as int16 bit patterns)."""
        dev = self.device
        compute = torch.cuda.current_stream(dev)
        h2d = torch.cuda.Stream(dev)
        d2h = torch.cuda.Stream(dev)
        dt = self.dtype
        xd = [torch.empty((self.T, self.h), dtype=dt, device=dev) for _ in range(2)]
        yd = [torch.empty((self.T, self.h), dtype=dt, device=dev) for _ in range(2)]
        x_free = [None, None]          # layer done reading xd[b]
        y_free = [None, None]          # d2h done reading yd[b]

        def as_dt(t):
            return t.view(dt) if t.dtype != dt else t

        for i, (xh, yh) in enumerate(zip(x_hosts, y_hosts)):
            b = i & 1
            with torch.cuda.stream(h2d):
                if x_free[b] is not None:
                    h2d.wait_event(x_free[b])
                xd[b].copy_(as_dt(xh), non_blocking=True)
                x_in = torch.cuda.Event()
                x_in.record(h2d)
            compute.wait_event(x_in)
            if y_free[b] is not None:
                compute.wait_event(y_free[b])
            self.forward(xd[b], y=yd[b])
            done = torch.cuda.Event()
            done.record(compute)
            x_free[b] = done
            with torch.cuda.stream(d2h):
                d2h.wait_event(done)
                as_dt(yh).copy_(yd[b], non_blocking=True)
                out = torch.cuda.Event()
                out.record(d2h)
            y_free[b] = out
        torch.cuda.synchronize(dev)
        return y_hosts
