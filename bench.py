"""MoE layer forward benchmark on GB300: tokens/s of router -> dispatch -> grouped SwiGLU FFN -> combine.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--workload NAME]

One step = one full forward of the layer over one batch of synthetic tokens (all four stages, plus the
shared expert where the workload has one). Default workload: the page-3 worked shape (T=4096, h=4096,
E=8, k=2, cf=1.25 -> C=1280, SwiGLU 4096->12288->4096, bf16 with fp32 accumulation). Weights and x are
resident in HBM before the timed region; L2 (129 MB) is flushed by a 512 MiB write between steps, outside
the per-step CUDA events. Under torchrun each rank runs its own replica on its own GPU (weak scaling, no
data-path collective); rank 0 prints one JSON line.

--impl reference times the CPU oracle (float64, numpy) on the host cores instead: each step runs the
oracle's router and dispatch over the whole batch and its FFN + combine on a bounded sample of tokens,
and the per-token FFN cost is extrapolated to the batch.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs  # noqa: E402

METRIC = "MoE-layer fwd tokens/s at 1 GB300; grouped-GEMM % bf16 peak; dispatch GB/s"

TIMING_NOTE = ("ms_per_step: K forwards, each after an L2 flush, with CUDA events at each step's start and end; "
               "stages_ms, roofline and the stage bandwidths: a second pass of K forwards with an event at every "
               "stage boundary (those events serialise the stages' launches: ms_per_step_instrumented)")

def _workload_desc(cfg, C):
    return (f"{cfg.name}: T={cfg.T} h={cfg.h} E={cfg.E} k={cfg.k} F={cfg.F} gating={cfg.gating} "
            + (f"cf={cfg.cf} (C={C})" if cfg.cf else "dropless") + f" R={cfg.R} shared={cfg.n_shared} {cfg.dtype}"
            + (" payload=fp8 (e4m3, per-128 scales)" if cfg.payload == "fp8" else ""))


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _smi_id(local):
    """nvidia-smi -i argument of this process's GPU (its UUID; nvidia-smi ignores CUDA_VISIBLE_DEVICES)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.window = (0.0, float("inf"))

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        """Keep only the samples that arrived inside the timed region [t0, t1]."""
        self.window = (t0, t1)

    def stop(self):
        self.__exit__()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, window=None):
        """Median SM clock, the maximum and the throttle reasons seen in `window` (default: the marked one)."""
        w0, w1 = window if window is not None else self.window
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in list(self.lines):
            if not (w0 <= ts <= w1 + 0.03):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------------------
# host inputs
# ---------------------------------------------------------------------------------------------------------

def host_inputs(cfg, seed=0):
    x = moe_inputs.make_x(cfg, seed)
    w_r, bias = moe_inputs.make_router(cfg, seed)
    wg, wu, wd = moe_inputs.all_expert_weights(cfg, seed)
    shared = None
    if cfg.n_shared:
        shared = tuple(a[0] for a in moe_inputs.all_expert_weights(cfg, seed, shared=True))
    return dict(x=x, w_r=w_r, bias=bias, wg=wg, wu=wu, wd=wd, shared=shared)


# ---------------------------------------------------------------------------------------------------------
# CPU oracle arm (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------------------------------------

def oracle_step(cfg, inp, w64, sample_tokens, keep=None):
    """One bounded oracle step: router + dispatch over all T tokens, FFN + combine for `sample_tokens`.
    Returns (seconds for router+dispatch, seconds for the sampled FFN); `keep` (a dict) receives the routing,
    the dispatch and the sampled tokens' y."""
    from oracle import moe_oracle as O
    t0 = time.perf_counter()
    x64 = moe_inputs.to_f64(inp["x"], cfg.dtype)
    L = O.router_logits(x64, moe_inputs.to_f64(inp["w_r"], cfg.dtype), inp["bias"], cfg.gating)
    r = O.route(L, cfg.k, cfg.gating, inp["bias"], cfg.alpha)
    d = O.dispatch(r["ids"], cfg.E, O.capacity(cfg.cf, cfg.k, cfg.T, cfg.E), cfg.R)
    t1 = time.perf_counter()
    y = O.moe_layer_tokens(sample_tokens, x64, r, d, lambda e: w64[e], shared=w64.get("shared"))
    t2 = time.perf_counter()
    if keep is not None:
        keep.update(route=r, dispatch=d, y=y, tokens=sample_tokens)
    return t1 - t0, t2 - t1


class _LazyWeights(dict):
    """Expert weights decoded to float64 on first use, one expert kept at a time (the DeepSeek-V3-shaped
    workload's 22.6 GB of bf16 weights would take 90 GB as float64)."""

    def __init__(self, cfg, inp):
        super().__init__()
        self.cfg, self.inp = cfg, inp
        if inp["shared"] is not None:
            sh = tuple(moe_inputs.to_f64(w, cfg.dtype) for w in inp["shared"])
            self["shared"] = lambda: sh

    def __missing__(self, e):
        for key in [k for k in self if k != "shared"]:
            del self[key]
        c, i = self.cfg, self.inp
        w = (moe_inputs.to_f64(i["wg"][e], c.dtype), moe_inputs.to_f64(i["wu"][e], c.dtype),
             moe_inputs.to_f64(i["wd"][e], c.dtype))
        self[e] = w
        return w


def decode_weights(cfg, inp, lazy=False):
    if lazy:
        return _LazyWeights(cfg, inp)
    w64 = {e: (moe_inputs.to_f64(inp["wg"][e], cfg.dtype), moe_inputs.to_f64(inp["wu"][e], cfg.dtype),
               moe_inputs.to_f64(inp["wd"][e], cfg.dtype)) for e in range(cfg.E)}
    if inp["shared"] is not None:
        sh = tuple(moe_inputs.to_f64(w, cfg.dtype) for w in inp["shared"])
        w64["shared"] = lambda: sh
    return w64


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_throughput(cfg, inp, w64, steps, n_sample, seed=1, keep=None):
    """Tokens/s of the oracle: T / (router+dispatch time + sampled FFN time scaled to T tokens)."""
    rng = np.random.default_rng(seed)
    vals = []
    for _ in range(steps):
        toks = np.sort(rng.choice(cfg.T, size=n_sample, replace=False))
        t_rd, t_ffn = oracle_step(cfg, inp, w64, toks, keep)
        vals.append(cfg.T / (t_rd + t_ffn * cfg.T / n_sample))
    return vals


def parity_report(cfg, layer, keep):
    """The GPU layer's output for the bench input against the oracle run of the cpu_baseline leg: router ids over
    all T tokens (tokens whose top-(k+1) selection scores lie within 1e-6 of each other are near ties, where
    the fp32 GPU and the float64 oracle may order experts differently), y on the sampled tokens."""
    from oracle import moe_oracle as O
    if cfg.routing != "token" or cfg.payload != "bf16":
        return {"skipped": f"{cfg.routing} routing / {cfg.payload} payload: see the parity tests"}
    r = keep["route"]
    ids = layer.r_out["topk_ids"].cpu().numpy()
    bad = np.nonzero((ids != r["ids"]).any(axis=1))[0]
    near = O.near_tie_rows(r["gaps"], 1e-6)
    toks = keep["tokens"]
    import torch
    y = layer.y[torch.as_tensor(np.asarray(toks), device=layer.y.device)].float().cpu().numpy().astype(np.float64)
    y_ref = keep["y"]
    ok = ~np.isin(toks, bad)
    d = y[ok] - y_ref[ok]
    if cfg.dtype == "bf16":
        kind, tol = "normwise rel l2", 2e-2
        err = float(np.linalg.norm(d) / max(np.linalg.norm(y_ref[ok]), 1e-300))
    else:
        kind, tol = "max abs / max |ref|", 1e-5
        err = float(np.max(np.abs(d)) / max(np.max(np.abs(y_ref[ok])), 1e-300))
    return {"tokens_checked": int(len(toks)), "ids_mismatched_tokens": int(bad.size),
            "near_tie_tokens": int(near.size), "y_err": err, "y_err_kind": kind, "tolerance": tol,
            "pass": bool(err <= tol and np.isin(bad, near).all())}


def run_reference(args, cfg, C):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = host_inputs(cfg)
    w64 = decode_weights(cfg, inp)
    n_sample = args.sample_tokens
    oracle_throughput(cfg, inp, w64, args.warmup, n_sample)
    t0 = time.perf_counter()
    vals = oracle_throughput(cfg, inp, w64, args.steps, n_sample)
    wall = time.perf_counter() - t0
    v = statistics.median(vals)
    cores = blas_threads()
    sample = (f"per step: oracle router+dispatch over all {cfg.T} tokens, FFN+combine on {n_sample} random tokens "
              f"(float64 numpy), FFN cost scaled to {cfg.T} tokens; median of {args.steps} steps")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _workload_desc(cfg, C), "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------------------

def max_over_ranks(v: float, world: int, device) -> float:
    """The slowest rank's value (the whole job ends when its slowest replica does)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


EXTRA_WORKLOADS = ["tiny_fp32", "mixtral_zipf", "deepseek_v3", "qwen3_moe"]


def fuses_combine(args, cfg) -> bool:
    """Whether the layer runs the combine inside the down GEMM's epilogue (bf16, token-choice or Sinkhorn
    routing, and no shared expert with the FP8 payload), unless --no-fuse-combine."""
    return (args.fuse_combine and cfg.dtype == "bf16" and cfg.routing != "expert_choice"
            and not (cfg.payload == "fp8" and cfg.n_shared))


def build_layer(cfg, inp, dev, backward, fuse_combine=False):
    import torch
    from top_routing_dispatch_moe_gb300.layer import MoELayer

    def up(a):
        if cfg.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    layer = MoELayer(T=cfg.T, h=cfg.h, E=cfg.E, k=cfg.k, F=cfg.F, gating=cfg.gating, cf=cfg.cf, R=cfg.R,
                     alpha=cfg.alpha, w_r=up(inp["w_r"]),
                     bias=torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None,
                     w_gate=up(inp["wg"]), w_up=up(inp["wu"]), w_down=up(inp["wd"]),
                     shared=tuple(up(np.ascontiguousarray(w)[None]) for w in inp["shared"])
                     if inp["shared"] is not None else None, device=dev, routing=cfg.routing,
                     backward=backward, payload=cfg.payload, fuse_combine=fuse_combine)
    return layer, up(inp["x"])


def time_forward(args, layer, x, flush, world, dev):
    """K device-resident layer forwards, each after an L2 flush, with CUDA events at each step's start and end on
    the launching stream (the step time); then K more with an event at every stage boundary (the stage times, and
    from them the up/gate roofline: an event between two launches serialises them, so those steps are longer).
    Returns both, the library's launch count over the first pass and the clocks of both."""
    import torch
    import torch.distributed as dist
    from top_routing_dispatch_moe_gb300 import moe
    for _ in range(args.warmup):
        layer.forward(x)
        flush.zero_()
    torch.cuda.synchronize()
    t_start = time.time()
    while time.time() - t_start < 0.3:                  # let the sampler start; keep the GPU busy meanwhile
        layer.forward(x)
        flush.zero_()
        torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = moe.moe_launch_count()
    t_clk0 = time.time()
    t_wall0 = time.perf_counter()
    # every step follows an L2 flush, the first one too (its launches then queue behind the flush instead of
    # reaching an idle GPU one by one from the host)
    flush.zero_()
    step_ev = []
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        layer.forward(x)
        e1.record()
        step_ev.append((e0, e1))
        flush.zero_()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    launches = moe.moe_launch_count() - launches0
    if world > 1:
        dist.barrier()
    # the instrumented pass: the same steps with an event at every stage boundary
    events: dict = {}
    flush.zero_()
    for _ in range(args.steps):
        layer.forward(x, events=events)
        flush.zero_()
    torch.cuda.synchronize()
    window = (t_clk0, time.time())
    if world > 1:
        dist.barrier()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    from top_routing_dispatch_moe_gb300.layer import MoELayer
    stage_names = [s for s in MoELayer.STAGES if s in events]
    order = ["start"] + stage_names
    stage_ms = {s: [] for s in stage_names}
    inst_ms = []
    for i in range(args.steps):
        for a, b in zip(order[:-1], order[1:]):
            stage_ms[b].append(events[a][i].elapsed_time(events[b][i]))
        inst_ms.append(events["start"][i].elapsed_time(events[order[-1]][i]))
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms = max_over_ranks(float(np.mean(step_ms)), world, dev)
    stats = {"median": float(np.median(step_ms)), "p10": float(np.percentile(step_ms, 10)),
             "p90": float(np.percentile(step_ms, 90))}
    return dict(stage_ms=stage_ms, ms=ms, stats=stats, launches=int(launches), wall=t_wall, window=window,
                ms_instrumented=max_over_ranks(float(np.mean(inst_ms)), world, dev))


def kept_and_active(cfg, layer):
    if cfg.routing == "expert_choice":
        return cfg.E * layer.C, cfg.E                 # every expert takes exactly C tokens
    kc = layer.d_out["kept_counts"]
    return int(kc.sum().item()), int((kc > 0).sum().item())   # active: experts whose weights the GEMMs read


def stage_metrics(cfg, stage_ms, kept, active, fused_combine=False):
    """Roofline of the dominant kernel (the up/gate grouped GEMM) and the bandwidth of the other stages, from the
    algorithmic work per unit: router T h el + h E el bytes, dispatch (T + kept) h el, combine (kept + T [+ T
    shared]) h el, FFN 6 h F flop per kept row (plus the shared expert's T rows). With the combine fused into the
    down GEMM the "down" stage holds both, and the combine has no bandwidth of its own (null)."""
    hbm, bf16_burst, bf16_sus, peak_src = _peaks()
    mean = {s: float(np.mean(v)) for s, v in stage_ms.items()}
    ug_ms, dn_ms = mean["up_gate"], mean["down"]
    # with bf16 the shared expert's tiles run inside the up/gate and down launches
    fused_shared = bool(cfg.n_shared) and "shared_up_gate" not in stage_ms
    ug_flops = 4.0 * (kept + (cfg.T if fused_shared else 0)) * cfg.h * cfg.F
    ffn_flops = 6.0 * kept * cfg.h * cfg.F + (6.0 * cfg.T * cfg.h * cfg.F if cfg.n_shared else 0.0)
    ffn_ms = ug_ms + dn_ms + sum(mean[s] for s in ("shared_up_gate", "shared_down") if s in mean)
    ug_tflops = ug_flops / (ug_ms * 1e-3) / 1e12
    if cfg.payload == "fp8":                         # read x once, write one byte per element + a scale per 128
        disp_bytes = cfg.T * cfg.h * cfg.el + kept * (cfg.h + cfg.h // 128 * 4)
    else:
        disp_bytes = (cfg.T + kept) * cfg.h * cfg.el
    comb_bytes = (kept + cfg.T + (cfg.T if cfg.n_shared else 0)) * cfg.h * cfg.el
    router_bytes = (cfg.T * cfg.h + cfg.h * cfg.E) * cfg.el
    gbs = lambda nbytes, stage: nbytes / (mean[stage] * 1e-3) / 1e9   # noqa: E731
    # The up/gate GEMM's algorithmic bytes: the gate and up weights of every expert that received rows (and the
    # shared expert's), its input rows read once, the activation written once. Below the ridge point (few rows
    # per expert) the weight stream, not the tensor cores, bounds it; the roofline takes whichever bound is
    # reached later at the measured peaks.
    ug_rows = kept + (cfg.T if fused_shared else 0)
    ug_bytes = ((active + (1 if fused_shared else 0)) * 2.0 * cfg.F * cfg.h + ug_rows * (cfg.h + cfg.F)) * cfg.el
    ug_gbs = ug_bytes / (ug_ms * 1e-3) / 1e9
    if ug_bytes / (hbm * 1e9) > ug_flops / (bf16_burst * 1e12):
        roofline = {"bound": "hbm", "kernel": "up/gate grouped GEMM (SwiGLU epilogue)", "achieved": ug_gbs,
                    "peak": hbm, "unit": "GB/s", "frac": ug_gbs / hbm, "traffic": None,
                    "peak_source": f"{peak_src} HBM copy", "tensor_tflops": ug_tflops}
    else:
        roofline = {"bound": "tensor", "kernel": "up/gate grouped GEMM (SwiGLU epilogue)", "achieved": ug_tflops,
                    "peak": bf16_burst, "unit": "TFLOP/s", "frac": ug_tflops / bf16_burst, "traffic": None,
                    "peak_source": f"{peak_src} bf16 burst"}
    if roofline["bound"] == "tensor" and bf16_sus:
        # the same kernel against the sustained (power-capped, seconds-long loop) bf16 peak: the timed region runs
        # the GEMMs back to back for the whole run, under the same cap
        roofline["frac_of_sustained_peak"] = ug_tflops / bf16_sus
    roofline["algorithmic_bytes"] = ug_bytes
    roofline["intensity_flop_per_byte"] = ug_flops / ug_bytes
    roofline["ridge_flop_per_byte"] = bf16_burst * 1e12 / (hbm * 1e9)
    out = {"stages_ms": mean, "roofline": roofline,
           "expert_tflops": ffn_flops / (ffn_ms * 1e-3) / 1e12,
           "grouped_gemm_pct_bf16_peak": 100.0 * ffn_flops / (ffn_ms * 1e-3) / 1e12 / bf16_burst,
           "router_gbs": gbs(router_bytes, "router"), "router_pct_hbm": 100.0 * gbs(router_bytes, "router") / hbm,
           "dispatch_gbs": gbs(disp_bytes, "dispatch"), "dispatch_pct_hbm": 100.0 * gbs(disp_bytes, "dispatch") / hbm,
           "combine_fused_into_down_gemm": bool(fused_combine)}
    if fused_combine:
        out.update(combine_gbs=None, combine_pct_hbm=None)
    else:
        out.update(combine_gbs=gbs(comb_bytes, "combine"), combine_pct_hbm=100.0 * gbs(comb_bytes, "combine") / hbm)
    return out


def measure_extra_workload(args, name, world, dev, flush, clk, rank):
    """One more workload of the default run: the forward timed as the headline's is (no backward, no e2e leg),
    with its stage bandwidths, its roofline and (rank 0, one GPU) its parity against the oracle on a sample."""
    import torch
    cfg = moe_inputs.get_config(name)
    C = 0
    if cfg.cf:
        import math
        C = int(math.ceil(cfg.cf * cfg.k * cfg.T / cfg.E - 1e-9))
    inp = host_inputs(cfg)
    layer, x = build_layer(cfg, inp, dev, backward=False, fuse_combine=fuses_combine(args, cfg))
    t = time_forward(args, layer, x, flush, world, dev)
    kept, active = kept_and_active(cfg, layer)
    out = {"workload": _workload_desc(cfg, C), "value": world * cfg.T / (t["ms"] * 1e-3), "unit": "tokens/s",
           "ms_per_step": t["ms"], "ms_per_step_stats": t["stats"], "ms_per_step_instrumented": t["ms_instrumented"],
           "kept_assignments": kept, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "gpu_launches": t["launches"]}
    out.update(stage_metrics(cfg, t["stage_ms"], kept, active, layer.fuse_combine))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        keep: dict = {}
        rng = np.random.default_rng(2)
        toks = np.sort(rng.choice(cfg.T, size=min(cfg.T, args.parity_tokens), replace=False))
        oracle_step(cfg, inp, decode_weights(cfg, inp, lazy=True), toks, keep)
        out["parity"] = parity_report(cfg, layer, keep)
    time.sleep(0.05)                                  # the sampler's last lines of the timed region
    out["clocks"] = clk.summary(t["window"])
    del layer, x
    torch.cuda.empty_cache()
    return out


def run_gpu(args, cfg, C):
    import torch
    import torch.distributed as dist
    from top_routing_dispatch_moe_gb300 import moe
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    inp = host_inputs(cfg)
    layer, x = build_layer(cfg, inp, dev, want_backward(args, cfg), fuse_combine=fuses_combine(args, cfg))
    flush = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    clk = ClockSampler(_smi_id(local)).start()
    # ---- device-resident timed region
    t = time_forward(args, layer, x, flush, world, dev)
    stage_ms, ms = t["stage_ms"], t["ms"]
    kept, active = kept_and_active(cfg, layer)
    value = world * cfg.T / (ms * 1e-3)

    # ---- end-to-end through the public API: every step copies its batch of tokens in from pinned host
    # memory and its output back to pinned host memory, overlapped with the neighbouring steps' layer work on
    # separate streams: one C-ABI call for all K steps (moe_layer_forward_host: the copies, the chain and the
    # overlap in the library); a layer with the combine fused into the down GEMM goes through the Python layer's
    # forward_host_batches instead. No L2 flush here (the weights already exceed L2), so the time of the whole K-step run
    # divided by K is the per-step time
    x_np = np.ascontiguousarray(inp["x"]).view(np.int16) if cfg.dtype == "bf16" else np.ascontiguousarray(inp["x"])
    x_hosts = [torch.from_numpy(x_np).pin_memory() for _ in range(2)]
    y_hosts = [torch.empty(x_np.shape, dtype=x_hosts[0].dtype).pin_memory() for _ in range(2)]
    try:
        desc = layer.native_desc()
        e2e_ws = moe._bytes_tensor(moe.moe_layer_host_workspace_size(desc), dev)
        e2e_path = "C ABI: moe_layer_forward_host (pinned host x in, y out)"

        def host_run(n):
            moe.moe_layer_forward_host(desc, [x_hosts[i % 2] for i in range(n)], [y_hosts[i % 2] for i in range(n)],
                                       e2e_ws, stream)
    except NotImplementedError:
        e2e_path = "Python: MoELayer.forward_host_batches over the C ABI (pinned host x in, y out)"

        def host_run(n):
            layer.forward_host_batches([x_hosts[i % 2] for i in range(n)], [y_hosts[i % 2] for i in range(n)])
    host_run(args.warmup)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    host_run(args.steps)
    e1.record(stream)
    e1.synchronize()
    e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    io_bytes = cfg.T * cfg.h * cfg.el

    # ---- backward of the layer (a separate timed loop; the headline value above is the forward): K backward
    # passes over the saved state of one forward of x, L2 flushed between them
    backward = None
    if want_backward(args, cfg):
        try:
            backward = time_backward(args, cfg, layer, x, flush, stream, kept)
        except Exception as exc:                      # reported in the line; the forward figures stand
            backward = {"error": f"{type(exc).__name__}: {exc}"}

    m = stage_metrics(cfg, stage_ms, kept, active, layer.fuse_combine)
    roofline = m.pop("roofline")
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            tr = json.load(fh).get(cfg.name, {})
        if tr.get("kernel_source_hash") == kernel_hash():
            roofline["traffic"] = tr.get("up_gate_dram_bytes")
    except Exception:
        pass

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_stats": t["stats"], "higher_is_better": True,
            "scaling": "weak", "timing": TIMING_NOTE, "ms_per_step_instrumented": t["ms_instrumented"],
            "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": _workload_desc(cfg, C), "global_batch": cfg.T * world, "tokens_per_gpu": cfg.T,
                       "parallelism": f"replicas x{world}", "l2": "flushed before every step (512 MiB write)",
                       "kept_assignments": kept},
            "roofline": roofline,
            **({"backward": backward} if backward is not None else {}),
            "e2e": {"value": world * cfg.T / (e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": io_bytes,
                    "d2h_bytes_per_step": io_bytes, "ms_per_step": e2e, "path": e2e_path},
            "gpu_launches": t["launches"],
            **m,
            "wall_s_timed_region": t["wall"]}
    line["clocks"] = clk.summary(t["window"])

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w64 = decode_weights(cfg, inp)
        keep: dict = {}
        vals = oracle_throughput(cfg, inp, w64, 1, args.baseline_tokens, keep=keep)
        line["cpu_baseline"] = {"value": vals[0], "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": f"oracle router+dispatch over all {cfg.T} tokens, FFN+combine on "
                                          f"{args.baseline_tokens} random tokens (float64 numpy), FFN cost scaled "
                                          f"to {cfg.T} tokens"}
        line["parity"] = parity_report(cfg, layer, keep)
        del w64

    # ---- the other workloads (forward only), measured the same way after the headline's memory is released
    extras = [w for w in args.workloads.split(",") if w and w != "none" and w != cfg.name]
    if extras:
        del layer, x, x_hosts, y_hosts
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name in extras:
            try:
                line["workloads"][name] = measure_extra_workload(args, name, world, dev, flush, clk, rank)
            except Exception as exc:                  # reported in the line; the headline figures stand
                line["workloads"][name] = {"error": f"{type(exc).__name__}: {exc}"}
                torch.cuda.empty_cache()
    clk.stop()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def want_backward(args, cfg) -> bool:
    return args.backward and cfg.dtype == "bf16" and cfg.routing in ("token", "sinkhorn") and cfg.payload == "bf16"


def time_backward(args, cfg, layer, x, flush, stream, kept):
    """Gradients of <dy, y> + aux, timed over K passes with CUDA events per stage, each from the state of a
    forward(x, save=True) (the forward keeps the experts' pre-activations g and u, so the backward does not
    recompute the up/gate GEMM); the K saving forwards are timed as well."""
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    dy = torch.randn(x.shape, generator=torch.Generator(device=x.device).manual_seed(5), device=x.device,
                     dtype=torch.float32).to(x.dtype)
    for _ in range(max(1, args.warmup)):
        layer.forward(x, save=True)
        layer.backward(x, dy)
        flush.zero_()
    torch.cuda.synchronize()
    events: dict = {}
    fwd = []
    flush.zero_()                                     # as in the forward timing: a flush before every pass
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        layer.forward(x, save=True)
        e1.record(stream)
        fwd.append((e0, e1))
        flush.zero_()
        layer.backward(x, dy, events=events)
        flush.zero_()
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    names = [s for s in ("combine_bwd", "expert_dgrad", "expert_wgrad", "shared_bwd", "router_bwd", "dispatch_bwd")
             if s in events]
    order = ["start"] + names
    st = {b: float(np.mean([events[a][i].elapsed_time(events[b][i]) for i in range(args.steps)]))
          for a, b in zip(order[:-1], order[1:])}
    ms = float(np.mean([events["start"][i].elapsed_time(events[order[-1]][i]) for i in range(args.steps)]))
    fwd_ms = float(np.mean([a.elapsed_time(b) for a, b in fwd]))
    # expert GEMM work per row: dgrad 6 h F (down 2, up/gate dgrad 4; g and u were saved) + wgrad 6 h F
    rows = kept + (cfg.T if cfg.n_shared else 0)
    gemm_flops = 12.0 * rows * cfg.h * cfg.F
    gemm_ms = st["expert_dgrad"] + st["expert_wgrad"] + st.get("shared_bwd", 0.0)
    return {"ms_per_step": ms, "tokens_per_s": cfg.T / (ms * 1e-3), "unit": "tokens/s", "stages_ms": st,
            "forward_save_ms": fwd_ms, "train_step_ms": fwd_ms + ms,
            "expert_gemm_tflops": gemm_flops / (gemm_ms * 1e-3) / 1e12,
            "what": "dx, dW_r, d_bias, every expert's and the shared expert's fp32 weight gradients for "
                    "<dy, y> + aux from a forward that kept the experts' pre-activations (forward_save_ms: that "
                    "forward); L2 flushed between passes"}


def kernel_hash():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "top_routing_dispatch_moe_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.startswith("ffn"):
            h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="page3_cf1.25", choices=list(moe_inputs.CONFIGS))
    ap.add_argument("--config", type=int, choices=range(1, len(moe_inputs.CONFIG_ORDER) + 1), default=None,
                    help="the workload by number, 1.." + str(len(moe_inputs.CONFIG_ORDER)) + " = "
                         + ", ".join(moe_inputs.CONFIG_ORDER) + " (overrides --workload)")
    ap.add_argument("--backward", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the layer's backward (bf16 token-choice workloads), reported under 'backward'")
    ap.add_argument("--sample-tokens", type=int, default=32, help="oracle tokens per reference-arm step")
    ap.add_argument("--baseline-tokens", type=int, default=128, help="oracle tokens of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default=None,
                    help="comma-separated further workloads timed after the headline one (forward only), reported "
                         "under 'workloads'; default: the other four named configurations when the headline is "
                         "the page-3 workload, none otherwise; 'none' for none")
    ap.add_argument("--parity-tokens", type=int, default=32, help="oracle tokens of each further workload's parity")
    ap.add_argument("--fuse-combine", action=argparse.BooleanOptionalAction, default=False,
                    help="run the combine in the down GEMM's epilogue (bf16 token-choice / Sinkhorn layers); off by "
                         "default: on GB300 the separate combine measured faster")
    args = ap.parse_args()
    if args.config is not None:
        args.workload = moe_inputs.CONFIG_ORDER[args.config - 1]
    assert args.warmup >= 3, "at least 3 warm-up steps"
    cfg = moe_inputs.get_config(args.workload)
    if args.workloads is None:
        args.workloads = ",".join(EXTRA_WORKLOADS) if args.workload == "page3_cf1.25" else "none"
    C = 0
    if cfg.cf:
        import math
        C = int(math.ceil(cfg.cf * cfg.k * cfg.T / cfg.E - 1e-9))
    if args.impl == "reference":
        run_reference(args, cfg, C)
    else:
        from top_routing_dispatch_moe_gb300 import build
        build.build()
        run_gpu(args, cfg, C)


if __name__ == "__main__":
    main()
