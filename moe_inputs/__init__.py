"""Seeded synthetic inputs for the MoE layer (shared by the oracle tests, the GPU tests and the bench).

This module only draws random numbers and stores them in the working dtype. It holds none of the
layer's arithmetic: no router, no top-k, no capacity formula, no FFN. Both sides of every parity test
(the plain CPU oracle and the CUDA path) receive the very same bits from here.

Random numbers come from numpy's Philox4x32-10 bit generator (Salmon et al., "Parallel random numbers:
as easy as 1, 2, 3", SC'11), one substream per tensor (and per expert / per redrawn row), keyed by
(seed, stream, sub). bf16 values are float32 draws rounded to nearest-even.

The five workloads follow the shapes the pages use: the page-3 worked example of "v6 长序列和 MoE: Context
Parallel 与 Expert Parallel" (section "NVIDIA 原题: Implement MoE and show the dimensions": T=4096, h=4096,
E=8, k=2, cf=1.25, FFN 4096->12288->4096), and Mixtral-, DeepSeek-V3- and Qwen3-MoE-shaped layers named in
"10.5 序列并行与专家并行" (section 10.5.4) and in "Megatron-LM 分布式训练（六）" (background list).
"""
from __future__ import annotations

import dataclasses
import json
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# ---------------------------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------------------------

GATING_SOFTMAX = "softmax"                      # gate = full-softmax probability of the chosen expert
GATING_SOFTMAX_RENORM = "softmax_renorm"        # gate = softmax prob renormalised over the k chosen
GATING_SIGMOID_BIAS_RENORM = "sigmoid_bias_renorm"  # select on sigmoid(L)+b, gate = s / sum_chosen s


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens (batch x sequence flattened)
    h: int            # hidden size
    E: int            # routed experts
    k: int            # experts per token
    F: int            # expert FFN inner size (SwiGLU)
    gating: str
    cf: float         # capacity factor; 0 = dropless
    R: int            # virtual expert-parallel ranks for the send layout (E % R == 0)
    n_shared: int     # shared experts (every token, gate 1)
    dtype: str        # "f32" or "bf16"
    alpha: float      # Switch aux-loss coefficient
    bias: str         # "none" | "zipf" (added to logits) | "normal" (selection only, std 0.1)
    routing: str = "token"   # "token": each token picks k experts; "expert_choice": each expert picks C tokens
    payload: str = "bf16"    # dispatch send buffer: "bf16" (the working dtype) or "fp8" (e4m3 + per-128 scales)

    @property
    def el(self) -> int:
        return 4 if self.dtype == "f32" else 2


CONFIGS = {
    # tiny fp32 layer, the case the oracle finishes in well under a second
    "tiny_fp32": MoEConfig("tiny_fp32", T=256, h=128, E=4, k=2, F=256, gating=GATING_SOFTMAX, cf=0.0,
                           R=2, n_shared=0, dtype="f32", alpha=0.01, bias="none"),
    # page-3 worked shape with capacity 1280 (cf=1.25) and drops in token order
    "page3_cf1.25": MoEConfig("page3_cf1.25", T=4096, h=4096, E=8, k=2, F=12288, gating=GATING_SOFTMAX,
                              cf=1.25, R=8, n_shared=0, dtype="bf16", alpha=0.01, bias="none"),
    # Mixtral-8x7B-shaped, dropless, top-2 renormalised, Zipf(1) skewed load through a logit bias
    "mixtral_zipf": MoEConfig("mixtral_zipf", T=8192, h=4096, E=8, k=2, F=14336,
                              gating=GATING_SOFTMAX_RENORM, cf=0.0, R=8, n_shared=0, dtype="bf16",
                              alpha=0.01, bias="zipf"),
    # DeepSeek-V3-shaped, sigmoid gating with selection-only bias, 1 shared expert, 8 virtual EP ranks
    "deepseek_v3": MoEConfig("deepseek_v3", T=4096, h=7168, E=256, k=8, F=2048,
                             gating=GATING_SIGMOID_BIAS_RENORM, cf=0.0, R=8, n_shared=1, dtype="bf16",
                             alpha=0.01, bias="normal"),
    # Qwen3-MoE-shaped, uniform routing, Switch aux with alpha = 0.01, 8 virtual EP ranks
    "qwen3_moe": MoEConfig("qwen3_moe", T=16384, h=2048, E=128, k=8, F=768, gating=GATING_SOFTMAX,
                           cf=0.0, R=8, n_shared=0, dtype="bf16", alpha=0.01, bias="none"),
    # page-3 shape with expert-choice routing: each of the 8 experts takes C = cf * k * T / E = 1024 tokens
    "page3_expert_choice": MoEConfig("page3_expert_choice", T=4096, h=4096, E=8, k=2, F=12288,
                                     gating=GATING_SOFTMAX, cf=1.0, R=8, n_shared=0, dtype="bf16", alpha=0.01,
                                     bias="none", routing="expert_choice"),
    # Mixtral-shaped layer with the Zipf-skewed logits routed by Sinkhorn balancing (top-2 of the balanced
    # matrix, softmax gates); the per-expert Zipf bias is a logit shift that Sinkhorn undoes exactly
    "mixtral_sinkhorn": MoEConfig("mixtral_sinkhorn", T=8192, h=4096, E=8, k=2, F=14336,
                                  gating="softmax_selbias", cf=0.0, R=8, n_shared=0, dtype="bf16", alpha=0.01,
                                  bias="zipf", routing="sinkhorn"),
    # profiling stand-in for the page-3 shape: identical GEMM tiles (K=4096, 128x256 tiles, same routing and
    # capacity) with F=1536, so that a full ncu capture of the grouped GEMM holds well under 1 GB on the device
    "page3_profile": MoEConfig("page3_profile", T=4096, h=4096, E=8, k=2, F=1536, gating=GATING_SOFTMAX, cf=1.25,
                               R=8, n_shared=0, dtype="bf16", alpha=0.01, bias="none"),
    # profiling stand-in for the DeepSeek-V3-shaped layer's weight-streaming GEMMs: the same h, F, gating, shared
    # expert and about the same rows per expert (k T / E = 128), with 32 experts, so that a full ncu capture of the
    # grouped GEMMs holds ~3 GB of weights on the device (still far more than L2)
    "deepseek_v3_profile": MoEConfig("deepseek_v3_profile", T=1024, h=7168, E=32, k=4, F=2048,
                                     gating=GATING_SIGMOID_BIAS_RENORM, cf=0.0, R=8, n_shared=1, dtype="bf16",
                                     alpha=0.01, bias="normal"),
    # profiling stand-in for the Qwen3-MoE-shaped layer's router and dispatch: the same T, h, E, k, with F = 128
    "qwen3_profile": MoEConfig("qwen3_profile", T=16384, h=2048, E=128, k=8, F=128, gating=GATING_SOFTMAX,
                               cf=0.0, R=8, n_shared=0, dtype="bf16", alpha=0.01, bias="none"),
    # page-3 worked shape with the dispatch send buffer in FP8 (e4m3, one scale per token and 128 columns)
    "page3_fp8": MoEConfig("page3_fp8", T=4096, h=4096, E=8, k=2, F=12288, gating=GATING_SOFTMAX, cf=1.25, R=8,
                           n_shared=0, dtype="bf16", alpha=0.01, bias="none", payload="fp8"),
}
CONFIG_ORDER = ["tiny_fp32", "page3_cf1.25", "mixtral_zipf", "deepseek_v3", "qwen3_moe"]


def get_config(name: str, **overrides) -> MoEConfig:
    """A named workload, optionally with fields replaced (used for reduced-size parity cases)."""
    return dataclasses.replace(CONFIGS[name], **overrides) if overrides else CONFIGS[name]


# ---------------------------------------------------------------------------------------------------------
# random streams and storage formats
# ---------------------------------------------------------------------------------------------------------

S_X, S_WR, S_BIAS, S_WG, S_WU, S_WD, S_SHG, S_SHU, S_SHD, S_XREDRAW = range(1, 11)


def stream(seed: int, stream_id: int, sub: int = 0) -> np.random.Generator:
    """Independent Philox4x32-10 substream for (seed, tensor, sub-index)."""
    key = (int(seed) << 64) | (int(stream_id) << 32) | int(sub)
    return np.random.Generator(np.random.Philox(key=key))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the 16-bit patterns as uint16."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Decode a stored tensor ("f32" float32 array or "bf16" uint16 bit patterns) to float64, exactly."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _normal(gen: np.random.Generator, shape, std: float, dtype: str) -> np.ndarray:
    z = gen.standard_normal(shape, dtype=np.float32)
    z *= np.float32(std)
    return f32_to_bf16_bits(z) if dtype == "bf16" else z


# ---------------------------------------------------------------------------------------------------------
# router inputs
# ---------------------------------------------------------------------------------------------------------

ZIPF_BIAS_FILE = os.path.join(os.path.dirname(__file__), "mixtral_zipf_router_bias.json")


def load_zipf_bias(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    if cfg.name == "mixtral_sinkhorn":                  # same inputs as the Mixtral-shaped workload
        cfg = dataclasses.replace(cfg, name="mixtral_zipf")
    """Per-expert logit bias that makes the Mixtral-shaped workload's expert load follow Zipf(1).

    The values were found by a fixed-point calibration against the oracle's router and stored by
    oracle/calibrate_zipf_bias.py; they are inputs here, not computed."""
    with open(ZIPF_BIAS_FILE) as fh:
        data = json.load(fh)
    key = f"{cfg.name}/T{cfg.T}/h{cfg.h}/E{cfg.E}/k{cfg.k}/seed{seed}"
    if key not in data:
        raise KeyError(f"no stored Zipf bias for {key}; run oracle/calibrate_zipf_bias.py")
    return np.asarray(data[key]["bias"], dtype=np.float32)


def make_x(cfg: MoEConfig, seed: int = 0, redraw: dict | None = None) -> np.ndarray:
    """Tokens x [T, h] ~ N(0, 1) in the working dtype.

    `redraw` maps a row index to a redraw count n > 0: that row is replaced by the n-th draw of its own
    secondary substream (used to move rows off near-ties of the top-k selection)."""
    x = _normal(stream(seed, S_X), (cfg.T, cfg.h), 1.0, cfg.dtype)
    for row, n in sorted((redraw or {}).items()):
        assert 0 <= row < cfg.T and 0 < n < 256
        x[row] = _normal(stream(seed, S_XREDRAW, (n << 24) | row), (cfg.h,), 1.0, cfg.dtype)
    return x


def make_router(cfg: MoEConfig, seed: int = 0, bias: np.ndarray | None = None):
    """Router weight W_r [h, E] ~ N(0, 0.02) and the per-expert bias (float32 [E] or None).

    bias kinds: "normal" draws N(0, 0.1) (selection-only bias of sigmoid gating); "zipf" loads the
    stored calibration unless `bias` is given explicitly; "none" returns None."""
    w_r = _normal(stream(seed, S_WR), (cfg.h, cfg.E), 0.02, cfg.dtype)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float32)
    elif cfg.bias == "normal":
        b = stream(seed, S_BIAS).standard_normal(cfg.E, dtype=np.float32) * np.float32(0.1)
    elif cfg.bias == "zipf":
        b = load_zipf_bias(cfg, seed)
    else:
        b = None
    return w_r, b


# ---------------------------------------------------------------------------------------------------------
# expert weights: nn.Linear layout, W_gate/W_up [F, h], W_down [h, F], std 1/sqrt(fan_in)
# ---------------------------------------------------------------------------------------------------------

def expert_weights(cfg: MoEConfig, e: int, seed: int = 0, shared: bool = False):
    """(W_gate [F,h], W_up [F,h], W_down [h,F]) of routed expert e (or shared expert e)."""
    sg, su, sd = (S_SHG, S_SHU, S_SHD) if shared else (S_WG, S_WU, S_WD)
    wg = _normal(stream(seed, sg, e), (cfg.F, cfg.h), 1.0 / np.sqrt(cfg.h), cfg.dtype)
    wu = _normal(stream(seed, su, e), (cfg.F, cfg.h), 1.0 / np.sqrt(cfg.h), cfg.dtype)
    wd = _normal(stream(seed, sd, e), (cfg.h, cfg.F), 1.0 / np.sqrt(cfg.F), cfg.dtype)
    return wg, wu, wd


def all_expert_weights(cfg: MoEConfig, seed: int = 0, shared: bool = False, threads: int | None = None):
    """Stacked (W_gate [n,F,h], W_up [n,F,h], W_down [n,h,F]) for all routed (or shared) experts."""
    n = cfg.n_shared if shared else cfg.E
    st = np.uint16 if cfg.dtype == "bf16" else np.float32
    wg = np.empty((n, cfg.F, cfg.h), st)
    wu = np.empty((n, cfg.F, cfg.h), st)
    wd = np.empty((n, cfg.h, cfg.F), st)

    def one(e):
        wg[e], wu[e], wd[e] = expert_weights(cfg, e, seed, shared)

    with ThreadPoolExecutor(max_workers=threads or min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(one, range(n)))
    return wg, wu, wd
