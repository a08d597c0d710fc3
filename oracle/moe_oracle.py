"""Plain, slow, obviously-correct CPU oracle of the MoE layer forward hot path (float64).

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this module. The CUDA product path never calls it, and it shares no code with that path: it reads the
same seeded inputs (moe_inputs) and nothing else.

Page keys used in the citations below:
  [MEG6]  "Megatron-LM 分布式训练（六）：MoE 专家并行 EP 与上下文并行 CP" (swordlidev blog)
  [EP7]   "专家并行" (formulaic docs, distributed training / 7-expert-parallel)
  [L7]    "v6 长序列和 MoE: Context Parallel 与 Expert Parallel" (ml-interview infra-l7)
  [B10.5] "10.5 序列并行与专家并行" (llm-fullstack-book)

Every step is the plain definition, in the pages' order: router -> top-k gates -> dispatch (with optional
capacity) -> per-expert SwiGLU FFN -> combine ([MEG6] "MoE 层的数据流"; [L7] shape table under
"NVIDIA 原题: Implement MoE and show the dimensions"). Library primitives used as steps: numpy matmul
(float64), numpy stable argsort, exp. Readings of points the pages leave open are noted where they apply.

Parity pins (tests/test_oracle_pins.py): shape table and C=1280 of [L7]; brute-force top-k by subset
enumeration; sum of counts = k*T; brute-force loop dispatch; stable per-expert token order; identity
experts giving y = sum gates*x (and y = x under renormalised gates); E=1,k=1 reducing to a dense SwiGLU
FFN checked against scalar loops; aux = alpha exactly at a uniform split and >= alpha when f = P;
FLOP and byte counts of [L7] "EP" (6.2 ms at 400 TFLOPS, 64 MiB per dispatch). The backward
(combine_backward, swiglu_ffn_backward, route_backward, moe_layer_backward) is pinned by central differences
of the forward in every gating mode with and without drops, a hand-derived 1 x 1 SwiGLU derivative, and zero
gradients on dropped pairs and pad rows. The FP8 payload (e4m3_value, e4m3_encode, fp8_quantize_rows,
fp8_dequantize_rows, dispatch_payload_fp8) is pinned by hand-written code values, a brute-force nearest
search with the tie rule, exact midpoints, saturation, the amax -> 448 scale and the half-ulp error bound. No
function is unpinned.
"""
from __future__ import annotations

import math

import numpy as np

SOFTMAX = "softmax"
SOFTMAX_RENORM = "softmax_renorm"
SIGMOID_BIAS_RENORM = "sigmoid_bias_renorm"


# ---------------------------------------------------------------------------------------------------------
# capacity
# ---------------------------------------------------------------------------------------------------------

def capacity(cf: float, k: int, T: int, E: int) -> int:
    """Per-expert slot limit C = cf * k * T / E ([L7] "Capacity" bullet under the shape table:
    1.25 * 2 * 4096 / 8 = 1280). cf = 0 means dropless (Megatron's default, same bullet) and returns 0.
    Reading: a non-integer product is rounded up, so that C >= the formula's value."""
    if cf <= 0:
        return 0
    return int(math.ceil(cf * k * T / E - 1e-9))


# ---------------------------------------------------------------------------------------------------------
# router: gating GEMM, gates, top-k, aux-loss terms
# ---------------------------------------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_r: np.ndarray, bias: np.ndarray | None, gating: str) -> np.ndarray:
    """logits = hidden_states @ W_router ([MEG6] "Router" step 1; [L7] table row "router": x times
    Wr [h, E]). In the softmax modes a per-expert bias (if given) is added to the logits; under sigmoid
    gating the bias is only a selection term ([L7] "Load balancing loss", DeepSeek-V3 aux-loss-free bias)
    and is applied in `route`, not here."""
    L = np.asarray(x, np.float64) @ np.asarray(w_r, np.float64)
    if bias is not None and gating != SIGMOID_BIAS_RENORM:
        L = L + np.asarray(bias, np.float64)[None, :]
    return L


def softmax(L: np.ndarray) -> np.ndarray:
    """Row softmax in float64, with the row max subtracted first."""
    z = np.exp(L - L.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def sigmoid(L: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-L))


def route(L: np.ndarray, k: int, gating: str, bias: np.ndarray | None = None, alpha: float = 0.01) -> dict:
    """Top-k routing and the Switch aux-loss terms ([MEG6] "Router" step 2; [L7] table row "top-k" and
    "Load balancing loss").

    selection score: the logits (softmax modes; softmax is monotone so this is selection on the
      probabilities), or sigmoid(L) + b (sigmoid mode, b used for selection only).
    order: descending score; equal scores -> lower expert index first (reading: the pages are silent).
    gates: softmax mode -> the full-softmax probability of each chosen expert, not renormalised (the table
      takes the top-k of the softmax output); softmax_renorm -> p / sum over the k chosen p;
      sigmoid -> s / sum over the k chosen s (bias excluded).
    counts n_e: assignments per expert before any capacity limit (sum = k*T).
    f_e = n_e / (k*T); P_e = mean over tokens of the router probability of e (softmax modes: the full
      softmax; sigmoid mode, reading: s_e / sum_e' s_e'); aux = alpha * E * sum_e f_e P_e.
    margins: per token, the gaps between consecutive entries of its top-(k+1) sorted scores (covering
      the order inside the top-k and the k / k+1 boundary)."""
    T, E = L.shape
    assert 1 <= k <= E
    if gating == SIGMOID_BIAS_RENORM:
        s = sigmoid(L)
        score = s + (np.asarray(bias, np.float64)[None, :] if bias is not None else 0.0)
        prob = s / s.sum(axis=1, keepdims=True)
    else:
        prob = softmax(L)
        score = L
    order = np.argsort(-score, axis=1, kind="stable")
    ids = order[:, :k]
    rows = np.arange(T)[:, None]
    if gating == SOFTMAX:
        gates = prob[rows, ids]
    elif gating == SOFTMAX_RENORM:
        pk = prob[rows, ids]
        gates = pk / pk.sum(axis=1, keepdims=True)
    elif gating == SIGMOID_BIAS_RENORM:
        sk = s[rows, ids]
        gates = sk / sk.sum(axis=1, keepdims=True)
    else:
        raise ValueError(gating)
    counts = np.bincount(ids.ravel(), minlength=E).astype(np.int64)
    f = counts / float(k * T)
    P = prob.mean(axis=0)
    aux = alpha * E * float(np.sum(f * P))
    top = np.take_along_axis(score, order[:, :min(k + 1, E)], axis=1)
    gaps = top[:, :-1] - top[:, 1:]
    return dict(logits=L, ids=ids.astype(np.int32), gates=gates, counts=counts, f=f, P=P, aux=aux,
                prob=prob, score=score, gaps=gaps)


def near_tie_rows(gaps: np.ndarray, thresh: float) -> np.ndarray:
    """Tokens whose top-k selection or order has a score gap below `thresh`."""
    if gaps.shape[1] == 0:
        return np.zeros(0, np.int64)
    return np.nonzero(gaps.min(axis=1) < thresh)[0]


# ---------------------------------------------------------------------------------------------------------
# dispatch: group by expert (stable, token order), capacity mask, EP-rank-major layout
# ---------------------------------------------------------------------------------------------------------

def dispatch(ids: np.ndarray, E: int, C: int, R: int) -> dict:
    """Token dispatch into per-expert contiguous blocks ([L7] table row "dispatch": group by expert, at
    most C tokens per group, pad the rest; [L7] "自测" answer: over-capacity tokens are dropped, unfilled
    slots padded; [L7] follow-up: sort tokens by expert and run one grouped GEMM; [EP7] "All2All": the
    (E, C, M) input pre-sorted into blocks by destination expert).

    slot(t, j) = number of earlier assignments (in token order t, then j) to the same expert.
    Reading: over-capacity drops go in token order (a token never picks one expert twice, so within an
    expert the order is by t alone). keep iff dropless (C == 0) or slot < C.
    dropless: offsets = exclusive prefix sum of n_e, rows = k*T. capacity: offsets[e] = e*C, rows = E*C.
    dest_row = offsets[e] + slot for kept pairs, -1 for dropped ones; src_token/src_slot invert it (-1 on
    pad rows). EP layout ([EP7] "All2All": experts on ranks in contiguous blocks, the all-to-all being a
    block transpose; [MEG6] "专家并行 EP"): rank r owns experts [r*E/R, (r+1)*E/R), so the expert-major
    buffer is already rank-major; rank_offsets[r] = offsets[r*E/R], rank_counts[r] = kept rows of r."""
    T, k = ids.shape
    assert E % R == 0
    flat = ids.ravel().astype(np.int64)
    A = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    order = np.argsort(flat, kind="stable")           # assignments grouped by expert, token order kept
    starts = np.concatenate([[0], np.cumsum(counts)])
    slot = np.empty(A, np.int64)
    slot[order] = np.arange(A) - starts[flat[order]]
    keep = np.ones(A, bool) if C == 0 else slot < C
    kept_counts = counts if C == 0 else np.minimum(counts, C)
    if C == 0:
        offsets = starts.copy()
        rows = A
    else:
        offsets = np.arange(E + 1, dtype=np.int64) * C
        rows = E * C
    dest = np.where(keep, offsets[flat] + slot, -1)
    src_token = np.full(rows, -1, np.int64)
    src_slot = np.full(rows, -1, np.int64)
    kept_idx = np.nonzero(keep)[0]
    src_token[dest[kept_idx]] = kept_idx // k
    src_slot[dest[kept_idx]] = kept_idx % k
    epr = E // R
    rank_offsets = offsets[::epr].copy()
    rank_counts = kept_counts.reshape(R, epr).sum(axis=1)
    return dict(counts=counts, kept_counts=kept_counts, offsets=offsets, rows=rows,
                slot=slot.reshape(T, k), dest_row=dest.reshape(T, k), drop_mask=(~keep).reshape(T, k),
                src_token=src_token, src_slot=src_slot, rank_offsets=rank_offsets, rank_counts=rank_counts)


def dispatch_payload(x: np.ndarray, d: dict) -> np.ndarray:
    """buf[rows, h]: buf[dest_row(t, j)] = x[t] for kept pairs; pad rows are zero (reading of [L7] table
    row "dispatch", which pads the unfilled slots of each expert)."""
    buf = np.zeros((d["rows"], x.shape[1]), dtype=x.dtype)
    live = d["src_token"] >= 0
    buf[live] = x[d["src_token"][live]]
    return buf


# ---------------------------------------------------------------------------------------------------------
# experts: SwiGLU FFN h -> F -> h (three matrices, [L7] "dense FFN ... 3 x 4096 x 12288")
# ---------------------------------------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(X: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """out = (silu(X W_gate^T) * (X W_up^T)) W_down^T, weights in nn.Linear layout ([F,h], [F,h], [h,F]).
    Reading: the standard SwiGLU, no biases (the page gives only its three matrices)."""
    X = np.asarray(X, np.float64)
    a = silu(X @ w_gate.T) * (X @ w_up.T)
    return a @ w_down.T


def expert_outputs(buf: np.ndarray, d: dict, weights) -> np.ndarray:
    """eout[rows, h] for every kept row: expert e's FFN on its block [offsets[e], offsets[e]+kept[e])
    ([MEG6] "experts ... (GroupedGEMM)"; [L7] table row "expert"). `weights(e)` returns float64
    (W_gate, W_up, W_down). Pad rows stay zero."""
    eout = np.zeros((d["rows"], buf.shape[1]), np.float64)
    for e in range(len(d["kept_counts"])):
        n = int(d["kept_counts"][e])
        if n == 0:
            continue
        o = int(d["offsets"][e])
        eout[o:o + n] = swiglu_ffn(buf[o:o + n], *weights(e))
    return eout


# ---------------------------------------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------------------------------------

def combine(eout: np.ndarray, dest_row: np.ndarray, gates: np.ndarray, shared_out: np.ndarray | None = None):
    """y[t] = sum over kept j of gate[t, j] * eout[dest_row[t, j]] (+ shared expert output, gate 1)
    ([L7] table row "combine": back to the original position, the k outputs summed weighted by gate;
    [EP7] forward pass: top-2 weighted; [MEG6] data flow: "+ shared_experts"). A dropped pair adds
    nothing (it reaches the next layer only through the residual, [L7] "自测"), and gates are not
    renormalised after a drop (reading). No residual is added here."""
    T, k = dest_row.shape
    y = np.zeros((T, eout.shape[1]), np.float64) if shared_out is None else np.array(shared_out, np.float64)
    for j in range(k):
        kept = dest_row[:, j] >= 0
        y[kept] += gates[kept, j][:, None] * eout[dest_row[kept, j]]
    return y


# ---------------------------------------------------------------------------------------------------------
# whole layer
# ---------------------------------------------------------------------------------------------------------

def moe_layer(x, w_r, bias, weights, *, k: int, gating: str, cf: float, R: int, alpha: float = 0.01,
              shared=None, experts: str = "swiglu", payload: str = "bf16") -> dict:
    """Full forward: router -> dispatch -> experts -> combine. Inputs are float64 arrays of the
    dtype-rounded values. `weights(e)` gives expert e's matrices; `shared()` the shared expert's (or
    None). experts="identity" replaces each expert by the identity (eout = buf) for the pins.
    payload="fp8": the routed experts read the dequantised FP8 send buffer (dispatch_payload_fp8); the shared
    expert reads x itself (it is not dispatched)."""
    x = np.asarray(x, np.float64)
    T, h = x.shape
    E = np.asarray(w_r).shape[1]
    L = router_logits(x, w_r, bias, gating)
    r = route(L, k, gating, bias, alpha)
    C = capacity(cf, k, T, E)
    d = dispatch(r["ids"], E, C, R)
    if payload == "fp8":
        buf = fp8_dequantize_rows(*dispatch_payload_fp8(x, d))
    else:
        buf = dispatch_payload(x, d)
    eout = buf.copy() if experts == "identity" else expert_outputs(buf, d, weights)
    sh = swiglu_ffn(x, *shared()) if shared is not None else None
    y = combine(eout, d["dest_row"], r["gates"], sh)
    return dict(router=r, dispatch=d, C=C, buf=buf, eout=eout, shared_out=sh, y=y)


def moe_layer_tokens(tokens, x, route_out: dict, disp: dict, weights, shared=None) -> np.ndarray:
    """y for a subset of tokens, from the full router and dispatch results: for each chosen token t,
    y[t] = sum over kept j of gate[t, j] * FFN_{e(t, j)}(x[t]) (+ shared FFN(x[t])). Dispatch copies x[t]
    to its row unchanged, so this is the layer's output for those tokens, computed one token at a time
    instead of for the whole batch."""
    tokens = np.asarray(tokens, np.int64)
    x = np.asarray(x, np.float64)
    ids, gates, dest = route_out["ids"], route_out["gates"], disp["dest_row"]
    y = np.zeros((tokens.size, x.shape[1]), np.float64)
    if shared is not None:
        y += swiglu_ffn(x[tokens], *shared())
    by_expert: dict[int, list[tuple[int, int]]] = {}
    for i, t in enumerate(tokens):
        for j in range(ids.shape[1]):
            if dest[t, j] >= 0:
                by_expert.setdefault(int(ids[t, j]), []).append((i, j))
    for e, pairs in sorted(by_expert.items()):
        ii = np.array([p[0] for p in pairs])
        jj = np.array([p[1] for p in pairs])
        out = swiglu_ffn(x[tokens[ii]], *weights(e))
        y[ii] += gates[tokens[ii], jj][:, None] * out
    return y


# ---------------------------------------------------------------------------------------------------------
# algorithmic work (the units the roofline numbers divide by)
# ---------------------------------------------------------------------------------------------------------

def ffn_flops(rows: int, h: int, F: int) -> int:
    """Multiply-adds of three h x F matmuls per row, 2 flops each: 6 h F per row ([L7] "EP": 6.2 ms at
    400 TFLOPS for T=4096, k=2, h=4096, F=12288)."""
    return 6 * h * F * rows


def dispatch_bytes(T: int, kept: int, h: int, el: int) -> int:
    """Bytes the dispatch must move: read T token rows, write one row per kept assignment ([L7] "EP":
    64 MiB for one dispatch at T=4096, k=2, h=4096 in bf16 counts the written rows)."""
    return (T + kept) * h * el


# ---------------------------------------------------------------------------------------------------------
# expert-choice routing ([B10.5] 10.5.6 "负载均衡问题", the expert-choice bullet: the routing direction is
# reversed, each expert takes the fixed number of highest-scoring tokens among all tokens)
# ---------------------------------------------------------------------------------------------------------

def expert_choice(L: np.ndarray, C: int) -> dict:
    """Each expert e selects the C tokens with the highest router probability p[t, e] (the full softmax over
    experts of token t's logits: the token-choice router's probability, reading).

    Readings (the page gives one sentence): equal scores -> lower token index first; the selected tokens of
    expert e occupy rows e*C .. e*C + C - 1 in ascending token order; the gate of a selected pair is p[t, e];
    a token no expert selects contributes nothing (y = 0 for it, the residual being outside the layer).
    Returns tokens [E, C], gates [E, C], slot [T, E] (j or -1) and gaps [E] (score gap between the C-th
    and the (C+1)-th selected candidate, for the near-tie policy)."""
    T, E = L.shape
    assert 1 <= C <= T
    p = softmax(L)
    tokens = np.empty((E, C), np.int64)
    gates = np.empty((E, C), np.float64)
    slot = np.full((T, E), -1, np.int64)
    gaps = np.full(E, np.inf)
    for e in range(E):
        order = np.argsort(-p[:, e], kind="stable")      # descending score, ties -> lower token index
        chosen = np.sort(order[:C])
        tokens[e] = chosen
        gates[e] = p[chosen, e]
        slot[chosen, e] = np.arange(C)
        if C < T:
            gaps[e] = p[order[C - 1], e] - p[order[C], e]
    return dict(prob=p, tokens=tokens, gates=gates, slot=slot, gaps=gaps)


def expert_choice_layer(x, w_r, weights, C: int, shared=None) -> dict:
    """Expert-choice layer forward: logits, selection, buf[e*C + j] = x[tokens[e, j]], expert FFN,
    y[t] = sum over the experts e that selected t (ascending e) of gate * FFN_e(x[t]) (+ shared FFN)."""
    x = np.asarray(x, np.float64)
    L = router_logits(x, w_r, None, SOFTMAX)
    ec = expert_choice(L, C)
    E = L.shape[1]
    buf = x[ec["tokens"].reshape(-1)]
    eout = np.empty_like(buf)
    for e in range(E):
        eout[e * C:(e + 1) * C] = swiglu_ffn(buf[e * C:(e + 1) * C], *weights(e))
    y = np.zeros_like(x) if shared is None else swiglu_ffn(x, *shared())
    for e in range(E):
        y[ec["tokens"][e]] += ec["gates"][e][:, None] * eout[e * C:(e + 1) * C]
    return dict(logits=L, ec=ec, buf=buf, eout=eout, y=y)


# ---------------------------------------------------------------------------------------------------------
# Sinkhorn routing ([MEG6] "Router": Sinkhorn iterations normalise the routing matrix to a doubly stochastic
# one, which balances the experts without an aux loss)
# ---------------------------------------------------------------------------------------------------------

SINKHORN_ITERS = 16
SOFTMAX_SELBIAS = "softmax_selbias"      # select on logits + bias, gate = the softmax probability


def sinkhorn_scaling(L: np.ndarray, n_iter: int = SINKHORN_ITERS):
    """Sinkhorn-Knopp on K = exp(L - rowmax) [T, E]: starting from r = 1, n_iter times set the column scalings
    c_e = (T / E) / sum_t K[t,e] r_t (columns sum to T / E), then the row scalings r_t = 1 / sum_e K[t,e] c_e
    (rows sum to 1). Readings (the page names the method only): a fixed number of iterations (16), column
    targets T / E. Returns (c, r)."""
    T, E = L.shape
    K = np.exp(L - L.max(axis=1, keepdims=True))
    r = np.ones(T)
    c = np.ones(E)
    for _ in range(n_iter):
        c = (T / E) / (K * r[:, None]).sum(axis=0)
        r = 1.0 / (K * c[None, :]).sum(axis=1)
    return c, r


def route_sinkhorn(L: np.ndarray, k: int, n_iter: int = SINKHORN_ITERS, alpha: float = 0.01) -> dict:
    """Top-k of the Sinkhorn-balanced matrix M = diag(r) K diag(c): a row scaling does not change a row's
    order, so this is the top-k of L[t,e] + log c_e. Reading: the gates stay the router's softmax
    probabilities of the chosen experts (not renormalised); counts, f, P and aux as in `route`."""
    c, _ = sinkhorn_scaling(L, n_iter)
    return route_selbias(L, k, np.log(c), alpha)


def route_selbias(L: np.ndarray, k: int, sel_bias: np.ndarray, alpha: float = 0.01) -> dict:
    """Select the top-k of L + sel_bias (descending, ties -> lower index); gates = softmax(L) of the chosen
    (not renormalised); counts, f, P = mean softmax, aux = alpha E sum f P; gaps on the selection score."""
    T, E = L.shape
    prob = softmax(L)
    score = L + np.asarray(sel_bias, np.float64)[None, :]
    order = np.argsort(-score, axis=1, kind="stable")
    ids = order[:, :k]
    gates = prob[np.arange(T)[:, None], ids]
    counts = np.bincount(ids.ravel(), minlength=E).astype(np.int64)
    f = counts / float(k * T)
    P = prob.mean(axis=0)
    top = np.take_along_axis(score, order[:, :min(k + 1, E)], axis=1)
    return dict(logits=L, ids=ids.astype(np.int32), gates=gates, counts=counts, f=f, P=P,
                aux=alpha * E * float(np.sum(f * P)), prob=prob, score=score, gaps=top[:, :-1] - top[:, 1:],
                sel_bias=np.asarray(sel_bias, np.float64))


# ---------------------------------------------------------------------------------------------------------
# backward of the layer ([EP7] "BWD（反向传播）": each expert computes its own weight gradients, and in the
# overlap notes the gradients return to the experts along the routing path). The pages give no formulas;
# reading: the chain rule through the forward above, with the top-k selection, the counts (hence f) and the
# capacity drops held constant (piecewise constant in the inputs). Upstream gradients: dy for y and d_aux
# for the aux loss, i.e. the gradient of <dy, y> + d_aux * aux.
# ---------------------------------------------------------------------------------------------------------

def combine_backward(dy: np.ndarray, eout: np.ndarray, dest_row: np.ndarray, gates: np.ndarray, rows: int):
    """Through y[t] = sum_kept gate[t,j] eout[dest_row[t,j]]: d_eout[r] = gate[t,j] dy[t] on kept rows (zero on
    pad rows); d_gates[t,j] = <dy[t], eout[dest_row[t,j]]> for kept pairs, 0 for dropped ones."""
    T, k = dest_row.shape
    d_eout = np.zeros((rows, dy.shape[1]), np.float64)
    d_gates = np.zeros((T, k), np.float64)
    for j in range(k):
        kept = dest_row[:, j] >= 0
        r = dest_row[kept, j]
        d_eout[r] = gates[kept, j][:, None] * dy[kept]
        d_gates[kept, j] = np.sum(dy[kept] * eout[r], axis=1)
    return d_eout, d_gates


def swiglu_ffn_backward(X: np.ndarray, w_gate, w_up, w_down, d_out: np.ndarray):
    """Backward of out = (silu(G) * U) W_down^T with G = X W_gate^T, U = X W_up^T:
    d_a = d_out W_down; dW_down = d_out^T a; dG = d_a * U * silu'(G) with silu'(z) = s(z) (1 + z (1 - s(z))),
    s the logistic function; dU = d_a * silu(G); dX = dG W_gate + dU W_up; dW_gate = dG^T X; dW_up = dU^T X."""
    X = np.asarray(X, np.float64)
    G = X @ w_gate.T
    U = X @ w_up.T
    s = sigmoid(G)
    a = G * s * U
    d_a = d_out @ w_down
    dG = d_a * U * s * (1.0 + G * (1.0 - s))
    dU = d_a * G * s
    return dict(dX=dG @ w_gate + dU @ w_up, dW_gate=dG.T @ X, dW_up=dU.T @ X, dW_down=d_out.T @ a,
                d_a=d_a, dG=dG, dU=dU)


def route_backward(L: np.ndarray, r: dict, d_gates: np.ndarray, gating: str, alpha: float, d_aux: float):
    """d_logits from the gate gradients and the aux loss.
    Gates (see `route`): softmax g_j = p[ids_j]; softmax_renorm g_j = p[ids_j] / S; sigmoid g_j = s[ids_j] / S
    (S the sum over the k chosen). aux = alpha E sum_e f_e P_e with P_e = mean_t q[t, e], q = p (softmax modes)
    or s / sum_e s (sigmoid mode), so d aux / d q[t, e] = alpha E f_e / T.
    Softmax modes: dq -> dL by the softmax Jacobian dL = p * (dp - <dp, p>). Sigmoid mode: dq -> ds by the
    Jacobian of s / sum(s), then dL = ds * s (1 - s). The softmax mode with a selection-only bias (Sinkhorn
    routing: the ids are chosen on L + log c, the gates are p[ids]) is the plain softmax mode here: the
    selection is held constant, so the bias and the column scalings that produced it carry no gradient."""
    T, E = L.shape
    ids, gates, f = r["ids"], r["gates"], r["f"]
    k = ids.shape[1]
    rows = np.arange(T)[:, None]
    c = d_aux * alpha * E * np.asarray(f, np.float64) / T          # d aux / d q[t, e], the same for every t
    if gating == SIGMOID_BIAS_RENORM:
        s = sigmoid(L)
        ds = np.zeros((T, E))
        Sk = s[rows, ids].sum(axis=1, keepdims=True)
        dsk = (d_gates - np.sum(d_gates * gates, axis=1, keepdims=True)) / Sk
        np.add.at(ds, (np.repeat(np.arange(T), k), ids.ravel()), dsk.ravel())
        Ssum = s.sum(axis=1, keepdims=True)
        q = s / Ssum
        dq = np.broadcast_to(c[None, :], (T, E))
        ds += (dq - np.sum(dq * q, axis=1, keepdims=True)) / Ssum
        return ds * s * (1.0 - s)
    p = softmax(L)
    dp = np.zeros((T, E))
    if gating in (SOFTMAX, SOFTMAX_SELBIAS):
        np.add.at(dp, (np.repeat(np.arange(T), k), ids.ravel()), d_gates.ravel())
    elif gating == SOFTMAX_RENORM:
        Sk = p[rows, ids].sum(axis=1, keepdims=True)
        dpk = (d_gates - np.sum(d_gates * gates, axis=1, keepdims=True)) / Sk
        np.add.at(dp, (np.repeat(np.arange(T), k), ids.ravel()), dpk.ravel())
    else:
        raise ValueError(gating)
    dp = dp + c[None, :]
    return p * (dp - np.sum(dp * p, axis=1, keepdims=True))


def moe_layer_backward(x, w_r, bias, weights, fwd: dict, dy, *, gating: str, alpha: float = 0.01,
                       d_aux: float = 1.0, shared=None) -> dict:
    """Gradients of <dy, y> + d_aux * aux for the forward `fwd` = moe_layer(...): dx, dW_r, d_bias (softmax
    modes; the sigmoid-mode bias only selects and gets none), per-expert dW_gate / dW_up / dW_down, the shared
    expert's, and the intermediate gradients (d_eout, d_gates, d_buf, d_logits)."""
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    r, d = fwd["router"], fwd["dispatch"]
    E = np.asarray(w_r).shape[1]
    d_eout, d_gates = combine_backward(dy, fwd["eout"], d["dest_row"], r["gates"], d["rows"])
    d_buf = np.zeros_like(fwd["buf"], dtype=np.float64)
    dW = []
    for e in range(E):
        n, o = int(d["kept_counts"][e]), int(d["offsets"][e])
        wg, wu, wd = weights(e)
        if n == 0:
            dW.append((np.zeros_like(wg), np.zeros_like(wu), np.zeros_like(wd)))
            continue
        g = swiglu_ffn_backward(fwd["buf"][o:o + n], wg, wu, wd, d_eout[o:o + n])
        d_buf[o:o + n] = g["dX"]
        dW.append((g["dW_gate"], g["dW_up"], g["dW_down"]))
    dx = np.zeros_like(x)
    live = d["src_token"] >= 0
    np.add.at(dx, d["src_token"][live], d_buf[live])                 # dispatch copied x[t] to each kept row
    sh = None
    if shared is not None:
        sh = swiglu_ffn_backward(x, *shared(), dy)
        dx += sh["dX"]
    d_logits = route_backward(fwd["router"]["logits"], r, d_gates, gating, alpha, d_aux)
    dx += d_logits @ np.asarray(w_r, np.float64).T
    dW_r = x.T @ d_logits
    d_bias = d_logits.sum(axis=0) if (bias is not None and gating != SIGMOID_BIAS_RENORM) else None
    return dict(dx=dx, dW_r=dW_r, d_bias=d_bias, dW=dW, shared=sh, d_eout=d_eout, d_gates=d_gates, d_buf=d_buf,
                d_logits=d_logits)


# ---------------------------------------------------------------------------------------------------------
# FP8 dispatch payload ([B10.5] 10.5.7 "低精度传输与压缩": activations crossing nodes can use a low-precision
# format such as FP8, halving the bytes with negligible effect on model quality). The page fixes neither the
# format nor the scaling; readings: e4m3 in its finite-only variant (1 sign, 4 exponent bits with bias 7, 3
# mantissa bits, subnormals, largest magnitude 448, no infinities), one fp32 scale per token and per 128 columns
# s = amax / 448 (s = 1 for an all-zero block), code = round-to-nearest-even of fp32(x) / s on the e4m3 grid
# with saturation to +-448; dequantisation as the GEMM prologue does it: bf16(fp32(value(code)) * s).
# ---------------------------------------------------------------------------------------------------------

E4M3_MAX = 448.0
FP8_BLOCK = 128


def e4m3_value(code: int) -> float:
    """Value of an e4m3 byte: exponent field 0 -> subnormal m/8 * 2^-6; else (1 + m/8) * 2^(e - 7);
    code 0x7f / 0xff (exponent and mantissa all ones) is NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_value(c) for c in range(256)])


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3 code of each float (ties to the code with an even mantissa), saturating beyond 448.
    Zero maps to +0 (code 0) and -0 to code 0x80."""
    v = np.asarray(v, np.float64)
    tab = e4m3_table()
    pos = np.array([c for c in range(0x7F)])                 # +0 .. 448, increasing values
    pv = tab[pos]
    a = np.minimum(np.abs(v), E4M3_MAX)
    idx = np.searchsorted(pv, a)                              # pv[idx-1] < a <= pv[idx]
    idx = np.clip(idx, 1, len(pv) - 1)
    lo, hi = pos[idx - 1], pos[idx]
    dlo, dhi = a - tab[lo], tab[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == 0, 0, code)
    neg = np.signbit(v)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def fp8_quantize_rows(X: np.ndarray):
    """Per row and per 128 columns: s = fp32(amax) / 448 in fp32 (1 for an all-zero block); codes =
    e4m3_encode(fp32(x) / s in fp32). Returns (codes uint8 [rows, h], scales float32 [rows, h / 128])."""
    X = np.asarray(X, np.float32)
    n, h = X.shape
    assert h % FP8_BLOCK == 0
    blocks = X.reshape(n, h // FP8_BLOCK, FP8_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    scales = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (blocks / scales[:, :, None]).astype(np.float32)
    return e4m3_encode(q).reshape(n, h), scales


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) and return them as float64."""
    b = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def fp8_dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """bf16(fp32(value(code)) * s) per element, as float64."""
    n, h = codes.shape
    vals = e4m3_table()[codes].astype(np.float32).reshape(n, h // FP8_BLOCK, FP8_BLOCK)
    return bf16_round((vals * np.asarray(scales, np.float32)[:, :, None]).reshape(n, h))


def dispatch_payload_fp8(x: np.ndarray, d: dict):
    """The dispatch send buffer in FP8: every kept row holds its token's codes and scales (each token quantised
    once); pad rows hold code 0 and scale 0."""
    codes_t, scales_t = fp8_quantize_rows(x)
    codes = np.zeros((d["rows"], x.shape[1]), np.uint8)
    scales = np.zeros((d["rows"], x.shape[1] // FP8_BLOCK), np.float32)
    live = d["src_token"] >= 0
    codes[live] = codes_t[d["src_token"][live]]
    scales[live] = scales_t[d["src_token"][live]]
    return codes, scales
