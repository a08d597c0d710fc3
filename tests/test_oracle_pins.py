"""Pins of the CPU oracle to facts fixed by the pages and by mathematics (no GPU).

Each test checks the oracle against something other than itself: values the pages print (golden files),
closed forms, invariants, or brute force on tiny inputs. tests/test_oracle_mutations.py plants plausible
mistakes in the oracle and checks that these pins catch them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# ------------------------------------------------------------------------------------------- page numbers

def test_page3_capacity_and_shapes():
    """Shape table and C = 1280 of the page-3 worked example, run through the oracle (identity experts,
    so no FFN is needed for the shapes)."""
    g = _golden("page3_shape_table.json")
    T, h, E, k = g["T"], g["h"], g["E"], g["k"]
    assert O.capacity(g["cf"], k, T, E) == g["capacity"]
    cfg = moe_inputs.get_config("page3_cf1.25")
    assert (cfg.T, cfg.h, cfg.E, cfg.k, cfg.cf, cfg.F) == (T, h, E, k, g["cf"], g["F"])
    x = moe_inputs.to_f64(moe_inputs.make_x(cfg), cfg.dtype)
    w_r, b = moe_inputs.make_router(cfg)
    out = O.moe_layer(x, moe_inputs.to_f64(w_r, cfg.dtype), b, None, k=k, gating=cfg.gating, cf=cfg.cf,
                      R=cfg.R, experts="identity")
    s = g["shapes"]
    assert list(x.shape) == s["input_x"]
    assert list(out["router"]["logits"].shape) == s["router"]
    assert list(out["router"]["ids"].shape) == s["top_k"]
    assert list(out["buf"].reshape(E, out["C"], h).shape) == s["dispatch"]
    assert list(out["eout"].reshape(E, out["C"], h).shape) == s["expert"]
    assert list(out["y"].shape) == s["combine_y"]


def test_page3_flops_and_dispatch_bytes():
    """6 h F flops per assignment reproduce the page's 6.2 ms at 400 TFLOPS; one bf16 dispatch of
    k*T rows of h is 64 MiB; a SwiGLU FFN of 3 h F parameters is ~151M (x8 experts ~1.21B)."""
    g = _golden("page3_ep_costs.json")
    T, h, k, F, E = g["T"], g["h"], g["k"], g["F"], g["E"]
    ms = O.ffn_flops(k * T, h, F) / (g["assumed_tflops"] * 1e12) * 1e3
    assert abs(ms - g["expert_compute_ms"]) < 0.05
    written = O.dispatch_bytes(T, k * T, h, 2) - T * h * 2
    assert written == g["dispatch_bytes_MiB"] * 2**20
    assert round(3 * h * F / 1e6) == g["dense_swiglu_params_M"]
    assert round(E * 3 * h * F / 1e9, 2) == g["moe_layer_params_B"]


def test_capacity_rounding():
    assert O.capacity(0, 2, 4096, 8) == 0
    assert O.capacity(1.0, 2, 4096, 8) == 1024
    assert O.capacity(1.0, 1, 10, 3) == 4          # 3.33 rounds up
    assert O.capacity(0.5, 2, 4096, 8) == 512


# ------------------------------------------------------------------------------------------------ router

def _brute_topk(score, k):
    """Max-sum k-subset; among equal sums the lexicographically smallest index set; ordered by
    descending score then index."""
    E = len(score)
    best, best_set = None, None
    for sub in itertools.combinations(range(E), k):
        s = sum(score[i] for i in sub)
        if best is None or s > best:
            best, best_set = s, sub
    return sorted(best_set, key=lambda i: (-score[i], i))


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (6, 3), (8, 2), (8, 8)])
def test_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    L = rng.standard_normal((48, E))
    r = O.route(L, k, O.SOFTMAX)
    for t in range(L.shape[0]):
        assert list(r["ids"][t]) == _brute_topk(list(L[t]), k)


def test_topk_exact_ties_take_lower_index():
    L = np.array([[3.0, 1.0, 1.0, 0.0], [0.0, 0.0, 0.0, 0.0], [1.0, 2.0, 2.0, 2.0]])
    r = O.route(L, 2, O.SOFTMAX)
    assert r["ids"].tolist() == [[0, 1], [0, 1], [1, 2]]
    for t in range(3):
        assert list(r["ids"][t]) == _brute_topk(list(L[t]), 2)


def test_sigmoid_selection_uses_bias_but_gates_do_not():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((40, 8))
    b = rng.standard_normal(8) * 0.5
    r = O.route(L, 3, O.SIGMOID_BIAS_RENORM, bias=b)
    for t in range(40):
        s = [1.0 / (1.0 + math.exp(-v)) for v in L[t]]
        sel = _brute_topk([s[e] + b[e] for e in range(8)], 3)
        assert list(r["ids"][t]) == sel
        tot = sum(s[e] for e in sel)
        assert np.allclose(r["gates"][t], [s[e] / tot for e in sel], rtol=1e-14)


def test_sigmoid_constant_bias_changes_nothing():
    """Under sigmoid gating the bias only ranks experts ([L7] "Load balancing loss", DeepSeek-V3's
    aux-loss-free bias): a bias equal for all experts keeps every token's order, so through the logits and the
    routing neither the chosen experts nor the gates may move. Under the softmax modes the same constant is a
    logit shift, which softmax ignores."""
    rng = np.random.default_rng(12)
    x, w_r = rng.standard_normal((30, 6)), rng.standard_normal((6, 8))
    for gating in (O.SIGMOID_BIAS_RENORM, O.SOFTMAX, O.SOFTMAX_RENORM):
        r0 = O.route(O.router_logits(x, w_r, np.zeros(8), gating), 3, gating, bias=np.zeros(8))
        b = np.full(8, 0.7)
        r1 = O.route(O.router_logits(x, w_r, b, gating), 3, gating, bias=b)
        assert np.array_equal(r0["ids"], r1["ids"])
        assert np.allclose(r0["gates"], r1["gates"], rtol=1e-13, atol=0), gating


def test_logit_bias_moves_softmax_selection():
    """In the softmax modes the per-expert bias is part of the logits (the Zipf load skew of the Mixtral-shaped
    workload is made that way): a bias of +50 on one expert makes it every token's first choice, with a
    softmax probability within e^-40 of 1."""
    rng = np.random.default_rng(15)
    x, w_r = rng.standard_normal((25, 6)), rng.standard_normal((6, 5)) * 0.5
    b = np.zeros(5)
    b[2] = 50.0
    for gating in (O.SOFTMAX, O.SOFTMAX_RENORM):
        r = O.route(O.router_logits(x, w_r, b, gating), 2, gating)
        assert np.all(r["ids"][:, 0] == 2)
        if gating == O.SOFTMAX:
            assert np.all(np.abs(r["gates"][:, 0] - 1.0) < math.exp(-40))


def test_softmax_gate_closed_forms():
    # two experts whose logits differ by ln 3: probabilities 3/4 and 1/4
    L = np.array([[math.log(3.0), 0.0]])
    r = O.route(L, 1, O.SOFTMAX)
    assert r["ids"][0, 0] == 0 and abs(r["gates"][0, 0] - 0.75) < 1e-15
    r2 = O.route(L, 2, O.SOFTMAX)
    assert np.allclose(r2["gates"][0], [0.75, 0.25], rtol=1e-15)
    # renormalised over the chosen: with k = E the gates are the probabilities themselves
    rr = O.route(L, 1, O.SOFTMAX_RENORM)
    assert abs(rr["gates"][0, 0] - 1.0) < 1e-15
    # equal logits -> uniform probabilities 1/E
    r3 = O.route(np.zeros((2, 5)), 2, O.SOFTMAX)
    assert np.allclose(r3["gates"], 0.2, rtol=1e-15) and np.allclose(r3["P"], 0.2)
    # shift invariance of softmax and large logits do not overflow
    r4 = O.route(np.array([[1000.0, 1000.0 - math.log(3.0)]]), 1, O.SOFTMAX)
    assert abs(r4["gates"][0, 0] - 0.75) < 1e-12


def test_counts_sum_and_f():
    rng = np.random.default_rng(1)
    for E, k in [(8, 2), (16, 4), (5, 5)]:
        L = rng.standard_normal((100, E))
        r = O.route(L, k, O.SOFTMAX)
        assert r["counts"].sum() == k * 100
        assert abs(r["f"].sum() - 1.0) < 1e-15
        assert np.allclose(r["P"].sum(), 1.0)
        brute = [sum(1 for t in range(100) for j in range(k) if r["ids"][t, j] == e) for e in range(E)]
        assert r["counts"].tolist() == brute


def test_aux_uniform_split_equals_alpha():
    """Cyclic logits: expert (t mod E) and (t+1 mod E) lead each token, so every expert receives the same
    number of assignments and the same mean probability: f = P = 1/E and aux = alpha exactly."""
    E, k, alpha = 8, 2, 0.01
    T = 4 * E
    L = np.zeros((T, E))
    for t in range(T):
        L[t, t % E] = 2.0
        L[t, (t + 1) % E] = 1.0
    r = O.route(L, k, O.SOFTMAX, alpha=alpha)
    assert np.allclose(r["f"], 1.0 / E) and np.allclose(r["P"], 1.0 / E)
    assert abs(r["aux"] - alpha) < 1e-15


def test_aux_closed_form_skewed():
    """k=1, E=2, every token prefers expert 0 with p0 = 3/4: f = (1, 0), P = (3/4, 1/4),
    aux = alpha * 2 * 3/4 = 1.5 alpha; balanced inputs give smaller aux than skewed ones."""
    alpha = 0.01
    L = np.tile([math.log(3.0), 0.0], (10, 1))
    r = O.route(L, 1, O.SOFTMAX, alpha=alpha)
    assert abs(r["aux"] - 1.5 * alpha) < 1e-15
    rng = np.random.default_rng(3)
    bal = O.route(rng.standard_normal((4000, 8)) * 0.01, 2, O.SOFTMAX, alpha=alpha)["aux"]
    sk = O.route(rng.standard_normal((4000, 8)) * 0.01 + np.arange(8)[None, :], 2, O.SOFTMAX, alpha=alpha)["aux"]
    assert abs(bal - alpha) < 2e-4 and sk > 1.5 * alpha


def test_aux_at_least_alpha_when_f_equals_P():
    """With f = P, aux = alpha E sum f^2 >= alpha (Cauchy-Schwarz), equality only at the uniform split.
    Here each token's softmax is one-hot on its single chosen expert, which makes f = P."""
    E = 4
    L = np.full((6, E), -1e6)
    hot = [0, 0, 1, 2, 2, 2]
    for t, e in enumerate(hot):
        L[t, e] = 0.0
    r = O.route(L, 1, O.SOFTMAX, alpha=1.0)
    assert np.allclose(r["f"], r["P"])
    assert r["aux"] > 1.0
    assert abs(r["aux"] - E * sum((hot.count(e) / 6.0) ** 2 for e in range(E))) < 1e-12


# ---------------------------------------------------------------------------------------------- dispatch

def _brute_dispatch(ids, E, C, R):
    """Walk assignments in token order with a running count per expert."""
    T, k = len(ids), len(ids[0])
    n = [0] * E
    slot = [[0] * k for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = int(ids[t][j])
            slot[t][j] = n[e]
            n[e] += 1
    kept = [min(c, C) if C else c for c in n]
    if C:
        off = [e * C for e in range(E + 1)]
    else:
        off = [0]
        for c in n:
            off.append(off[-1] + c)
    rows = E * C if C else T * k
    dest = [[-1] * k for _ in range(T)]
    src_t = [-1] * rows
    src_j = [-1] * rows
    for t in range(T):
        for j in range(k):
            e = int(ids[t][j])
            if C == 0 or slot[t][j] < C:
                dest[t][j] = off[e] + slot[t][j]
                src_t[dest[t][j]] = t
                src_j[dest[t][j]] = j
    epr = E // R
    rank_off = [off[r * epr] for r in range(R + 1)]
    rank_cnt = [sum(kept[r * epr:(r + 1) * epr]) for r in range(R)]
    return dict(counts=n, kept_counts=kept, offsets=off, dest_row=dest, src_token=src_t, src_slot=src_j,
                rank_offsets=rank_off, rank_counts=rank_cnt, rows=rows)


@pytest.mark.parametrize("T,E,k,C,R", [(50, 4, 2, 0, 2), (50, 4, 2, 20, 2), (64, 8, 2, 10, 4), (33, 8, 3, 0, 8),
                                       (40, 6, 6, 0, 3), (40, 6, 1, 3, 1), (1, 4, 2, 1, 2)])
def test_dispatch_brute_force(T, E, k, C, R):
    rng = np.random.default_rng(T + E + k + C)
    L = rng.standard_normal((T, E)) + np.linspace(0, 2, E)[None, :]
    ids = O.route(L, k, O.SOFTMAX)["ids"]
    d = O.dispatch(ids, E, C, R)
    b = _brute_dispatch(ids.tolist(), E, C, R)
    for key in ["counts", "kept_counts", "offsets", "src_token", "src_slot", "rank_offsets", "rank_counts"]:
        assert list(d[key]) == b[key], key
    assert d["dest_row"].tolist() == b["dest_row"]
    assert d["rows"] == b["rows"]
    assert d["drop_mask"].tolist() == [[v < 0 for v in row] for row in b["dest_row"]]


def test_dispatch_stable_and_bijective():
    rng = np.random.default_rng(11)
    ids = O.route(rng.standard_normal((500, 16)), 4, O.SOFTMAX)["ids"]
    for C in [0, 100, 40]:
        d = O.dispatch(ids, 16, C, 4)
        for e in range(16):
            o, n = d["offsets"][e], d["kept_counts"][e]
            blk = d["src_token"][o:o + n]
            assert np.all(np.diff(blk) > 0)                 # stable: token order inside each block
            assert np.all(d["src_token"][o + n:d["offsets"][e + 1]] == -1)   # pad
            assert np.all(ids[blk, d["src_slot"][o:o + n]] == e)
        kept = np.argwhere(d["dest_row"] >= 0)
        assert len(kept) == d["kept_counts"].sum()
        assert np.all(d["src_token"][d["dest_row"][kept[:, 0], kept[:, 1]]] == kept[:, 0])
        assert np.all(d["src_slot"][d["dest_row"][kept[:, 0], kept[:, 1]]] == kept[:, 1])


def test_dispatch_payload_rows_and_zero_pads():
    """Brute force over (t, j): the row dest_row[t, j] of the send buffer is x[t] for every kept pair; every
    other row (a pad) is zero ([L7] table row "dispatch": unfilled slots are padded)."""
    rng = np.random.default_rng(13)
    T, h, E, k = 30, 5, 4, 2
    x = rng.standard_normal((T, h)) + 3.0                     # no zero entries in real rows
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    for C in (0, 9, 20):
        d = O.dispatch(ids, E, C, 1)
        buf = O.dispatch_payload(x, d)
        used = set()
        for t in range(T):
            for j in range(k):
                r = int(d["dest_row"][t, j])
                if r >= 0:
                    assert np.array_equal(buf[r], x[t])
                    used.add(r)
        for r in range(buf.shape[0]):
            if r not in used:
                assert not buf[r].any()
        assert len(used) == int(d["kept_counts"].sum())


def test_capacity_drops_in_token_order():
    """Every token picks expert 0 first: with C = 3 the first three tokens keep it, the rest drop it."""
    ids = np.array([[0, 1], [0, 2], [0, 1], [0, 3], [0, 1]], np.int32)
    d = O.dispatch(ids, 4, 3, 2)
    assert d["drop_mask"][:, 0].tolist() == [False, False, False, True, True]
    assert d["drop_mask"][:, 1].tolist() == [False] * 5
    assert d["counts"].tolist() == [5, 3, 1, 1] and d["kept_counts"].tolist() == [3, 3, 1, 1]
    assert d["src_token"][0:3].tolist() == [0, 1, 2]


def test_send_layout_is_block_transpose():
    """Rank-major send buffer: the concatenation of the R rank blocks (rank r owning experts
    [r E/R, (r+1) E/R)) is the expert-major dispatch buffer itself."""
    rng = np.random.default_rng(2)
    cfg_T, E, k, R = 64, 8, 2, 4
    x = rng.standard_normal((cfg_T, 6))
    ids = O.route(rng.standard_normal((cfg_T, E)), k, O.SOFTMAX)["ids"]
    for C in [0, 12]:
        d = O.dispatch(ids, E, C, R)
        buf = O.dispatch_payload(x, d)
        blocks = [buf[d["rank_offsets"][r]:d["rank_offsets"][r + 1]] for r in range(R)]
        assert np.array_equal(np.concatenate(blocks), buf)
        for r in range(R):
            toks = [t for t in range(cfg_T) for j in range(k)
                    if ids[t, j] // (E // R) == r and d["dest_row"][t, j] >= 0]
            assert d["rank_counts"][r] == len(toks)


# ------------------------------------------------------------------------------------ experts and combine

def _scalar_swiglu(x, wg, wu, wd):
    F, h = len(wg), len(x)
    a = []
    for f in range(F):
        g = sum(x[i] * wg[f][i] for i in range(h))
        u = sum(x[i] * wu[f][i] for i in range(h))
        a.append(g / (1.0 + math.exp(-g)) * u)
    return [sum(a[f] * wd[o][f] for f in range(F)) for o in range(len(wd))]


def test_single_expert_reduces_to_dense_swiglu():
    """E = 1, k = 1, dropless: the gate is 1 and the layer is one dense SwiGLU FFN."""
    rng = np.random.default_rng(4)
    T, h, F = 5, 8, 16
    x = rng.standard_normal((T, h))
    wr = rng.standard_normal((h, 1))
    wg, wu, wd = rng.standard_normal((F, h)), rng.standard_normal((F, h)), rng.standard_normal((h, F))
    out = O.moe_layer(x, wr, None, lambda e: (wg, wu, wd), k=1, gating=O.SOFTMAX, cf=0, R=1)
    assert np.allclose(out["router"]["gates"], 1.0)
    ref = np.array([_scalar_swiglu(list(x[t]), wg.tolist(), wu.tolist(), wd.tolist()) for t in range(T)])
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_swiglu_closed_forms():
    h, F = 3, 2
    wg = np.zeros((F, h)); wu = np.ones((F, h)); wd = np.ones((h, F))
    assert np.all(O.swiglu_ffn(np.ones((1, h)), wg, wu, wd) == 0.0)     # silu(0) = 0
    wg = np.eye(F, h); wu = np.eye(F, h); wd = np.eye(h, F)
    x = np.array([[2.0, -1.0, 7.0]])
    want = [2.0 * 2.0 / (1 + math.exp(-2.0)), -1.0 * -1.0 / (1 + math.exp(1.0)), 0.0]
    assert np.allclose(O.swiglu_ffn(x, wg, wu, wd), [want], rtol=1e-15)


@pytest.mark.parametrize("gating,cf", [(O.SOFTMAX, 0), (O.SOFTMAX, 1.0), (O.SOFTMAX_RENORM, 0),
                                       (O.SIGMOID_BIAS_RENORM, 0), (O.SOFTMAX_RENORM, 0.5)])
def test_identity_experts(gating, cf):
    """Identity experts: y[t] = sum over kept j of gate[t, j] * x[t]; with renormalised gates and no
    drops, y = x."""
    rng = np.random.default_rng(7)
    T, h, E, k = 96, 12, 8, 2
    x = rng.standard_normal((T, h))
    wr = rng.standard_normal((h, E))
    b = rng.standard_normal(E) * 0.3
    out = O.moe_layer(x, wr, b, None, k=k, gating=gating, cf=cf, R=4, experts="identity")
    g = out["router"]["gates"] * (~out["dispatch"]["drop_mask"])
    assert np.allclose(out["y"], g.sum(axis=1)[:, None] * x, rtol=1e-13, atol=1e-13)
    if gating != O.SOFTMAX and cf == 0:
        assert np.allclose(out["y"], x, rtol=1e-13, atol=1e-13)
    if cf:
        assert out["dispatch"]["drop_mask"].any()


def test_token_sampled_layer_matches_full_layer():
    rng = np.random.default_rng(8)
    T, h, E, k, F = 40, 8, 4, 2, 12
    x = rng.standard_normal((T, h))
    wr = rng.standard_normal((h, E))
    W = [tuple(rng.standard_normal(s) for s in [(F, h), (F, h), (h, F)]) for _ in range(E)]
    Ws = tuple(rng.standard_normal(s) for s in [(F, h), (F, h), (h, F)])
    out = O.moe_layer(x, wr, None, lambda e: W[e], k=k, gating=O.SOFTMAX, cf=0.75, R=2, shared=lambda: Ws)
    toks = [0, 3, 17, 39]
    y = O.moe_layer_tokens(toks, x, out["router"], out["dispatch"], lambda e: W[e], shared=lambda: Ws)
    assert np.allclose(y, out["y"][toks], rtol=1e-13, atol=1e-13)
    # and against scalar loops for one token
    t = 17
    ref = np.array(_scalar_swiglu(list(x[t]), *[w.tolist() for w in Ws]))
    for j in range(k):
        if out["dispatch"]["dest_row"][t, j] >= 0:
            e = out["router"]["ids"][t, j]
            ref += out["router"]["gates"][t, j] * np.array(_scalar_swiglu(list(x[t]), *[w.tolist() for w in W[e]]))
    assert np.allclose(out["y"][t], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------ input recipe

def test_generator_deterministic_and_bf16_exact():
    cfg = moe_inputs.get_config("tiny_fp32")
    a, b = moe_inputs.make_x(cfg), moe_inputs.make_x(cfg)
    assert np.array_equal(a, b)
    cfg2 = moe_inputs.get_config("page3_cf1.25", T=64, h=256)
    xb = moe_inputs.make_x(cfg2)
    assert xb.dtype == np.uint16
    f = moe_inputs.to_f64(xb, "bf16")
    assert np.array_equal(moe_inputs.f32_to_bf16_bits(f.astype(np.float32)), xb)   # exactly representable
    assert abs(f.std() - 1.0) < 0.05
    v = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -1.0 - 2.0**-9], np.float32)  # ties to even
    assert moe_inputs.bf16_bits_to_f32(moe_inputs.f32_to_bf16_bits(v)).tolist() == [1.0, 1.0 + 2**-6, -1.0]
    red = moe_inputs.make_x(cfg2, redraw={5: 1})
    assert not np.array_equal(red[5], xb[5]) and np.array_equal(np.delete(red, 5, 0), np.delete(xb, 5, 0))


def test_zipf_bias_gives_zipf_load():
    cfg = moe_inputs.get_config("mixtral_zipf")
    x = moe_inputs.to_f64(moe_inputs.make_x(cfg), cfg.dtype)
    w_r, b = moe_inputs.make_router(cfg)
    r = O.route(O.router_logits(x, moe_inputs.to_f64(w_r, cfg.dtype), b, cfg.gating), cfg.k, cfg.gating)
    p = 1.0 / np.arange(1, 9)
    p /= p.sum()
    assert np.max(np.abs(r["counts"] / (cfg.k * cfg.T) / p - 1)) < 0.02


# -------------------------------------------------------------------------------------- expert choice

def _brute_expert_choice(col, C):
    """Max-sum C-subset of tokens; among equal sums the lexicographically smallest index set."""
    best, best_set = None, None
    for sub in itertools.combinations(range(len(col)), C):
        s = sum(col[i] for i in sub)
        if best is None or s > best:
            best, best_set = s, sub
    return list(best_set)


@pytest.mark.parametrize("T,E,C", [(7, 3, 2), (9, 4, 4), (8, 2, 8), (6, 5, 1)])
def test_expert_choice_brute_force(T, E, C):
    rng = np.random.default_rng(T * 100 + E * 10 + C)
    L = rng.standard_normal((T, E))
    ec = O.expert_choice(L, C)
    p = O.softmax(L)
    for e in range(E):
        assert ec["tokens"][e].tolist() == _brute_expert_choice(list(p[:, e]), C)
        assert np.allclose(ec["gates"][e], p[ec["tokens"][e], e], rtol=1e-15)
    assert (ec["slot"] >= 0).sum() == E * C                 # every expert takes exactly C tokens
    for t in range(T):
        for e in range(E):
            j = ec["slot"][t, e]
            assert (j < 0) == (t not in ec["tokens"][e]) and (j < 0 or ec["tokens"][e][j] == t)


def test_expert_choice_ties_take_lower_token():
    L = np.zeros((6, 2))                                   # all scores equal
    ec = O.expert_choice(L, 3)
    assert ec["tokens"].tolist() == [[0, 1, 2], [0, 1, 2]]
    assert np.allclose(ec["gates"], 0.5)


def test_expert_choice_full_capacity_is_dense():
    """C = T: every expert takes every token, the gates of a token sum to 1, and with identical experts the
    layer is one dense SwiGLU FFN."""
    rng = np.random.default_rng(12)
    T, h, E, F = 10, 6, 3, 8
    x = rng.standard_normal((T, h))
    wr = rng.standard_normal((h, E))
    W = tuple(rng.standard_normal(s) for s in [(F, h), (F, h), (h, F)])
    out = O.expert_choice_layer(x, wr, lambda e: W, C=T)
    assert np.allclose(out["ec"]["gates"].sum(axis=0), 1.0)
    ref = np.array([_scalar_swiglu(list(x[t]), *[w.tolist() for w in W]) for t in range(T)])
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_expert_choice_layer_against_scalar_loops():
    rng = np.random.default_rng(13)
    T, h, E, F, C = 12, 5, 3, 7, 4
    x = rng.standard_normal((T, h))
    wr = rng.standard_normal((h, E))
    W = [tuple(rng.standard_normal(s) for s in [(F, h), (F, h), (h, F)]) for _ in range(E)]
    out = O.expert_choice_layer(x, wr, lambda e: W[e], C=C)
    p = O.softmax(x @ wr)
    for t in range(T):
        want = np.zeros(h)
        for e in range(E):
            col = sorted(range(T), key=lambda i: (-p[i, e], i))[:C]
            if t in col:
                want += p[t, e] * np.array(_scalar_swiglu(list(x[t]), *[w.tolist() for w in W[e]]))
        assert np.allclose(out["y"][t], want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------------ sinkhorn

def test_sinkhorn_converges_to_doubly_stochastic():
    """With many iterations the scaled matrix has rows summing to 1 and columns to T/E."""
    rng = np.random.default_rng(21)
    T, E = 64, 8
    L = rng.standard_normal((T, E)) + np.linspace(0, 2, E)[None, :]
    c, r = O.sinkhorn_scaling(L, n_iter=300)
    K = np.exp(L - L.max(axis=1, keepdims=True))
    M = r[:, None] * K * c[None, :]
    assert np.allclose(M.sum(axis=1), 1.0, atol=1e-12)
    assert np.allclose(M.sum(axis=0), T / E, rtol=1e-9)


def test_sinkhorn_selection_equals_topk_of_balanced_matrix():
    """Top-k of L + log c equals the top-k of diag(r) K diag(c) itself (brute force on the matrix)."""
    rng = np.random.default_rng(22)
    T, E, k = 40, 6, 2
    L = rng.standard_normal((T, E)) * 2
    c, r = O.sinkhorn_scaling(L)
    M = r[:, None] * np.exp(L - L.max(axis=1, keepdims=True)) * c[None, :]
    out = O.route_sinkhorn(L, k)
    for t in range(T):
        assert list(out["ids"][t]) == _brute_topk(list(M[t]), k)
        assert np.allclose(out["gates"][t], O.softmax(L)[t, out["ids"][t]], rtol=1e-14)


def test_sinkhorn_closed_forms_and_balance():
    # uniform logits: K is constant, c uniform, the selection is plain top-k (ties -> lowest experts)
    out = O.route_sinkhorn(np.zeros((12, 4)), 2)
    assert out["ids"].tolist() == [[0, 1]] * 12
    # a constant per-expert logit offset is exactly undone by the column scaling
    rng = np.random.default_rng(23)
    L = rng.standard_normal((200, 8))
    shifted = O.route_sinkhorn(L + np.arange(8)[None, :] * 3.0, 1)
    plain = O.route_sinkhorn(L, 1)
    assert np.array_equal(shifted["ids"], plain["ids"])
    # and the loads are far more even than plain top-1 on the shifted logits
    raw = O.route(L + np.arange(8)[None, :] * 3.0, 1, O.SOFTMAX)
    assert raw["counts"].max() > 150 and shifted["counts"].max() < 60


# ------------------------------------------------------------------------------------------------ backward

def _bwd_problem(gating, cf, seed=0, T=7, h=5, E=4, k=2, F=3):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, h))
    w_r = rng.normal(size=(h, E))
    bias = rng.normal(size=E) * 0.3
    W = [(rng.normal(size=(F, h)), rng.normal(size=(F, h)), rng.normal(size=(h, F))) for _ in range(E)]
    Ws = (rng.normal(size=(F, h)), rng.normal(size=(F, h)), rng.normal(size=(h, F)))
    dy = rng.normal(size=(T, h))
    return x, w_r, bias, W, Ws, dy, k


@pytest.mark.parametrize("gating", [O.SOFTMAX, O.SOFTMAX_RENORM, O.SIGMOID_BIAS_RENORM])
@pytest.mark.parametrize("cf", [0.0, 0.6])
def test_backward_matches_finite_differences(gating, cf):
    """Every gradient of <dy, y> + d_aux * aux (dx, dW_r, d_bias, each expert's three matrices, the shared
    expert's) against central differences of the forward, which is pinned on its own (selection, counts and
    drops do not move under a 1e-6 step at these random inputs)."""
    x, w_r, bias, W, Ws, dy, k = _bwd_problem(gating, cf, seed=int(cf * 10) + len(gating))
    alpha, d_aux = 0.3, 0.7

    def loss(x, w_r, bias, W, Ws):
        f = O.moe_layer(x, w_r, bias, lambda e: W[e], k=k, gating=gating, cf=cf, R=1, alpha=alpha,
                        shared=lambda: Ws)
        return float(np.sum(dy * f["y"]) + d_aux * f["router"]["aux"]), f

    _, fwd = loss(x, w_r, bias, W, Ws)
    g = O.moe_layer_backward(x, w_r, bias, lambda e: W[e], fwd, dy, gating=gating, alpha=alpha, d_aux=d_aux,
                             shared=lambda: Ws)
    eps = 1e-6

    def check(got, perturb):
        num = (loss(*perturb(eps))[0] - loss(*perturb(-eps))[0]) / (2 * eps)
        assert abs(num - got) <= 1e-6 * max(1.0, abs(num)), (num, got)

    def bump(a, idx, e):
        b = a.copy()
        b[idx] += e
        return b

    for idx in [(0, 0), (3, 2), (6, 4)]:
        check(g["dx"][idx], lambda e: (bump(x, idx, e), w_r, bias, W, Ws))
    for idx in [(0, 1), (4, 3), (2, 0)]:
        check(g["dW_r"][idx], lambda e: (x, bump(w_r, idx, e), bias, W, Ws))
    if gating != O.SIGMOID_BIAS_RENORM:
        check(g["d_bias"][2], lambda e: (x, w_r, bump(bias, 2, e), W, Ws))
    else:
        assert g["d_bias"] is None
    for ex in range(len(W)):
        for m, idx in [(0, (1, 2)), (1, (2, 4)), (2, (3, 1))]:
            def pert(e, ex=ex, m=m, idx=idx):
                W2 = [list(w) for w in W]
                W2[ex][m] = bump(W2[ex][m], idx, e)
                return x, w_r, bias, [tuple(w) for w in W2], Ws
            check(g["dW"][ex][m][idx], pert)
    for m, idx in [(0, (0, 1)), (1, (2, 3)), (2, (4, 2))]:
        def pert_s(e, m=m, idx=idx):
            Ws2 = list(Ws)
            Ws2[m] = bump(Ws2[m], idx, e)
            return x, w_r, bias, W, tuple(Ws2)
        check({0: g["shared"]["dW_gate"], 1: g["shared"]["dW_up"], 2: g["shared"]["dW_down"]}[m][idx], pert_s)


def test_swiglu_backward_scalar_closed_form():
    """h = F = 1: out = wd * silu(wg x) * (wu x), so d out / dx = wd (silu'(wg x) wg (wu x) + silu(wg x) wu)
    with silu'(z) = s(z) + z s(z) (1 - s(z)), written out by hand."""
    x, wg, wu, wd = 0.7, -1.3, 0.9, 2.1
    z = wg * x
    s = 1 / (1 + math.exp(-z))
    silu_z, dsilu = z * s, s + z * s * (1 - s)
    g = O.swiglu_ffn_backward(np.array([[x]]), np.array([[wg]]), np.array([[wu]]), np.array([[wd]]),
                              np.array([[1.0]]))
    assert g["dX"][0, 0] == pytest.approx(wd * (dsilu * wg * wu * x + silu_z * wu), rel=1e-12)
    assert g["dW_gate"][0, 0] == pytest.approx(wd * dsilu * x * wu * x, rel=1e-12)
    assert g["dW_up"][0, 0] == pytest.approx(wd * silu_z * x, rel=1e-12)
    assert g["dW_down"][0, 0] == pytest.approx(silu_z * wu * x, rel=1e-12)


def test_backward_dropped_pairs_and_pad_rows_get_zero():
    """A dropped pair contributes nothing to y, so its gate gradient is 0; pad rows carry no gradient."""
    x, w_r, _, W, Ws, dy, k = _bwd_problem(O.SOFTMAX, 1.0, seed=3, T=12, E=4)
    bias = np.array([4.0, 0.0, 0.0, 0.0])            # every token picks expert 0: it overflows, the others pad
    fwd = O.moe_layer(x, w_r, bias, lambda e: W[e], k=k, gating=O.SOFTMAX, cf=1.0, R=1)
    d = fwd["dispatch"]
    assert d["drop_mask"].any()
    g = O.moe_layer_backward(x, w_r, bias, lambda e: W[e], fwd, dy, gating=O.SOFTMAX)
    assert np.all(g["d_gates"][d["drop_mask"]] == 0)
    pad = d["src_token"] < 0
    assert pad.any() and np.all(g["d_eout"][pad] == 0) and np.all(g["d_buf"][pad] == 0)


# ------------------------------------------------------------------------------------------------ fp8 payload

def test_e4m3_table_closed_form():
    """Values written out by hand from the e4m3 definition (bias 7, 3 mantissa bits, no infinities)."""
    t = O.e4m3_table()
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 / 8 * 2.0 ** -6, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0,
            0x7E: 448.0, 0x78: 256.0, 0xB8: -1.0, 0xFE: -448.0, 0x30: 0.5}
    for c, v in hand.items():
        assert t[c] == v, (hex(c), t[c], v)
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF]) and np.isfinite(t).sum() == 254
    assert np.all(np.diff(t[:0x7F]) > 0)                      # codes 0 .. 0x7e increase
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])        # sign bit mirrors


def test_e4m3_encode_brute_force_and_ties():
    """Nearest finite code by exhaustive search (ties -> even mantissa), midpoints, saturation."""
    t = O.e4m3_table()
    fin = np.array([c for c in range(256) if np.isfinite(t[c])])
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(size=2000) * 50, rng.normal(size=500) * 0.01, [0.0, 447.0, 448.0]])
    got = O.e4m3_encode(v)
    for x, c in zip(v, got):
        d = np.abs(t[fin] - x)
        best = fin[d == d.min()]
        if len(best) > 1:                                     # a tie (or +-0): prefer the even mantissa, same sign
            best = [b for b in best if (b & 1) == 0 and (np.signbit(t[b]) == np.signbit(x) or t[b] != 0)] or best
        assert c in best, (x, hex(c), [hex(b) for b in best])
    pos = np.arange(0x7F)
    mids = (t[pos[:-1]] + t[pos[1:]]) / 2                     # exact midpoints between neighbours
    m = O.e4m3_encode(mids)
    assert np.all((m & 1) == 0) and np.all((m == pos[:-1]) | (m == pos[1:]))
    assert np.all(O.e4m3_encode(np.array([449.0, 500.0, 1e30])) == 0x7E)
    assert np.all(O.e4m3_encode(np.array([-449.0, -1e30])) == 0xFE)


def test_bf16_round_against_torch_and_ties():
    """Round to nearest bfloat16, ties to even: against torch's float32 -> bfloat16 conversion on normal,
    subnormal and large values, and three ties written out by hand (1 + 2^-8 lies midway between 1 and
    1 + 2^-7, 1 + 3 * 2^-8 midway between 1 + 2^-7 and 1 + 2^-6)."""
    import torch
    rng = np.random.default_rng(14)
    v = np.concatenate([rng.standard_normal(4000), rng.standard_normal(500) * 1e-39, rng.standard_normal(500) * 1e30])
    v = v.astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(v), want)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -20], np.float32)
    assert O.bf16_round(ties).tolist() == [1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7]


def test_fp8_quantize_rows_scale_and_error_bound():
    """The block's largest magnitude maps to +-448 exactly; an all-zero block gets scale 1 and code 0; the
    dequantised value is within half an e4m3 ulp (relative 2^-4 for normals, 2^-10 s for subnormals) plus the
    bf16 rounding of x itself."""
    rng = np.random.default_rng(1)
    X = rng.normal(size=(6, 384)).astype(np.float32)
    X[2, 128:256] = 0.0
    X[3, :128] *= 1e-3
    codes, scales = O.fp8_quantize_rows(X)
    assert codes.shape == X.shape and scales.shape == (6, 3) and scales.dtype == np.float32
    t = O.e4m3_table()
    for r in range(6):
        for b in range(3):
            blk = X[r, 128 * b:128 * (b + 1)]
            if not blk.any():
                assert scales[r, b] == 1.0 and not codes[r, 128 * b:128 * (b + 1)].any()
                continue
            i = int(np.argmax(np.abs(blk)))
            assert abs(t[codes[r, 128 * b + i]]) == 448.0
            assert scales[r, b] == np.float32(np.abs(blk).max()) / np.float32(448.0)
    Xd = O.fp8_dequantize_rows(codes, scales)
    s = np.repeat(scales, 128, axis=1).astype(np.float64)
    bound = 2.0 ** -4 * np.abs(X) + 2.0 ** -10 * s + 2.0 ** -8 * np.abs(Xd)
    assert np.all(np.abs(Xd - X) <= bound)


def test_fp8_payload_rows_and_pads():
    """Every kept row of the FP8 send buffer is its token's quantisation; pad rows are code 0, scale 0."""
    rng = np.random.default_rng(2)
    T, h, E, k = 20, 256, 4, 2
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    d = O.dispatch(ids, E, 8, 1)
    x = rng.normal(size=(T, h)).astype(np.float32)
    codes, scales = O.dispatch_payload_fp8(x, d)
    ct, st = O.fp8_quantize_rows(x)
    for r in range(d["rows"]):
        t = d["src_token"][r]
        if t < 0:
            assert not codes[r].any() and not scales[r].any()
        else:
            assert np.array_equal(codes[r], ct[t]) and np.array_equal(scales[r], st[t])


def test_backward_sinkhorn_matches_finite_differences():
    """Sinkhorn routing (ids chosen on L + log c, gates softmax(L)[ids]) through the layer: the backward in the
    selection-bias mode against central differences of that forward (the Sinkhorn scalings move with L, but the
    selection does not move under a 1e-6 step, and the scalings enter only the selection)."""
    rng = np.random.default_rng(21)
    T, h, E, k, F = 9, 5, 4, 2, 3
    x = rng.normal(size=(T, h))
    w_r = rng.normal(size=(h, E))
    bias = rng.normal(size=E) * 0.3
    W = [(rng.normal(size=(F, h)), rng.normal(size=(F, h)), rng.normal(size=(h, F))) for _ in range(E)]
    dy = rng.normal(size=(T, h))
    alpha, d_aux = 0.3, 0.7

    def forward(x, w_r, bias):
        L = O.router_logits(x, w_r, bias, O.SOFTMAX)
        r = O.route_sinkhorn(L, k, alpha=alpha)
        d = O.dispatch(r["ids"], E, 0, 1)
        buf = O.dispatch_payload(x, d)
        eout = O.expert_outputs(buf, d, lambda e: W[e])
        y = O.combine(eout, d["dest_row"], r["gates"])
        return float(np.sum(dy * y) + d_aux * r["aux"]), dict(router=r, dispatch=d, buf=buf, eout=eout)

    _, fwd = forward(x, w_r, bias)
    g = O.moe_layer_backward(x, w_r, bias, lambda e: W[e], fwd, dy, gating=O.SOFTMAX_SELBIAS, alpha=alpha, d_aux=d_aux)
    eps = 1e-6

    def bump(a, idx, e):
        b = a.copy()
        b[idx] += e
        return b

    for got, pert in [(g["dx"][2, 3], lambda e: (bump(x, (2, 3), e), w_r, bias)),
                      (g["dx"][7, 0], lambda e: (bump(x, (7, 0), e), w_r, bias)),
                      (g["dW_r"][1, 2], lambda e: (x, bump(w_r, (1, 2), e), bias)),
                      (g["d_bias"][3], lambda e: (x, w_r, bump(bias, 3, e)))]:
        num = (forward(*pert(eps))[0] - forward(*pert(-eps))[0]) / (2 * eps)
        assert abs(num - got) <= 1e-6 * max(1.0, abs(num)), (num, got)
