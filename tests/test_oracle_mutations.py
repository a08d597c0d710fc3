"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each one.

Each mutant replaces one oracle function for the duration of a test; the pin tests of
test_oracle_pins.py are then run against the mutant and at least one must fail."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from tests import test_oracle_pins as P

_route, _dispatch, _swiglu, _combine, _capacity = O.route, O.dispatch, O.swiglu_ffn, O.combine, O.capacity
_ec = O.expert_choice
_sk = O.sinkhorn_scaling
_cbwd, _swbwd, _rbwd = O.combine_backward, O.swiglu_ffn_backward, O.route_backward
_enc, _q8, _dq8 = O.e4m3_encode, O.fp8_quantize_rows, O.fp8_dequantize_rows
_logits, _payload, _eout, _selb, _ecl = O.router_logits, O.dispatch_payload, O.expert_outputs, O.route_selbias, \
    O.expert_choice_layer


def mut_renormalise_softmax(L, k, gating, bias=None, alpha=0.01):
    g = O.SOFTMAX_RENORM if gating == O.SOFTMAX else gating
    return _route(L, k, g, bias, alpha)


def mut_ascending_order(L, k, gating, bias=None, alpha=0.01):
    r = _route(L, k, gating, bias, alpha)
    r["ids"] = r["ids"][:, ::-1].copy()
    r["gates"] = r["gates"][:, ::-1].copy()
    return r


def mut_bias_in_sigmoid_gates(L, k, gating, bias=None, alpha=0.01):
    r = _route(L, k, gating, bias, alpha)
    if gating == O.SIGMOID_BIAS_RENORM and bias is not None:
        sc = np.take_along_axis(r["score"], r["ids"].astype(np.int64), axis=1)
        r["gates"] = sc / sc.sum(axis=1, keepdims=True)
    return r


def mut_aux_denominator_T(L, k, gating, bias=None, alpha=0.01):
    r = _route(L, k, gating, bias, alpha)
    r["aux"] *= k              # f_e = n_e / T instead of n_e / (k T)
    return r


def mut_drop_latest_first(ids, E, C, R):
    """Keeps the LAST C assignments of each expert instead of the first C."""
    d = _dispatch(ids[::-1].copy(), E, C, R)
    T = ids.shape[0]
    out = _dispatch(ids, E, C, R)
    keep_rev = ~d["drop_mask"][::-1]
    if C:
        out["drop_mask"] = ~keep_rev
    return out


def mut_dispatch_unstable(ids, E, C, R):
    d = _dispatch(ids, E, C, R)
    for e in range(E):
        o, n = d["offsets"][e], d["kept_counts"][e]
        if n > 1:
            d["src_token"][o:o + n] = d["src_token"][o:o + n][::-1].copy()
    return d


def mut_swap_gate_up(X, w_gate, w_up, w_down):
    return _swiglu(X, w_up, w_gate, w_down)


def mut_transpose_down(X, w_gate, w_up, w_down):
    """Reads the [h, F] down matrix with the wrong layout ([F, h] row-major)."""
    X = np.asarray(X, np.float64)
    a = O.silu(X @ w_gate.T) * (X @ w_up.T)
    return a @ w_down.reshape(w_down.shape[1], w_down.shape[0])


def mut_combine_no_gate(eout, dest_row, gates, shared_out=None):
    return _combine(eout, dest_row, np.ones_like(gates), shared_out)


def mut_capacity_floor_over_E(cf, k, T, E):
    return 0 if cf <= 0 else int(cf * T / E)      # forgot the k


def mut_ec_select_on_logits(L, C):
    """Selects each expert's tokens on the raw logits instead of the per-token softmax probability."""
    out = _ec(L, C)
    E = L.shape[1]
    for e in range(E):
        chosen = np.sort(np.argsort(-L[:, e], kind="stable")[:C])
        out["tokens"][e] = chosen
        out["gates"][e] = out["prob"][chosen, e]
    return out


def mut_ec_ties_higher_token(L, C):
    out = _ec(L[::-1].copy(), C)
    T = L.shape[0]
    out["tokens"] = np.sort(T - 1 - out["tokens"], axis=1)
    out["prob"] = out["prob"][::-1]
    out["gates"] = np.take_along_axis(out["prob"].T, out["tokens"], axis=1)
    return out


def mut_sinkhorn_columns_only(L, n_iter=O.SINKHORN_ITERS):
    """Normalises the columns once and never rescales the rows."""
    T, E = L.shape
    K = np.exp(L - L.max(axis=1, keepdims=True))
    c = (T / E) / K.sum(axis=0)
    return c, np.ones(T)


def mut_sinkhorn_rows_first(L, n_iter=O.SINKHORN_ITERS):
    """Swaps the targets: columns to 1, rows to T / E."""
    T, E = L.shape
    K = np.exp(L - L.max(axis=1, keepdims=True))
    r = np.ones(T)
    for _ in range(n_iter):
        c = 1.0 / (K * r[:, None]).sum(axis=0)
        r = (T / E) / (K * c[None, :]).sum(axis=1)
    return c, r


def mut_silu_prime_plain_sigmoid(X, w_gate, w_up, w_down, d_out):
    """Takes silu'(z) = s(z), dropping the z s (1 - s) term."""
    g = _swbwd(X, w_gate, w_up, w_down, d_out)
    X = np.asarray(X, np.float64)
    G, U = X @ w_gate.T, X @ w_up.T
    s = O.sigmoid(G)
    dG = g["d_a"] * U * s
    g["dX"] = dG @ w_gate + g["dU"] @ w_up
    g["dW_gate"] = dG.T @ X
    return g


def mut_route_backward_no_aux(L, r, d_gates, gating, alpha, d_aux):
    return _rbwd(L, r, d_gates, gating, alpha, 0.0)


def mut_route_backward_renorm_as_plain(L, r, d_gates, gating, alpha, d_aux):
    return _rbwd(L, r, d_gates, O.SOFTMAX if gating == O.SOFTMAX_RENORM else gating, alpha, d_aux)


def mut_combine_backward_no_gate(dy, eout, dest_row, gates, rows):
    return _cbwd(dy, eout, dest_row, np.ones_like(gates), rows)


def mut_e4m3_ties_away(v):
    """Rounds ties away from zero instead of to the even mantissa."""
    v = np.asarray(v, np.float64)
    code = _enc(v)
    t = O.e4m3_table()
    a = np.abs(v)
    c = code & 0x7F
    up = np.minimum(c + 1, 0x7E)
    tie = (np.abs(t[up] - a) == np.abs(a - t[c])) & (t[up] > t[c])
    return np.where(tie, up | (code & 0x80), code).astype(np.uint8)


def mut_fp8_scale_240(X):
    """Takes the scale for a largest value of 240 (another fp8 variant's)."""
    codes, scales = _q8(X)
    X = np.asarray(X, np.float32)
    n, h = X.shape
    amax = np.abs(X.reshape(n, h // 128, 128)).max(axis=2)
    sc = np.where(amax > 0, amax / np.float32(240.0), np.float32(1.0)).astype(np.float32)
    q = (X.reshape(n, h // 128, 128) / sc[:, :, None]).astype(np.float32)
    return _enc(q).reshape(n, h), sc


def mut_fp8_dequant_no_scale(codes, scales):
    return _dq8(codes, np.ones_like(scales))


def mut_logits_bias_in_sigmoid(x, w_r, bias, gating):
    # the selection-only bias of sigmoid gating also added to the logits
    L = np.asarray(x, np.float64) @ np.asarray(w_r, np.float64)
    return L + np.asarray(bias, np.float64)[None, :] if bias is not None else L


def mut_logits_no_bias(x, w_r, bias, gating):
    # the logit bias of the softmax modes dropped
    return np.asarray(x, np.float64) @ np.asarray(w_r, np.float64)


def mut_softmax_over_tokens(L):
    z = np.exp(L - L.max(axis=0, keepdims=True))
    return z / z.sum(axis=0, keepdims=True)


def mut_sigmoid_sign(L):
    return 1.0 / (1.0 + np.exp(L))


def mut_silu_sign(z):
    return z / (1.0 + np.exp(z))


def mut_payload_pads_first_token(x, d):
    buf = _payload(x, d)
    buf[d["src_token"] < 0] = x[0]
    return buf


def mut_payload_next_token(x, d):
    buf = np.zeros((d["rows"], x.shape[1]), dtype=x.dtype)
    live = d["src_token"] >= 0
    buf[live] = x[(d["src_token"][live] + 1) % x.shape[0]]
    return buf


def mut_eout_next_expert(buf, d, weights):
    E = len(d["kept_counts"])
    return _eout(buf, d, lambda e: weights((e + 1) % E))


def mut_combine_drops_shared(eout, dest_row, gates, shared_out=None):
    return _combine(eout, dest_row, gates, None)


def mut_ffn_flops_two_matrices(rows, h, F):
    return 4 * h * F * rows


def mut_dispatch_bytes_writes_only(T, kept, h, el):
    return kept * h * el


def mut_selbias_gates_renormalised(L, k, sel_bias, alpha=0.01):
    r = _selb(L, k, sel_bias, alpha)
    r["gates"] = r["gates"] / r["gates"].sum(axis=1, keepdims=True)
    return r


def mut_ec_layer_gate_one(x, w_r, weights, C, shared=None):
    # expert-choice outputs summed with weight 1 instead of the expert's gate for the token
    out = _ecl(x, w_r, weights, C, shared)
    ec, eout = out["ec"], out["eout"]
    y = np.zeros_like(out["y"]) if shared is None else O.swiglu_ffn(np.asarray(x, np.float64), *shared())
    for e in range(ec["tokens"].shape[0]):
        y[ec["tokens"][e]] += eout[e * C:(e + 1) * C]
    return dict(out, y=y)


def mut_bf16_truncate(v):
    b = np.asarray(v, np.float32).view(np.uint32) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def mut_e4m3_bias_8(code):
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -7
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 8)


def mut_dispatch_rank_offsets_first(ids, E, C, R):
    d = _dispatch(ids, E, C, R)
    d["rank_offsets"] = d["offsets"][:R + 1].copy()
    return d


MUTANTS = [
    ("route", mut_renormalise_softmax), ("route", mut_ascending_order), ("route", mut_bias_in_sigmoid_gates),
    ("route", mut_aux_denominator_T), ("dispatch", mut_drop_latest_first), ("dispatch", mut_dispatch_unstable),
    ("swiglu_ffn", mut_swap_gate_up), ("swiglu_ffn", mut_transpose_down), ("combine", mut_combine_no_gate),
    ("capacity", mut_capacity_floor_over_E), ("expert_choice", mut_ec_select_on_logits),
    ("expert_choice", mut_ec_ties_higher_token), ("sinkhorn_scaling", mut_sinkhorn_columns_only),
    ("sinkhorn_scaling", mut_sinkhorn_rows_first), ("swiglu_ffn_backward", mut_silu_prime_plain_sigmoid),
    ("route_backward", mut_route_backward_no_aux), ("route_backward", mut_route_backward_renorm_as_plain),
    ("combine_backward", mut_combine_backward_no_gate), ("e4m3_encode", mut_e4m3_ties_away),
    ("fp8_quantize_rows", mut_fp8_scale_240), ("fp8_dequantize_rows", mut_fp8_dequant_no_scale),
    ("router_logits", mut_logits_bias_in_sigmoid), ("router_logits", mut_logits_no_bias),
    ("softmax", mut_softmax_over_tokens), ("sigmoid", mut_sigmoid_sign), ("silu", mut_silu_sign),
    ("dispatch_payload", mut_payload_pads_first_token), ("dispatch_payload", mut_payload_next_token),
    ("expert_outputs", mut_eout_next_expert), ("combine", mut_combine_drops_shared),
    ("ffn_flops", mut_ffn_flops_two_matrices), ("dispatch_bytes", mut_dispatch_bytes_writes_only),
    ("route_selbias", mut_selbias_gates_renormalised), ("bf16_round", mut_bf16_truncate),
    ("e4m3_value", mut_e4m3_bias_8), ("dispatch", mut_dispatch_rank_offsets_first),
    ("expert_choice_layer", mut_ec_layer_gate_one),
]

PINS = [
    P.test_page3_capacity_and_shapes, P.test_capacity_rounding, P.test_softmax_gate_closed_forms,
    P.test_topk_exact_ties_take_lower_index, P.test_sigmoid_selection_uses_bias_but_gates_do_not,
    P.test_aux_uniform_split_equals_alpha, P.test_aux_closed_form_skewed, P.test_capacity_drops_in_token_order,
    P.test_dispatch_stable_and_bijective, P.test_single_expert_reduces_to_dense_swiglu, P.test_swiglu_closed_forms,
    lambda: P.test_topk_brute_force(8, 2), lambda: P.test_dispatch_brute_force(64, 8, 2, 10, 4),
    lambda: P.test_identity_experts(O.SOFTMAX, 0), lambda: P.test_identity_experts(O.SOFTMAX_RENORM, 0),
    P.test_token_sampled_layer_matches_full_layer, lambda: P.test_expert_choice_brute_force(9, 4, 4),
    P.test_expert_choice_ties_take_lower_token, P.test_expert_choice_full_capacity_is_dense,
    P.test_sinkhorn_converges_to_doubly_stochastic, P.test_sinkhorn_closed_forms_and_balance,
    lambda: P.test_backward_matches_finite_differences(O.SOFTMAX, 0.0),
    lambda: P.test_backward_matches_finite_differences(O.SOFTMAX_RENORM, 0.6),
    lambda: P.test_backward_matches_finite_differences(O.SIGMOID_BIAS_RENORM, 0.0),
    P.test_swiglu_backward_scalar_closed_form, P.test_backward_dropped_pairs_and_pad_rows_get_zero,
    P.test_e4m3_table_closed_form, P.test_e4m3_encode_brute_force_and_ties,
    P.test_fp8_quantize_rows_scale_and_error_bound, P.test_fp8_payload_rows_and_pads,
    P.test_sigmoid_constant_bias_changes_nothing, P.test_dispatch_payload_rows_and_zero_pads,
    P.test_bf16_round_against_torch_and_ties, P.test_page3_flops_and_dispatch_bytes, P.test_logit_bias_moves_softmax_selection,
    P.test_sinkhorn_selection_equals_topk_of_balanced_matrix, P.test_send_layout_is_block_transpose,
    P.test_expert_choice_layer_against_scalar_loops,
]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_pins_catch_mutant(name, fn, monkeypatch):
    monkeypatch.setattr(O, name, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(getattr(pin, "__name__", "lambda"))
    assert caught, f"no pin caught mutant {fn.__name__}"
