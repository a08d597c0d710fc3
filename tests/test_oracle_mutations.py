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
