"""The host-side dispatch checker (top_routing_dispatch_moe_gb300.checks) on the CPU: it accepts the oracle's
dispatch in dropless and capacity mode, and it names each planted corruption of the index outputs or the
payload."""
import numpy as np
import pytest

from oracle import moe_oracle as O


def _case(C, R=2, seed=0):
    rng = np.random.default_rng(seed)
    T, E, k, h = 60, 8, 2, 4
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[:20, 0] = 3                                   # an over-loaded expert, so capacity mode drops
    ids[:20, 1] = np.where(ids[:20, 1] == 3, 4, ids[:20, 1])
    x = rng.standard_normal((T, h)) + 5.0
    d = O.dispatch(ids, E, C, R)
    d = {key: np.array(v) for key, v in d.items()}
    d["buf"] = O.dispatch_payload(x, d)
    return ids, x, d, E, C, R


@pytest.mark.parametrize("C", [0, 12])
def test_accepts_the_oracle_dispatch(C):
    from top_routing_dispatch_moe_gb300.checks import check_dispatch
    ids, x, d, E, C, R = _case(C)
    if C:
        assert d["drop_mask"].any()
    assert check_dispatch(d, ids, E, C, R, x=x) == []


def _first_two_kept_of(d, ids, e):
    tt, jj = np.nonzero((ids == e) & (d["dest_row"] >= 0))
    return (tt[0], jj[0]), (tt[1], jj[1])


@pytest.mark.parametrize("C", [0, 12])
def test_names_each_corruption(C):
    from top_routing_dispatch_moe_gb300.checks import check_dispatch
    ids, x, d0, E, C, R = _case(C)

    def run(mutate):
        d = {key: v.copy() for key, v in d0.items()}
        mutate(d)
        return " | ".join(check_dispatch(d, ids, E, C, R, x=x))

    def swap_order(d):                                # two rows of one expert exchanged: unstable order
        (t0, j0), (t1, j1) = _first_two_kept_of(d, ids, 3)
        r0, r1 = d["dest_row"][t0, j0], d["dest_row"][t1, j1]
        d["dest_row"][t0, j0], d["dest_row"][t1, j1] = r1, r0
        d["src_token"][r0], d["src_token"][r1] = t1, t0
        d["src_slot"][r0], d["src_slot"][r1] = j1, j0
        d["buf"][[r0, r1]] = d["buf"][[r1, r0]]
    assert "token order" in run(swap_order)

    def stale_inverse(d):
        r = d["dest_row"][5, 0]
        d["src_token"][r] = 6
    assert "inverse" in run(stale_inverse)

    def wrong_offsets(d):
        d["offsets"][1] += 1
    assert "offsets" in run(wrong_offsets)

    def wrong_rank_counts(d):
        d["rank_counts"][0] -= 1
    assert "rank_counts" in run(wrong_rank_counts)

    def wrong_payload(d):
        d["buf"][d["dest_row"][7, 1]] += 1.0
    assert "token's row" in run(wrong_payload)

    def mask_mismatch(d):
        d["drop_mask"][9, 0] = 1 - d["drop_mask"][9, 0]
    assert "drop_mask" in run(mask_mismatch)

    if C:
        def dirty_pad(d):
            pad = np.nonzero(d["src_token"] < 0)[0][0]
            d["buf"][pad, 0] = 1.0
        assert "pad row" in run(dirty_pad)

        def drop_the_wrong_pair(d):                   # keep expert 3's first dropped pair, drop its first kept one
            (t0, j0), _ = _first_two_kept_of(d, ids, 3)
            tt, jj = np.nonzero((ids == 3) & (d["dest_row"] < 0))
            t1, j1 = tt[0], jj[0]
            r = d["dest_row"][t0, j0]
            d["dest_row"][t0, j0], d["drop_mask"][t0, j0] = -1, 1
            d["dest_row"][t1, j1], d["drop_mask"][t1, j1] = r, 0
            d["src_token"][r], d["src_slot"][r] = t1, j1
            d["buf"][r] = x[t1]
        assert "latest assignments" in run(drop_the_wrong_pair)


def test_out_of_range_ids_are_reported():
    from top_routing_dispatch_moe_gb300.checks import check_dispatch
    ids, x, d, E, C, R = _case(0)
    ids = ids.copy()
    ids[0, 0] = E
    assert check_dispatch(d, ids, E, C, R) == ["topk_ids outside [0, E)"]


def _router_case(gating, seed=3):
    rng = np.random.default_rng(seed)
    T, E, k = 50, 8, 3
    L = rng.standard_normal((T, E))
    b = rng.standard_normal(E) * 0.3 if gating in (O.SIGMOID_BIAS_RENORM, "softmax_selbias") else None
    if gating == "softmax_selbias":
        r = O.route_selbias(L, k, b)
    else:
        r = O.route(L, k, gating, b)
    out = dict(ids=r["ids"].astype(np.int32), gates=r["gates"].astype(np.float32),
               counts=r["counts"].astype(np.int32), f=r["f"].astype(np.float32), P=r["P"].astype(np.float32),
               aux=np.array([r["aux"]], np.float32))
    return out, L.astype(np.float32), b, E


@pytest.mark.parametrize("gating", [O.SOFTMAX, O.SOFTMAX_RENORM, O.SIGMOID_BIAS_RENORM, "softmax_selbias"])
def test_router_checker_accepts_the_oracle_and_names_corruptions(gating):
    from top_routing_dispatch_moe_gb300.checks import check_router
    r0, L, b, E = _router_case(gating)
    assert check_router(r0, E, gating, logits=L, bias=b) == []

    def run(mutate):
        r = {key: v.copy() for key, v in r0.items()}
        mutate(r)
        return " | ".join(check_router(r, E, gating, logits=L, bias=b))

    def dup(r):
        r["ids"][0, 1] = r["ids"][0, 0]
    assert "twice" in run(dup)

    def swap(r):
        r["ids"][1, [0, 1]] = r["ids"][1, [1, 0]]
    assert "descending" in run(swap)

    def unchosen(r):                                  # replace a choice by the token's lowest-scoring expert
        sc = L[2] if gating in (O.SOFTMAX, O.SOFTMAX_RENORM) else None
        if sc is None:
            sc = (1 / (1 + np.exp(-L[2])) + b) if gating == O.SIGMOID_BIAS_RENORM else L[2] + b
        r["ids"][2, -1] = int(np.argmin(sc))
    assert "unchosen" in run(unchosen)

    def counts_off(r):
        r["counts"][0] += 1
    assert "histogram" in run(counts_off)

    def aux_off(r):
        r["aux"][0] *= 1.5
    assert "aux" in run(aux_off)

    def gate_zero(r):
        r["gates"][3, 0] = 0.0
    assert "gate" in run(gate_zero)
