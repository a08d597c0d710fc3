"""Host-side checks of moe_router's and moe_dispatch's outputs: a debugging aid standing in for a device race
detector.

Every index output of a dispatch is checked against the invariants that define it (the v6 MoE page, table
row "dispatch" and the "Capacity" bullet: group by expert in token order, at most C rows per expert, the
rest dropped, unfilled slots padded; the formulaic expert-parallel page, section "All2All": expert blocks in
rank order). The check needs only the outputs and the router's ids, not a second implementation of the
dispatch. It copies the outputs to the host, so it synchronises; call it from tests or while debugging, never
on a timed path.
"""
from __future__ import annotations

import numpy as np

KEYS = ("offsets", "kept_counts", "dest_row", "drop_mask", "src_token", "src_slot", "rank_counts", "rank_offsets")


def _host(a):
    if hasattr(a, "detach"):                          # a torch tensor: bf16 has no numpy type, compare its bits
        import torch
        a = a.detach().cpu()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        a = a.numpy()
    return np.asarray(a)


def check_dispatch(d: dict, topk_ids, E: int, capacity: int, num_ranks: int = 1, x=None) -> list[str]:
    """Violations of the dispatch invariants by the outputs `d` (the dict moe_dispatch returns, or host arrays
    under the same names) for the router's ids [T, k]; an empty list when every invariant holds.

    Checked: ids in [0, E); offsets (e*C in capacity mode, the exclusive prefix of the kept counts when
    dropless) and the row count; kept counts min(n_e, C) (n_e when dropless); dest_row of each kept pair inside
    its expert's kept block, -1 exactly on the dropped pairs, drop_mask its mirror; src_token / src_slot the
    inverse of dest_row, -1 on every other row; token order inside every expert block (stability); drops only
    past the first C assignments of an expert, in token order; the rank layout (rank r owns experts
    [r E/R, (r+1) E/R)). With `x` (tokens [T, h]) and d["buf"], also every kept row equal to its token's row and
    every pad row zero."""
    ids = _host(topk_ids).astype(np.int64)
    T, k = ids.shape
    o = {key: _host(d[key]).astype(np.int64) for key in KEYS}
    bad: list[str] = []
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        bad.append("topk_ids outside [0, E)")
        return bad
    if num_ranks < 1 or E % num_ranks:
        return [f"num_ranks {num_ranks} does not divide E={E}"]
    rows = E * capacity if capacity > 0 else T * k
    counts = np.bincount(ids.ravel(), minlength=E)
    kept = np.minimum(counts, capacity) if capacity > 0 else counts
    offsets = np.arange(E + 1) * capacity if capacity > 0 else np.concatenate([[0], np.cumsum(kept)])
    if o["src_token"].shape != (rows,) or o["src_slot"].shape != (rows,):
        bad.append(f"src_token / src_slot must have {rows} rows")
        return bad
    if not np.array_equal(o["kept_counts"], kept):
        bad.append("kept_counts differ from min(assignments per expert, C)")
    if not np.array_equal(o["offsets"], offsets):
        bad.append("offsets are not the expert blocks' first rows")
    dest, drop = o["dest_row"].reshape(T, k), o["drop_mask"].reshape(T, k)
    if not np.array_equal(drop != 0, dest < 0):
        bad.append("drop_mask does not mirror dest_row < 0")
    lo, hi = offsets[ids], offsets[ids] + kept[ids]
    live = dest >= 0
    if np.any(live & ((dest < lo) | (dest >= hi))):
        bad.append("a kept pair's row lies outside its expert's kept block")
        return bad
    src_t, src_j = o["src_token"], o["src_slot"]
    tt, jj = np.nonzero(live)
    rr = dest[tt, jj]
    if len(np.unique(rr)) != len(rr):
        bad.append("two kept pairs share a row")
    if not (np.array_equal(src_t[rr], tt) and np.array_equal(src_j[rr], jj)):
        bad.append("src_token / src_slot are not the inverse of dest_row")
    other = np.ones(rows, bool)
    other[rr] = False
    if np.any(src_t[other] != -1) or np.any(src_j[other] != -1):
        bad.append("a row no pair uses has src_token / src_slot != -1")
    if int(live.sum()) != int(kept.sum()):
        bad.append("kept pairs differ from the sum of kept counts")
    for e in range(E):
        blk = src_t[offsets[e]:offsets[e] + kept[e]]
        if np.any(np.diff(blk) <= 0):
            bad.append(f"expert {e}: block not in token order")
            break
    # drops: for every expert, the kept pairs are its first min(n_e, C) assignments in token order
    flat_e, flat_live = ids.ravel(), live.ravel()
    order = np.argsort(flat_e, kind="stable")
    starts = np.concatenate([[0], np.cumsum(counts)])
    slot = np.empty(T * k, np.int64)
    slot[order] = np.arange(T * k) - starts[flat_e[order]]
    want_live = slot < kept[flat_e]
    if not np.array_equal(flat_live, want_live):
        bad.append("dropped pairs are not the latest assignments of over-capacity experts")
    epr = E // num_ranks
    if not np.array_equal(o["rank_offsets"], offsets[::epr]):
        bad.append("rank_offsets are not the first rows of the rank blocks")
    if not np.array_equal(o["rank_counts"], kept.reshape(num_ranks, epr).sum(axis=1)):
        bad.append("rank_counts are not the kept rows of each rank")
    if x is not None and "buf" in d:
        xb, buf = _host(x), _host(d["buf"])
        if not np.array_equal(buf[rr], xb[tt]):
            bad.append("a kept row differs from its token's row")
        if capacity > 0 and np.any(buf[other] != 0):
            bad.append("a pad row is not zero")
    return bad


GATINGS = ("softmax", "softmax_renorm", "sigmoid_bias_renorm", "softmax_selbias")


def check_router(r: dict, E: int, gating: str, alpha: float = 0.01, logits=None, bias=None,
                 tol: float = 1e-5) -> list[str]:
    """Violations of the router's output invariants by `r` (the dict moe_router returns: ids, gates, counts,
    f, P, aux); an empty list when every invariant holds. ("Megatron-LM ... (6)", section "Router": top-k with
    softmax or sigmoid weights; the v6 MoE page, "Load balancing loss": aux = alpha E sum f_i P_i.)

    Checked: ids in [0, E) and distinct within a token; gates positive, at most 1, summing to 1 over the k
    choices in the renormalised modes; counts the histogram of ids, f = counts / (k T); P a distribution over
    the experts; aux = alpha E sum f P. With the fp32 `logits` [T, E] (and the selection bias of the sigmoid
    and selection-bias modes), also: every chosen expert's selection score at least every unchosen one's, the
    k choices in descending score order (up to `tol`, so near ties pass either way)."""
    if gating not in GATINGS:
        return [f"unknown gating {gating!r}"]
    ids = _host(r["ids"]).astype(np.int64)
    gates = _host(r["gates"]).astype(np.float64)
    T, k = ids.shape
    bad: list[str] = []
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        return ["ids outside [0, E)"]
    if T and np.any(np.sort(ids, axis=1)[:, 1:] == np.sort(ids, axis=1)[:, :-1]):
        bad.append("a token chose one expert twice")
    if np.any(gates <= 0) or np.any(gates > 1 + tol):
        bad.append("a gate outside (0, 1]")
    if gating in ("softmax_renorm", "sigmoid_bias_renorm") and T:
        if np.max(np.abs(gates.sum(axis=1) - 1.0)) > tol * k:
            bad.append("renormalised gates do not sum to 1")
    counts = _host(r["counts"]).astype(np.int64)
    if not np.array_equal(counts, np.bincount(ids.ravel(), minlength=E)):
        bad.append("counts are not the histogram of ids")
    f, P = _host(r["f"]).astype(np.float64), _host(r["P"]).astype(np.float64)
    if T and np.max(np.abs(f - counts / float(k * T))) > tol:
        bad.append("f differs from counts / (k T)")
    if T and (np.any(P < 0) or abs(P.sum() - 1.0) > tol * E):
        bad.append("P is not a distribution over the experts")
    aux = float(_host(r["aux"]).reshape(-1)[0])
    if T and abs(aux - alpha * E * float(np.sum(f * P))) > tol * max(1.0, abs(aux)):
        bad.append("aux differs from alpha E sum f P")
    if logits is not None and T:
        L = _host(logits).astype(np.float64)
        b = np.zeros(E) if bias is None else _host(bias).astype(np.float64)
        if gating == "sigmoid_bias_renorm":
            score = 1.0 / (1.0 + np.exp(-L)) + b[None, :]
        elif gating == "softmax_selbias":
            score = L + b[None, :]
        else:
            score = L                                  # the logits already hold a softmax-mode bias
        chosen = np.take_along_axis(score, ids, axis=1)
        if k > 1 and np.any(chosen[:, 1:] > chosen[:, :-1] + tol):
            bad.append("the k choices are not in descending score order")
        mask = np.ones((T, E), bool)
        np.put_along_axis(mask, ids, False, axis=1)
        if E > k:
            best_other = np.where(mask, score, -np.inf).max(axis=1)
            if np.any(best_other > chosen.min(axis=1) + tol):
                bad.append("an unchosen expert scores above a chosen one")
    return bad
