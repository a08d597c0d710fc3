"""Host-side checks of moe_dispatch's outputs: a debugging aid standing in for a device race detector.

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
        a = a.detach().cpu()
        if str(a.dtype) == "torch.bfloat16":
            a = a.view(dtype=__import__("torch").int16)
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
