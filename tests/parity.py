"""Comparison rules between the GPU path and the oracle (test helpers).

Acceptance per query row:
  * the number of selected positions equals min(k, visible keys); unused
    slots are -1 / -inf; selected positions are distinct and visible;
  * the GPU's list is ordered by (score desc, position asc) on its own scores;
  * sets: a position selected by one side only is allowed when its oracle
    score, and the oracle score of the position it displaced, both lie within
    swap_tol * max|s| of the oracle's k-th score (max|s| over the row's
    visible keys);
  * logits: max |gpu score - oracle score at the same position| divided by
    max |oracle top-k score| is at most logit_tol (2e-3 bf16, 3e-2 fp8 and
    fp4: the fp4 keys are widened to e4m3 exactly, so their scores carry the
    same query-side rounding as fp8 keys).
"""
from __future__ import annotations

import dataclasses

import numpy as np

SWAP_TOL = 1e-3
LOGIT_TOL = {0: 2e-3, 1: 3e-2, 2: 3e-2}


@dataclasses.dataclass
class RowReport:
    row: int
    ok: bool
    swaps: int
    logit_err: float
    why: str = ""


def compare_row(row, g_idx, g_sc, o_idx, o_sc, s_full, k, logit_tol, swap_tol=SWAP_TOL):
    n = s_full.shape[0]
    want_n = min(k, n)
    gi = np.asarray(g_idx, dtype=np.int64)
    gs = np.asarray(g_sc, dtype=np.float64)
    valid = gi >= 0
    nv = int(valid.sum())
    if nv != want_n or not np.all(valid[:nv]) or np.any(valid[nv:]):
        return RowReport(row, False, 0, np.inf, f"count {nv} vs {want_n} or holes")
    if np.any(~np.isneginf(gs[nv:])):
        return RowReport(row, False, 0, np.inf, "padding scores not -inf")
    sel = gi[:nv]
    if len(np.unique(sel)) != nv or sel.min(initial=0) < 0 or sel.max(initial=-1) >= n:
        return RowReport(row, False, 0, np.inf, "duplicate or invisible positions")
    s = gs[:nv]
    if nv > 1:
        bad = (s[1:] > s[:-1]) | ((s[1:] == s[:-1]) & (sel[1:] < sel[:-1]))
        if np.any(bad):
            return RowReport(row, False, 0, np.inf, "not sorted by (score desc, pos asc)")
    if nv == 0:
        return RowReport(row, True, 0, 0.0)
    oset = set(np.asarray(o_idx[:nv], dtype=np.int64).tolist())
    gset = set(sel.tolist())
    only_g = gset - oset
    only_o = oset - gset
    M = float(np.abs(s_full).max())
    kth = float(s_full[o_idx[nv - 1]])
    tol = swap_tol * M
    for j in list(only_g) + list(only_o):
        if abs(float(s_full[j]) - kth) > tol:
            return RowReport(row, False, len(only_g), np.inf,
                             f"swap of pos {j}: |s-kth|={abs(float(s_full[j]) - kth):.3g} > {tol:.3g}")
    denom = float(np.abs(s_full[np.asarray(o_idx[:nv], dtype=np.int64)]).max())
    err = float(np.abs(s - s_full[sel]).max()) / max(denom, 1e-30)
    ok = err <= logit_tol
    return RowReport(row, ok, len(only_g), err, "" if ok else f"logit err {err:.3g}")


def compare(rows, g_idx, g_sc, o_idx, o_sc, full, k, fmt, swap_tol=SWAP_TOL):
    """Compare GPU results (indexed like rows) with the oracle's. Returns
    (all_ok, reports)."""
    reps = []
    for t, r in enumerate(rows):
        reps.append(compare_row(int(r), g_idx[t], g_sc[t], o_idx[t], o_sc[t], full[int(r)], k,
                                LOGIT_TOL[fmt], swap_tol))
    return all(r.ok for r in reps), reps


def summary(reps):
    bad = [r for r in reps if not r.ok]
    return {"rows": len(reps), "failed": len(bad),
            "swaps": int(sum(r.swaps for r in reps)),
            "max_logit_err": float(max((r.logit_err for r in reps), default=0.0)),
            "first_failure": None if not bad else f"row {bad[0].row}: {bad[0].why}"}
