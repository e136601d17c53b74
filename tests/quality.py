"""Selection-fidelity statistics of "Locks: Page-Local Compact Key Summaries
for Efficient Long-Context Decoding" on the synthetic workloads (test
infrastructure; uses the oracle).

Table B.1 (App. B) measures a page selection S against exact-mass selection
(the same forced pages plus the top-(k-2) candidates by the share-average of the
exact per-head page masses s_j = log sum_i exp(q^T k_i / sqrt d)):

* gamma    -- attention mass of S, averaged over the group's query heads;
* gamma_c  -- contested mass: the always-kept (forced) pages' mass taken out
              of numerator and denominator;
* recall   -- |S_cand  intersect  S*_cand| / |S*_cand| against the exact
              selection S*;
* needle   -- planted carrier pages kept, conditional on S* keeping them.

Rival selectors for comparison (scored here from the keys, like the exact
ceiling; they are not part of the product path): "centroid-only" scores a page
as if every token were its centroid, log nv + q.mu/sqrt(d), a lower bound of
the exact log-mass by Jensen's inequality; "Quest" scores it by the elementwise
key envelope of Lemma 2, log nv + sum_d max(q_d min_d, q_d max_d)/sqrt(d), an
upper bound of every logit and so of the log-mass.  Both then go through the
same shares, share-average and forced-page top-(k-2) as Locks.

Table D.17 (App. D) compares GQA combine rules on the exact per-head shares:
share-average (the shipped rule, Cor. 3), group-max, group-mass, and a
per-head oracle (each head its own selection); per head the coverage is the
head's contested mass captured, reported as mean, worst head and 5th
percentile over heads.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np

import oracle as O


def _logsumexp(x: np.ndarray, axis: int) -> np.ndarray:
    m = np.max(x, axis=axis, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    return np.squeeze(m, axis=axis) + np.log(np.sum(np.exp(x - m), axis=axis))


def unit_exact(inputs, b: int, h: int) -> Dict:
    """Exact per-head log masses of every page of unit (b, h) and the exact
    share-average selection."""
    w = inputs.workload
    B, G = w.page_size, w.group
    t = int(inputs.seq_lens[b])
    n = -(-t // B)
    q = O.bf16_to_f64(inputs.q[b, h * G:(h + 1) * G])
    s = np.full((G, n), -np.inf)
    for j in range(n):
        nv = O.valid_tokens(t, B, j)
        if nv > 0:
            s[:, j] = O.exact_log_mass(q, O.page_keys(inputs.k_cache, inputs.block_table, b, h, j, nv))
    forced, cand = O.forced_and_candidates(t, B)
    k = O.page_budget(w.budget_tokens, B)
    mbar = O.share_average(O.page_shares(s[:, cand]))
    best = O.select_from_shares(mbar, cand, forced, n, k)
    return {"s": s, "forced": forced, "cand": cand, "k": k, "n": n, "best": best,
            "carriers": np.asarray(inputs.carriers[b][h], dtype=np.int64)}


def rival_log_mass(inputs, b: int, h: int, rule: str) -> np.ndarray:
    """Per-head page scores [G][n] of a rival selector on the log-mass scale
    (-inf for pages without valid tokens): rule "centroid" or "quest"."""
    w = inputs.workload
    B, G, d = w.page_size, w.group, w.head_dim
    t = int(inputs.seq_lens[b])
    n = -(-t // B)
    q = O.bf16_to_f64(inputs.q[b, h * G:(h + 1) * G])          # [G][d]
    s = np.full((G, n), -np.inf)
    for j in range(n):
        nv = O.valid_tokens(t, B, j)
        if nv <= 0:
            continue
        k = O.page_keys(inputs.k_cache, inputs.block_table, b, h, j, nv)   # [nv][d]
        if rule == "centroid":
            s[:, j] = np.log(nv) + (q @ k.mean(axis=0)) / np.sqrt(d)
        elif rule == "quest":
            lo, hi = k.min(axis=0), k.max(axis=0)
            s[:, j] = np.log(nv) + np.maximum(q * lo, q * hi).sum(axis=1) / np.sqrt(d)
        else:
            raise ValueError(rule)
    return s


def rival_selection(ex: Dict, s_rival: np.ndarray):
    """The forced pages plus the top-(k-2) candidates by the share-average of a
    rival selector's per-head scores."""
    cand = ex["cand"]
    mbar = O.share_average(O.page_shares(s_rival[:, cand]))
    return O.select_from_shares(mbar, cand, ex["forced"], ex["n"], ex["k"])


def _mass(s: np.ndarray, pages) -> np.ndarray:
    """Per-head share of the total attention mass held by the given pages."""
    logz = _logsumexp(s, axis=1)
    idx = np.asarray(sorted(set(int(p) for p in pages if 0 <= p < s.shape[1])), dtype=np.int64)
    if idx.size == 0:
        return np.zeros(s.shape[0])
    return np.exp(_logsumexp(s[:, idx], axis=1) - logz)


def contested_coverage(ex: Dict, pages) -> np.ndarray:
    """Per head: (mass(S) - mass(forced)) / (1 - mass(forced))."""
    m = _mass(ex["s"], pages)
    mf = _mass(ex["s"], ex["forced"])
    return (m - mf) / np.maximum(1.0 - mf, 1e-300)


def unit_stats(ex: Dict, pages) -> Dict:
    sel = set(int(p) for p in pages if p >= 0)
    cand = set(int(c) for c in ex["cand"])
    best = set(int(p) for p in ex["best"]) & cand
    got = sel & cand
    car_best = [c for c in ex["carriers"] if int(c) in best]
    return {
        "gamma": float(np.mean(_mass(ex["s"], sel))),
        "gamma_c": float(np.mean(contested_coverage(ex, sel))),
        "recall": len(got & best) / len(best) if best else 1.0,
        "needle": (sum(int(c) in sel for c in car_best) / len(car_best)) if car_best else None,
    }


def aggregate(rows: Sequence[Dict]) -> Dict:
    out = {}
    for key in ("gamma", "gamma_c", "recall"):
        out[key] = float(np.mean([r[key] for r in rows]))
    needles = [r["needle"] for r in rows if r["needle"] is not None]
    out["needle"] = float(np.mean(needles)) if needles else None
    return out


# ---- Table D.17: combine rules on exact per-head shares ---------------------
def combine_selection(ex: Dict, rule: str) -> List:
    """One shared selection per unit under a combine rule, or (per-head
    oracle) one selection per head."""
    s, cand, forced, n, k = ex["s"], ex["cand"], ex["forced"], ex["n"], ex["k"]
    shares = O.page_shares(s[:, cand])
    if rule == "share-average":
        return [O.select_from_shares(O.share_average(shares), cand, forced, n, k)]
    if rule == "group-max":
        return [O.select_from_shares(shares.max(axis=0), cand, forced, n, k)]
    if rule == "group-mass":
        # the group's summed raw page mass (heads weighted by their own logit scale)
        return [O.select_from_shares(_logsumexp(s[:, cand], axis=0), cand, forced, n, k)]
    if rule == "per-head":
        return [O.select_from_shares(shares[g], cand, forced, n, k) for g in range(s.shape[0])]
    raise ValueError(rule)


def combine_coverage(ex: Dict, rule: str) -> np.ndarray:
    """Per-head contested coverage under the rule's selection(s)."""
    sels = combine_selection(ex, rule)
    if len(sels) == 1:
        return contested_coverage(ex, sels[0])
    return np.array([contested_coverage(ex, sels[g])[g] for g in range(len(sels))])
