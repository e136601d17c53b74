"""Plain fp64 CPU oracle of the Locks decode hot path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
bench's CPU-baseline / reference arm may import this module.  The product path
(the CUDA library and its Python binding) never calls it, and it shares no code
with that path: it reads the same seeded input arrays and nothing else.

Everything is NumPy in float64 on inputs widened exactly from bf16.  Each step
follows a passage of "Locks: Page-Local Compact Key Summaries for Efficient
Long-Context Decoding" (arXiv 2607.24555), cited by section / equation:

* decode attention and the page budget      -- section 2 (o = sum_i alpha_i v_i,
  alpha = softmax(q^T k / sqrt d); k = ceil(b / B); sink and most recent page
  counted inside k)
* page summary build                         -- section 4 "Build" (centre the
  page, eigendecompose the B x B Gram D D^T, keep r modes, V = D^T U_r S_r^-1,
  C = U_r S_r, zero modes dropped with zero coefficients, tail tau)
* reconstructed page score                   -- section 4, Eq. (1)
* page-mass share and GQA share-average      -- section 4 (m_hat_g(j), m_bar_j)
* selection                                  -- section 4 and Cor. 3 (sink and
  most recent page forced, top-(k-2) of the rest by m_bar)
* exact page log-mass                        -- Lemma 1 (App. A.1)

Readings where the pages leave a step open (each also listed in the design
notes):
  R1  the forced pair is {page 0, page n-1}; page n-1 is the tail, complete or
      not; both count inside k.
  R2  shares are normalised over the candidate set (complete pages other than
      the forced pair) -- the only pages that have summaries to score.
  R3  ties in m_bar: the smaller logical page index wins; outputs are sorted.
  R4  n <= k selects every page; fewer than k-2 candidates selects them all;
      k < 2 is invalid.
  R5  a mode is "zero" when sigma^2 <= 1e-12 * sigma_1^2 (or <= 0).
  R6  scale 1/sqrt(d); one query per (sequence, query head); the cache holds
      every token including the current one.
  R7  a sequence of length 0 attends nothing: output 0, lse -inf.
  R8  quantised summary (the deployed form: int4 basis, int8 coefficients and
      centroid, "per-column and per-row scales"): one scale per basis column,
      one for the centroid, one per coefficient row; symmetric absmax scales,
      scale = absmax / qmax (qmax 7 for int4, 127 for int8), code =
      round-half-even(x / scale) clamped to [-qmax, qmax], all in float32 --
      the quantiser's own precision, so an integer code is decided in the same
      precision on both sides; an all-zero group has scale 0 and codes 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np

ZERO_MODE_REL = 1e-12


# --------------------------------------------------------------------------
# bf16 widening (exact)
# --------------------------------------------------------------------------
def bf16_to_f64(x: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly to float64."""
    u = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Build: one page summary (section 4 "Build")
# --------------------------------------------------------------------------
@dataclass
class PageSummary:
    mu: np.ndarray        # (d,)      page centroid
    V: np.ndarray         # (d, r)    orthonormal basis, zero columns for dropped modes
    C: np.ndarray         # (B, r)    per-token coefficients c_i = V^T delta_i
    sigma2: np.ndarray    # (B,)      Gram eigenvalues sigma_k^2, descending
    tau: float            # spectral tail sum_{k>r} sigma_k^2
    kept: int             # number of non-zero modes among the first r


def page_summary(keys: np.ndarray, r: int) -> PageSummary:
    """Rank-r spectral summary of one complete page of keys (B x d)."""
    K = np.asarray(keys, dtype=np.float64)
    Bt, d = K.shape
    mu = K.mean(axis=0)                         # k_i = mu + delta_i, sum delta_i = 0
    D = K - mu                                  # deviations as rows, B x d
    gram = D @ D.T                              # B x B Gram  D D^T = U S^2 U^T
    w, U = np.linalg.eigh(gram)                 # ascending
    order = np.argsort(-w, kind="stable")       # descending sigma^2
    w = w[order]
    U = U[:, order]
    top = w[0] if Bt else 0.0
    V = np.zeros((d, r))
    C = np.zeros((Bt, r))
    kept = 0
    for k in range(min(r, Bt)):
        s2 = w[k]
        if s2 <= 0.0 or s2 <= ZERO_MODE_REL * top:
            continue                            # zero mode: dropped, coefficients 0
        s = math.sqrt(s2)
        V[:, k] = D.T @ U[:, k] / s             # V = D^T U_r S_r^{-1}
        C[:, k] = U[:, k] * s                   # C = U_r S_r
        kept += 1
    tail = np.clip(w[r:], 0.0, None).sum() if Bt > r else 0.0
    return PageSummary(mu=mu, V=V, C=C, sigma2=w, tau=float(tail), kept=kept)


# --------------------------------------------------------------------------
# Quantised summary (section 4 "Build": int4 basis, int8 coefficients and
# centroid, per-column and per-row scales; reading R8)
# --------------------------------------------------------------------------
INT4_QMAX = 7
INT8_QMAX = 127


def quantize_symmetric(x, qmax: int) -> Tuple[np.ndarray, np.float32]:
    """Codes and scale of one group: scale = absmax / qmax, code = x / scale
    rounded half to even, clamped to [-qmax, qmax]; float32 throughout."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    if amax == 0.0:
        return np.zeros(x.shape, dtype=np.int32), np.float32(0.0)
    scale = np.float32(amax / np.float32(qmax))
    codes = np.rint(x / scale)
    return np.clip(codes, -qmax, qmax).astype(np.int32), scale


def dequantize(codes, scale) -> np.ndarray:
    return np.asarray(codes, dtype=np.float64) * float(scale)


@dataclass
class QuantizedSummary:
    mu_codes: np.ndarray      # (d,)   int8 codes of the centroid
    mu_scale: np.float32
    v_codes: np.ndarray       # (d, r) int4 codes, one scale per column
    v_scales: np.ndarray      # (r,)
    c_codes: np.ndarray       # (B, r) int8 codes, one scale per row (token)
    c_scales: np.ndarray      # (B,)


def quantize_summary(mu, V, C) -> QuantizedSummary:
    """The deployed record of one page summary (mu, V, C given in the values
    the quantiser reads; float32 rounding is part of the quantiser)."""
    V = np.asarray(V)
    C = np.asarray(C)
    mu_codes, mu_scale = quantize_symmetric(mu, INT8_QMAX)
    r = V.shape[1]
    v_codes = np.zeros(V.shape, dtype=np.int32)
    v_scales = np.zeros(r, dtype=np.float32)
    for k in range(r):                               # per column
        v_codes[:, k], v_scales[k] = quantize_symmetric(V[:, k], INT4_QMAX)
    c_codes = np.zeros(C.shape, dtype=np.int32)
    c_scales = np.zeros(C.shape[0], dtype=np.float32)
    for i in range(C.shape[0]):                      # per row
        c_codes[i], c_scales[i] = quantize_symmetric(C[i], INT8_QMAX)
    return QuantizedSummary(mu_codes, mu_scale, v_codes, v_scales, c_codes, c_scales)


def dequantized_summary(qs: QuantizedSummary) -> PageSummary:
    """The page summary a quantised record stands for (what the scorer reads)."""
    mu = dequantize(qs.mu_codes, qs.mu_scale)
    V = qs.v_codes.astype(np.float64) * qs.v_scales.astype(np.float64)[None, :]
    C = qs.c_codes.astype(np.float64) * qs.c_scales.astype(np.float64)[:, None]
    sig = (C ** 2).sum(axis=0)
    return PageSummary(mu=mu, V=V, C=C, sigma2=sig, tau=0.0, kept=int((sig > 0).sum()))


# --------------------------------------------------------------------------
# Score: Eq. (1), brute-force log-sum-exp over the B reconstructed logits
# --------------------------------------------------------------------------
def _lse(x: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(x, axis=axis, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    return np.squeeze(m, axis=axis) + np.log(np.sum(np.exp(x - m), axis=axis))


def reconstructed_logits(q: np.ndarray, s: PageSummary) -> np.ndarray:
    """(q^T mu + (V^T q)^T c_i) / sqrt(d) for every token i; q is (G, d)."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    d = q.shape[1]
    a = q @ s.mu                                 # (G,)
    p = q @ s.V                                  # (G, r) = (V^T q)^T
    return (a[:, None] + p @ s.C.T) / math.sqrt(d)   # (G, B)


def reconstructed_score(q: np.ndarray, s: PageSummary) -> np.ndarray:
    """s_hat_j(q) of Eq. (1) for each query row of q."""
    return _lse(reconstructed_logits(q, s), axis=-1)


def exact_log_mass(q: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """s_j(q) = log sum_i exp(q^T k_i / sqrt d) over the page's true keys (Lemma 1)."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    K = np.asarray(keys, dtype=np.float64)
    return _lse(q @ K.T / math.sqrt(q.shape[1]), axis=-1)


# --------------------------------------------------------------------------
# Shares and selection (section 4; Cor. 3)
# --------------------------------------------------------------------------
def page_shares(scores: np.ndarray) -> np.ndarray:
    """m_hat_g(j) = exp(s_g,j) / sum_j' exp(s_g,j'); scores is (G, n_cand)."""
    scores = np.atleast_2d(scores)
    if scores.shape[1] == 0:
        return scores.copy()
    logz = _lse(scores, axis=1)
    return np.exp(scores - logz[:, None])


def share_average(shares: np.ndarray) -> np.ndarray:
    """m_bar_j = (1/G) sum_g m_hat_g(j)."""
    return np.mean(np.atleast_2d(shares), axis=0)


def page_budget(budget_tokens: int, page_size: int) -> int:
    return -(-budget_tokens // page_size)        # k = ceil(b / B)


def forced_and_candidates(seq_len: int, page_size: int) -> Tuple[List[int], np.ndarray]:
    """Forced pages {0, n-1} and candidates (complete pages other than those)."""
    n = -(-seq_len // page_size)
    if n <= 0:
        return [], np.zeros(0, dtype=np.int64)
    forced = sorted({0, n - 1})
    n_complete = seq_len // page_size
    hi = min(n - 1, n_complete)
    cand = np.arange(1, hi, dtype=np.int64) if hi > 1 else np.zeros(0, dtype=np.int64)
    return forced, cand


def select_from_shares(mbar: np.ndarray, cand: np.ndarray, forced: List[int], n: int,
                       k: int) -> np.ndarray:
    """Forced pages plus the top-(k-2) candidates by m_bar (ties -> lower index)."""
    if k < 2:
        raise ValueError("page budget k must be at least 2")
    if n <= k:
        return np.arange(n, dtype=np.int64)
    order = sorted(range(len(cand)), key=lambda i: (-mbar[i], cand[i]))   # full sort
    chosen = [int(cand[i]) for i in order[:k - 2]]
    return np.array(sorted(set(forced) | set(chosen)), dtype=np.int64)


# --------------------------------------------------------------------------
# Attention (section 2): dense and restricted to a page set
# --------------------------------------------------------------------------
def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """softmax(q K^T / sqrt d) V for each query row; returns (o, lse).

    An empty token set gives o = 0 and lse = -inf (reading R7)."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    K = np.asarray(keys, dtype=np.float64)
    Vv = np.asarray(values, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], Vv.shape[-1])), np.full(q.shape[0], -np.inf)
    logits = q @ K.T / math.sqrt(q.shape[1])
    lse = _lse(logits, axis=1)
    alpha = np.exp(logits - lse[:, None])
    return alpha @ Vv, lse


# --------------------------------------------------------------------------
# Whole-cache drivers over the paged layout
# --------------------------------------------------------------------------
def page_keys(k_cache: np.ndarray, block_table: np.ndarray, b: int, h: int, j: int,
              n_valid: int) -> np.ndarray:
    blk = int(block_table[b, j])
    return bf16_to_f64(k_cache[blk, h, :n_valid])


def page_values(v_cache: np.ndarray, block_table: np.ndarray, b: int, h: int, j: int,
                n_valid: int) -> np.ndarray:
    blk = int(block_table[b, j])
    return bf16_to_f64(v_cache[blk, h, :n_valid])


def valid_tokens(seq_len: int, page_size: int, j: int) -> int:
    return max(0, min(page_size, seq_len - j * page_size))


def build_unit(k_cache, block_table, seq_len: int, b: int, h: int, r: int,
               pages: Optional[np.ndarray] = None) -> Dict[int, PageSummary]:
    """Summaries of the complete pages of one (sequence, KV head)."""
    B = k_cache.shape[2]
    n_complete = seq_len // B
    if pages is None:
        pages = np.arange(n_complete)
    return {int(j): page_summary(page_keys(k_cache, block_table, b, h, int(j), B), r)
            for j in pages if int(j) < n_complete}


@dataclass
class UnitSelection:
    selected: np.ndarray       # ascending logical page ids
    cand: np.ndarray           # candidate logical page ids
    scores: np.ndarray         # (G, n_cand) reconstructed scores s_hat
    shares: np.ndarray         # (G, n_cand) m_hat
    mbar: np.ndarray           # (n_cand,)
    forced: List[int]


def select_unit(q_group: np.ndarray, summaries: Dict[int, PageSummary], seq_len: int,
                page_size: int, k: int) -> UnitSelection:
    """Score, normalise, share-average and select for one (sequence, KV head)."""
    q_group = np.atleast_2d(q_group)
    n = -(-seq_len // page_size)
    forced, cand = forced_and_candidates(seq_len, page_size)
    G = q_group.shape[0]
    scores = np.zeros((G, len(cand)))
    for c, j in enumerate(cand):
        scores[:, c] = reconstructed_score(q_group, summaries[int(j)])
    shares = page_shares(scores) if len(cand) else scores
    mbar = share_average(shares) if len(cand) else np.zeros(0)
    if n <= 0:
        sel = np.zeros(0, dtype=np.int64)
    else:
        sel = select_from_shares(mbar, cand, forced, n, k)
    return UnitSelection(selected=sel, cand=cand, scores=scores, shares=shares, mbar=mbar,
                         forced=forced)


def attend_pages(q_group: np.ndarray, k_cache, v_cache, block_table, seq_len: int, b: int,
                 h: int, pages) -> Tuple[np.ndarray, np.ndarray]:
    """Attention of the group's queries restricted to the given logical pages."""
    B = k_cache.shape[2]
    Ks, Vs = [], []
    for j in pages:
        nv = valid_tokens(seq_len, B, int(j))
        if nv <= 0:
            continue
        Ks.append(page_keys(k_cache, block_table, b, h, int(j), nv))
        Vs.append(page_values(v_cache, block_table, b, h, int(j), nv))
    d = k_cache.shape[3]
    K = np.concatenate(Ks) if Ks else np.zeros((0, d))
    Vv = np.concatenate(Vs) if Vs else np.zeros((0, d))
    return attend(q_group, K, Vv)


def dense_unit(q_group, k_cache, v_cache, block_table, seq_len, b, h):
    B = k_cache.shape[2]
    n = -(-seq_len // B)
    return attend_pages(q_group, k_cache, v_cache, block_table, seq_len, b, h, range(n))


# --------------------------------------------------------------------------
# One decode step over chosen (sequence, KV head) units
# --------------------------------------------------------------------------
@dataclass
class UnitResult:
    b: int
    h: int
    summaries: Dict[int, PageSummary]
    sel: UnitSelection
    o_sparse: np.ndarray       # (G, d) attention over sel.selected
    lse_sparse: np.ndarray     # (G,)
    o_dense: Optional[np.ndarray] = None
    lse_dense: Optional[np.ndarray] = None


def run_unit(q_bits, k_cache, v_cache, block_table, seq_lens, n_kv_heads: int, r: int,
             budget_tokens: int, b: int, h: int, dense: bool = False,
             summaries: Optional[Dict[int, PageSummary]] = None) -> UnitResult:
    """Build, select and attend for one (sequence b, KV head h)."""
    B = k_cache.shape[2]
    Hq = q_bits.shape[1]
    G = Hq // n_kv_heads
    q = bf16_to_f64(q_bits[b, h * G:(h + 1) * G])
    t = int(seq_lens[b])
    if summaries is None:
        summaries = build_unit(k_cache, block_table, t, b, h, r)
    k = page_budget(budget_tokens, B)
    sel = select_unit(q, summaries, t, B, k)
    o, lse = attend_pages(q, k_cache, v_cache, block_table, t, b, h, sel.selected)
    res = UnitResult(b=b, h=h, summaries=summaries, sel=sel, o_sparse=o, lse_sparse=lse)
    if dense:
        res.o_dense, res.lse_dense = dense_unit(q, k_cache, v_cache, block_table, t, b, h)
    return res
