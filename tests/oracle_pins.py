"""Checks that pin the oracle to facts other than itself.

Each ``pin_*`` takes an oracle module ``O`` and raises AssertionError when the
oracle disagrees with something the pages or the mathematics fix:

* numbers printed in the pages (the worked toy example of the blog review,
  section 5.1; the isotropic-null statistic of the Locks paper, App. D;
  Table D.12's captured energy 1.0000 at r = 15, B = 16);
* closed forms (2 x 2 eigenpairs, the r = 0 score, uniform and two-token
  softmax attention, k = ceil(b / B));
* an independent library route (singular values of D by SVD instead of the
  eigendecomposition of D D^T);
* the inequalities the paper proves (Prop. 2, Lemma 3, the group-share
  sandwich, Cor. 2 / Thm. 1(ii) retention, Lemma 1's exact identity);
* brute force over every candidate subset (Cor. 3).

They are plain functions so that ``test_oracle_mutants`` can run them against
copies of the oracle with a planted mistake and show that each mistake trips
at least one of them.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _low_rank_page(rng, B, d, rank, noise=0.0, offset=None):
    A = rng.standard_normal((B, rank))
    G = rng.standard_normal((rank, d))
    K = A @ G / math.sqrt(rank) + noise * rng.standard_normal((B, d))
    if offset is not None:
        K = K + offset
    return K


# ---------------------------------------------------------------- build
def pin_worked_example(O):
    """Blog review, section 5.1: B=4, d=4, r=1 toy deviations."""
    fx = _golden("p2_worked_example.json")
    delta = np.array(fx["deviations"], dtype=np.float64)
    mu0 = np.array([0.3, -0.2, 0.5, 1.0])
    s = O.page_summary(mu0 + delta, fx["rank"])
    # closed form: the deviations span the first two axes with 2x2 scatter
    # [[3.62, 0.18], [0.18, 0.02]] (sums of squares / cross products by hand)
    a, b, c = 3.62, 0.18, 0.02
    tr, det = a + c, a * c - b * b
    lam_hi = (tr + math.sqrt(tr * tr - 4 * det)) / 2
    lam_lo = (tr - math.sqrt(tr * tr - 4 * det)) / 2
    assert abs(lam_hi - 3.628978) < 1e-6 and abs(lam_lo - 0.011022) < 1e-6
    assert np.allclose(s.mu, mu0, atol=1e-12), "centroid"
    assert np.allclose(s.sigma2[:2], [lam_hi, lam_lo], atol=1e-12), s.sigma2
    assert np.allclose(s.sigma2[2:], 0.0, atol=1e-12)
    assert abs(s.tau - lam_lo) < 1e-12, "spectral tail tau_{j,1}"
    v_hi = np.array([lam_hi - c, b, 0.0, 0.0])
    v_hi /= np.linalg.norm(v_hi)
    assert abs(abs(float(s.V[:, 0] @ v_hi)) - 1.0) < 1e-12, "dominant direction"
    assert np.allclose(s.C[:, 0], delta @ s.V[:, 0], atol=1e-12), "c_i = V^T delta_i"
    # the page's dominant axis is close to (1, 0, 0, 0), as the example says
    assert abs(s.V[0, 0]) > 0.99
    # a query along the discarded second axis sees nearly flat reconstructed
    # logits although its true logits differ
    q = np.array([[0.0, 40.0, 0.0, 0.0]])
    rec = O.reconstructed_logits(q, s)[0]
    true = (q @ (mu0 + delta).T / 2.0)[0]
    assert np.ptp(rec) < 0.5 * np.ptp(true)


def pin_isotropic_null(O):
    """Locks App. D: rank 8 captures a median 67.8% of isotropic B=16, d=128 pages."""
    fx = _golden("isotropic_null.json")
    rng = _rng(20240)
    B, d, r, N = fx["page_size"], fx["head_dim"], fx["rank"], fx["n_pages"]
    cap = np.empty(N)
    for i in range(N):
        s = O.page_summary(rng.standard_normal((B, d)), r)
        tot = np.clip(s.sigma2, 0, None).sum()
        cap[i] = np.clip(s.sigma2[:r], 0, None).sum() / tot
    med, mean, std = np.median(cap), cap.mean(), cap.std()
    assert abs(med - fx["median"]) < 0.003, med
    assert abs(mean - fx["mean"]) < 0.003, mean
    assert abs(std - fx["std"]) < 0.002, std


def pin_exact_rank(O):
    """Section 4 / Prop. 2: rank(D) <= r gives exact reconstruction and s_hat = s."""
    rng = _rng(7)
    B, d, r = 64, 128, 8
    K = _low_rank_page(rng, B, d, 5, offset=rng.standard_normal(d))
    s = O.page_summary(K, r)
    D = K - K.mean(axis=0)
    scale = np.abs(D).max()
    assert s.kept == 5, s.kept
    assert np.abs(s.C @ s.V.T - D).max() < 1e-9 * scale
    assert s.tau < 1e-9 * (D * D).sum()
    q = rng.standard_normal((4, d)) * 2.0
    assert np.abs(O.reconstructed_score(q, s) - O.exact_log_mass(q, K)).max() < 1e-9


def pin_full_rank_r15(O):
    """Table D.12: per-page rank 15 at B=16 captures energy 1.0000 (B-1 modes)."""
    rng = _rng(11)
    K = rng.standard_normal((16, 128))
    s = O.page_summary(K, 15)
    D = K - K.mean(axis=0)
    assert np.abs(s.C @ s.V.T - D).max() < 1e-9
    cap = np.clip(s.sigma2[:15], 0, None).sum() / np.clip(s.sigma2, 0, None).sum()
    assert abs(cap - 1.0) < 1e-12
    assert s.sigma2[15] < 1e-9 * s.sigma2[0]         # centring leaves at most B-1 modes


def pin_svd_route(O):
    """Eigenvalues of D D^T are the squared singular values of D (SVD route),
    V is orthonormal, C = D V, and tau is the Eckart-Young residual (Cor. 1)."""
    rng = _rng(3)
    B, d, r = 64, 128, 8
    K = _low_rank_page(rng, B, d, 8, noise=0.05) + _low_rank_page(rng, B, d, 16) * 0.5
    s = O.page_summary(K, r)
    D = K - K.mean(axis=0)
    sv = np.linalg.svd(D, compute_uv=False)
    assert np.allclose(s.sigma2[:B], sv ** 2, rtol=1e-9, atol=1e-9 * sv[0] ** 2)
    assert np.all(np.diff(s.sigma2) <= 1e-12 * s.sigma2[0])
    assert np.allclose(s.V.T @ s.V, np.eye(r), atol=1e-10)
    assert np.allclose(s.C, D @ s.V, atol=1e-10)
    resid = D - D @ s.V @ s.V.T
    assert abs((resid * resid).sum() - s.tau) < 1e-9 * (D * D).sum()
    assert abs((sv[r:] ** 2).sum() - s.tau) < 1e-9 * (D * D).sum()


# ---------------------------------------------------------------- score
def pin_centroid_closed_form(O):
    """r = 0: Eq. (1) reduces to q^T mu / sqrt(d) + log B."""
    rng = _rng(5)
    B, d = 64, 128
    K = rng.standard_normal((B, d))
    q = rng.standard_normal((3, d))
    s = O.page_summary(K, 0)
    want = q @ K.mean(axis=0) / math.sqrt(d) + math.log(B)
    assert np.allclose(O.reconstructed_score(q, s), want, atol=1e-12)


def pin_prop2(O):
    """Prop. 2: |s_hat - s| <= max_i |q_perp^T delta_perp_i| / sqrt d <= |q_perp| sqrt(tau) / sqrt d."""
    rng = _rng(9)
    B, d, r = 64, 128, 8
    for t in range(20):
        K = _low_rank_page(rng, B, d, 8, noise=0.2) + 0.5 * _low_rank_page(rng, B, d, 16)
        s = O.page_summary(K, r)
        D = K - K.mean(axis=0)
        Dp = D - s.C @ s.V.T
        q = rng.standard_normal((4, d)) * (1 + t % 3)
        err = np.abs(O.reconstructed_score(q, s) - O.exact_log_mass(q, K))
        qp = q - (q @ s.V) @ s.V.T
        b1 = np.abs(qp @ Dp.T).max(axis=1) / math.sqrt(d)
        b2 = np.linalg.norm(qp, axis=1) * math.sqrt(s.tau) / math.sqrt(d)
        assert np.all(err <= b1 + 1e-10), (err, b1)
        assert np.all(b1 <= b2 + 1e-10)
        assert err.max() > 0


def pin_lemma3(O):
    """Lemma 3 (outlier capture) on pages with one dominant key."""
    rng = _rng(13)
    B, d, r = 64, 128, 8
    for _ in range(10):
        K = _low_rank_page(rng, B, d, 12, noise=0.1)
        K[rng.integers(B)] += 3.0 * rng.standard_normal(d)
        s = O.page_summary(K, r)
        D = K - K.mean(axis=0)
        q = rng.standard_normal(d)
        proj = (s.V.T @ q) ** 2
        lhs = (s.sigma2[:r] * proj).sum()
        for i in range(B):
            assert lhs >= (q @ D[i]) ** 2 - s.sigma2[r] * (q @ q) - 1e-9 * (q @ q) * s.sigma2[0]
            E = D.T @ D - np.outer(D[i], D[i])
            lam = np.sort(np.linalg.eigvalsh(E))[::-1]
            assert s.sigma2[r] <= lam[r - 1] + 1e-9 * s.sigma2[0]


# ---------------------------------------------------------------- shares / selection
def _unit_pages(rng, n, B, d, rank, noise, carriers=()):
    pages = []
    for j in range(n):
        K = _low_rank_page(rng, B, d, rank, noise=noise)
        if j in carriers:
            K = K + 1.5
        pages.append(K)
    return pages


def pin_shares_and_sandwich(O):
    """m_hat sums to 1 per head, m_bar sums to 1, and |log m_bar_hat - log m_bar| <= 2 eta."""
    rng = _rng(17)
    B, d, r, G, n = 64, 128, 8, 4, 40
    pages = _unit_pages(rng, n, B, d, 12, 0.1)
    q = rng.standard_normal((G, d)) * 1.5
    S = [O.page_summary(K, r) for K in pages]
    sh = np.stack([O.reconstructed_score(q, s) for s in S], axis=1)
    se = np.stack([O.exact_log_mass(q, K) for K in pages], axis=1)
    mh, me = O.page_shares(sh), O.page_shares(se)
    assert np.allclose(mh.sum(axis=1), 1.0, atol=1e-12)
    mbh, mbe = O.share_average(mh), O.share_average(me)
    assert abs(mbh.sum() - 1.0) < 1e-12
    eta = np.abs(sh - se).max()
    assert eta > 0
    with np.errstate(divide="ignore"):     # a broken oracle may give a zero share
        assert np.all(np.abs(np.log(mbh) - np.log(mbe)) <= 2 * eta + 1e-12)
    # a head's share is its own exp-normalisation: a shift of one head's
    # scores changes nothing
    assert np.allclose(O.page_shares(sh + np.array([[3.0], [0], [0], [-2.0]])), mh, atol=1e-12)


def pin_budget_rule(O):
    """Section 2: k = ceil(b / B)."""
    assert O.page_budget(2048, 64) == 32
    assert O.page_budget(512, 64) == 8
    assert O.page_budget(256, 64) == 4
    assert O.page_budget(100, 64) == 2
    assert O.page_budget(2048, 16) == 128


def pin_forced_pages(O):
    """Sink page and the most recent page are always kept, inside k (section 2)."""
    f, c = O.forced_and_candidates(10 * 64, 64)
    assert f == [0, 9] and list(c) == list(range(1, 9))
    f, c = O.forced_and_candidates(10 * 64 + 5, 64)          # partial tail page 10
    assert f == [0, 10] and list(c) == list(range(1, 10))
    f, c = O.forced_and_candidates(64, 64)
    assert f == [0] and len(c) == 0
    f, c = O.forced_and_candidates(0, 64)
    assert f == [] and len(c) == 0
    mbar = np.linspace(0.2, 0.05, 8)
    sel = O.select_from_shares(mbar, np.arange(1, 9), [0, 9], 10, 5)
    assert list(sel) == [0, 1, 2, 3, 9]
    assert list(O.select_from_shares(mbar[:2], np.arange(1, 3), [0, 3], 4, 5)) == [0, 1, 2, 3]
    # ties go to the lower page index
    sel = O.select_from_shares(np.array([0.1, 0.3, 0.3, 0.3]), np.arange(1, 5), [0, 5], 6, 4)
    assert list(sel) == [0, 2, 3, 5]


def pin_select_bruteforce(O):
    """Cor. 3: the selected set maximises the summed averaged share over all
    shared sets that contain the forced pages (exhaustive on n = 10, k = 5)."""
    rng = _rng(19)
    B, d, r, G = 64, 128, 8, 4
    n, k = 10, 5
    T = n * B
    for trial in range(5):
        pages = _unit_pages(rng, n, B, d, 10, 0.1, carriers=rng.choice(n, 2))
        q = rng.standard_normal((G, d))
        S = {j: O.page_summary(pages[j], r) for j in range(n)}
        u = O.select_unit(q, S, T, B, k)
        assert set(u.forced) <= set(u.selected.tolist()) and len(u.selected) == k
        best = max(sum(u.mbar[list(u.cand).index(j)] for j in sub)
                   for sub in itertools.combinations(u.cand.tolist(), k - 2))
        got = sum(u.mbar[list(u.cand).index(j)] for j in u.selected if j in set(u.cand.tolist()))
        assert abs(got - best) < 1e-15


def pin_exact_rank_selection_and_retention(O):
    """Thm. 1(i): exactly rank-r pages select as the exact-LSE rule does;
    Thm. 1(ii): on noisy pages the retained exact share is >= e^{-4 eta} of the best."""
    rng = _rng(23)
    B, d, r, G, n, k = 64, 128, 8, 4, 48, 10
    T = n * B
    q = rng.standard_normal((G, d)) * 2.0
    for noise, exact in ((0.0, True), (0.3, False)):
        pages = _unit_pages(rng, n, B, d, 6 if exact else 12, noise, carriers=(7, 30))
        S = {j: O.page_summary(pages[j], r) for j in range(n)}
        u = O.select_unit(q, S, T, B, k)
        se = np.stack([O.exact_log_mass(q, pages[j]) for j in u.cand], axis=1)
        mbe = O.share_average(O.page_shares(se))
        exact_sel = O.select_from_shares(mbe, u.cand, u.forced, n, k)
        eta = np.abs(u.scores - se).max()
        if exact:
            assert eta < 1e-9
            assert list(exact_sel) == list(u.selected)
        idx = {int(j): i for i, j in enumerate(u.cand)}
        got = sum(mbe[idx[j]] for j in u.selected if j in idx)
        best = sum(mbe[idx[j]] for j in exact_sel if j in idx)
        assert got >= math.exp(-4 * eta) * best - 1e-15


# ---------------------------------------------------------------- attention
def pin_attention(O):
    """Section 2 attention: uniform and two-token closed forms; Lemma 1's exact
    identity o - o_S = eps (v_bar_Sc - v_bar_S); restriction to all pages = dense."""
    rng = _rng(29)
    d = 128
    q = rng.standard_normal((2, d))
    k = rng.standard_normal(d)
    V = rng.standard_normal((7, d))
    o, lse = O.attend(q, np.tile(k, (7, 1)), V)
    assert np.allclose(o, V.mean(axis=0), atol=1e-12)
    assert np.allclose(lse, q @ k / math.sqrt(d) + math.log(7), atol=1e-12)
    K2 = rng.standard_normal((2, d))
    V2 = rng.standard_normal((2, d))
    o, _ = O.attend(q, K2, V2)
    a1 = 1.0 / (1.0 + np.exp((q @ K2[1] - q @ K2[0]) / math.sqrt(d)))
    assert np.allclose(o, a1[:, None] * V2[0] + (1 - a1)[:, None] * V2[1], atol=1e-12)
    # Lemma 1 identity on a random cache
    T = 300
    K = rng.standard_normal((T, d))
    Vv = rng.standard_normal((T, d))
    keep = rng.random(T) < 0.3
    o_all, l_all = O.attend(q, K, Vv)
    o_s, l_s = O.attend(q, K[keep], Vv[keep])
    o_c, _ = O.attend(q, K[~keep], Vv[~keep])
    eps = 1.0 - np.exp(l_s - l_all)
    assert np.allclose(o_all - o_s, eps[:, None] * (o_c - o_s), atol=1e-12)
    o0, l0 = O.attend(q, np.zeros((0, d)), np.zeros((0, d)))
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))


def pin_paged_attention(O):
    """Paged gather: attending every page of a paged cache equals attending the
    contiguous token array; the partial tail contributes only its valid tokens."""
    rng = _rng(31)
    B, d, Hk, G = 16, 128, 2, 2
    T = 5 * B + 7
    n = -(-T // B)
    nb = n + 3
    K = rng.standard_normal((Hk, T, d))
    Vv = rng.standard_normal((Hk, T, d))
    perm = rng.permutation(nb)
    k_cache = np.full((nb, Hk, B, d), 0x7FC0, dtype=np.uint16)
    v_cache = np.full((nb, Hk, B, d), 0x7FC0, dtype=np.uint16)

    def bits(x):
        u = x.astype(np.float32).view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    Kb, Vb = bits(K), bits(Vv)
    for j in range(n):
        nv = min(B, T - j * B)
        k_cache[perm[j], :, :nv] = Kb[:, j * B:j * B + nv]
        v_cache[perm[j], :, :nv] = Vb[:, j * B:j * B + nv]
    bt = np.full((1, n + 2), -1, dtype=np.int32)
    bt[0, :n] = perm[:n]
    q = rng.standard_normal((G, d))
    for h in range(Hk):
        o, lse = O.dense_unit(q, k_cache, v_cache, bt, T, 0, h)
        Kf = O.bf16_to_f64(Kb[h])
        Vf = O.bf16_to_f64(Vb[h])
        o2, l2 = O.attend(q, Kf, Vf)
        assert np.allclose(o, o2, atol=1e-12) and np.allclose(lse, l2, atol=1e-12)
        assert np.all(np.isfinite(o))




def pin_quantizer_example(O):
    """Quantised summary (section 4 "Build", reading R8): hand-computed int4
    and int8 codes, exact in float32, whose ties fix round-half-even."""
    fx = _golden("quantizer_example.json")
    for key in ("int4", "int8"):
        e = fx[key]
        codes, scale = O.quantize_symmetric(np.array(e["x"], dtype=np.float32), e["qmax"])
        assert float(scale) == e["scale"], (key, scale)
        assert codes.tolist() == e["codes"], (key, codes.tolist())
    assert O.INT4_QMAX == 7 and O.INT8_QMAX == 127


def pin_quantizer_bounds(O):
    """Symmetric absmax quantisation: |x - code * scale| <= scale / 2, the
    largest |x| maps to +-qmax, codes stay in [-qmax, qmax], an all-zero group
    has scale 0 and zero codes, and scaling a group by a power of two scales
    only its scale."""
    rng = _rng(23)
    for qmax in (7, 127):
        for _ in range(200):
            x = (rng.standard_normal(int(rng.integers(1, 130))) * rng.uniform(1e-3, 10)).astype(np.float32)
            codes, scale = O.quantize_symmetric(x, qmax)
            assert np.abs(codes).max() == qmax
            assert codes.min() >= -qmax and codes.max() <= qmax
            err = np.abs(x.astype(np.float64) - codes * float(scale)).max()
            assert err <= float(scale) * (0.5 + 1e-5), (err, scale)
            c2, s2 = O.quantize_symmetric(np.float32(4.0) * x, qmax)
            assert np.array_equal(c2, codes) and float(s2) == 4.0 * float(scale)
        z, zs = O.quantize_symmetric(np.zeros(9, dtype=np.float32), qmax)
        assert float(zs) == 0.0 and not z.any()


def pin_quantized_summary_groups(O):
    """Section 4 "Build": one scale per basis column (int4), one per
    coefficient row and one for the centroid (int8).  Scaling one column of V
    or one row of C by 2 changes that group's scale only; the dequantised
    record reconstructs the summary to within half a step per entry."""
    rng = _rng(29)
    keys = rng.standard_normal((16, 32))
    s = O.page_summary(keys, 6)
    mu, V, C = s.mu.astype(np.float32), s.V.astype(np.float32), s.C.astype(np.float32)
    q = O.quantize_summary(mu, V, C)
    assert q.v_codes.shape == V.shape and q.v_scales.shape == (V.shape[1],)
    assert q.c_codes.shape == C.shape and q.c_scales.shape == (C.shape[0],)
    assert np.abs(q.v_codes).max() <= 7 and np.abs(q.c_codes).max() <= 127
    V2 = V.copy(); V2[:, 2] *= 2
    q2 = O.quantize_summary(mu, V2, C)
    assert np.array_equal(q2.v_codes, q.v_codes)
    assert q2.v_scales[2] == 2 * q.v_scales[2]
    assert np.array_equal(np.delete(q2.v_scales, 2), np.delete(q.v_scales, 2))
    C2 = C.copy(); C2[5] *= 2
    q3 = O.quantize_summary(mu, V, C2)
    assert np.array_equal(q3.c_codes, q.c_codes) and q3.c_scales[5] == 2 * q.c_scales[5]
    assert np.array_equal(np.delete(q3.c_scales, 5), np.delete(q.c_scales, 5))
    d = O.dequantized_summary(q)
    assert np.all(np.abs(d.V - V) <= q.v_scales[None, :] * 0.5 + 1e-7)
    assert np.all(np.abs(d.C - C) <= q.c_scales[:, None] * 0.5 + 1e-6)
    assert np.all(np.abs(d.mu - mu) <= float(q.mu_scale) * 0.5 + 1e-7)


def pin_unit_driver(O):
    """The whole-unit drivers follow the stated conventions (section 2; section
    4 "Build"): query head g uses KV head g // G (contiguous groups), the page
    budget is k = ceil(b / B) pages, and only complete pages get a summary
    ("once, when a page completes").  The other groups' queries and every slot
    past a sequence's last token are NaN, so a driver that reads them gives a
    NaN result; sparse and dense outputs are checked against attention over
    the contiguous arrays the cache was filled from."""
    rng = _rng(37)
    B, d, Hk, G, r = 16, 128, 2, 2, 4
    Hq = Hk * G
    T = 5 * B + 7                     # five complete pages and a partial tail
    n = -(-T // B)
    nb = n + 2
    K = rng.standard_normal((Hk, T, d))
    Vv = rng.standard_normal((Hk, T, d))
    K[:, 3 * B:4 * B] += 1.0          # one page that should win the selection

    def bits(x):
        u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    perm = rng.permutation(nb)
    k_cache = np.full((nb, Hk, B, d), 0x7FC0, dtype=np.uint16)
    v_cache = np.full((nb, Hk, B, d), 0x7FC0, dtype=np.uint16)
    Kb, Vb = bits(K), bits(Vv)
    for j in range(n):
        nv = min(B, T - j * B)
        k_cache[perm[j], :, :nv] = Kb[:, j * B:j * B + nv]
        v_cache[perm[j], :, :nv] = Vb[:, j * B:j * B + nv]
    bt = np.full((1, n + 1), -1, dtype=np.int32)
    bt[0, :n] = perm[:n]
    seq = np.array([T], dtype=np.int32)
    budget = 3 * B + 1                # k = ceil(49 / 16) = 4, floor would give 3
    for h in range(Hk):
        qf = rng.standard_normal((Hq, d))
        qf[np.arange(Hq) // G != h] = np.nan          # other groups' queries
        q_bits = bits(qf)[None]
        res = O.run_unit(q_bits, k_cache, v_cache, bt, seq, Hk, r, budget, 0, h, dense=True)
        # complete pages only: pages 0..4 summarised, the partial tail is not
        assert sorted(res.summaries) == list(range(n - 1)), sorted(res.summaries)
        for s in res.summaries.values():
            assert np.all(np.isfinite(s.V)) and np.all(np.isfinite(s.C))
        # k = ceil(b / B) pages, the forced pair inside
        sel = [int(j) for j in res.sel.selected]
        assert len(sel) == 4 and sel[0] == 0 and sel[-1] == n - 1, sel
        # the group's own queries, against the contiguous arrays
        q_own = O.bf16_to_f64(q_bits[0, h * G:(h + 1) * G])
        Kf, Vf = O.bf16_to_f64(Kb[h]), O.bf16_to_f64(Vb[h])
        o2, l2 = O.attend(q_own, Kf, Vf)
        assert np.all(np.isfinite(res.o_dense))
        assert np.allclose(res.o_dense, o2, atol=1e-12) and np.allclose(res.lse_dense, l2, atol=1e-12)
        idx = np.concatenate([np.arange(j * B, min(T, (j + 1) * B)) for j in sel])
        o3, l3 = O.attend(q_own, Kf[idx], Vf[idx])
        assert np.allclose(res.o_sparse, o3, atol=1e-12) and np.allclose(res.lse_sparse, l3, atol=1e-12)
    # a length that is a multiple of B: the last page is complete and summarised
    res = O.run_unit(q_bits, k_cache, v_cache, bt, np.array([5 * B], dtype=np.int32), Hk, r,
                     budget, 0, Hk - 1)
    assert sorted(res.summaries) == list(range(5))


ALL_PINS = [
    pin_worked_example, pin_isotropic_null, pin_exact_rank, pin_full_rank_r15,
    pin_svd_route, pin_centroid_closed_form, pin_prop2, pin_lemma3,
    pin_shares_and_sandwich, pin_budget_rule, pin_forced_pages, pin_select_bruteforce,
    pin_exact_rank_selection_and_retention, pin_attention, pin_paged_attention,
    pin_quantizer_example, pin_quantizer_bounds, pin_quantized_summary_groups,
    pin_unit_driver,
]
# the cheap ones, for the planted-mistake runs
FAST_PINS = [p for p in ALL_PINS if p is not pin_isotropic_null]
