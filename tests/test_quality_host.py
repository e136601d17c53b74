"""The quality harness's rival selectors against what bounds them (CPU):
centroid-only scores are at most the exact page log-mass (Jensen's inequality:
the log-sum-exp of the logits is at least log nv plus their mean), and Quest's
envelope scores are at least it (Lemma 2: the elementwise key envelope bounds
every logit from above).  A dropped term or a swapped min/max breaks one of
the two inequalities."""
import numpy as np

import workloads as W
from tests import quality as Q

W_SMALL = W.get("tiny").with_(carrier_count=2, carrier_token=True, carrier_bias=4.0, seed=5101)


def test_rival_scores_bracket_the_exact_log_mass():
    inputs = W.generate(W_SMALL)
    w = inputs.workload
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            ex = Q.unit_exact(inputs, b, h)
            s = ex["s"]
            cen = Q.rival_log_mass(inputs, b, h, "centroid")
            qst = Q.rival_log_mass(inputs, b, h, "quest")
            ok = np.isfinite(s)
            assert np.array_equal(ok, np.isfinite(cen)) and np.array_equal(ok, np.isfinite(qst))
            assert np.all(cen[ok] <= s[ok] + 1e-9)
            assert np.all(qst[ok] >= s[ok] - 1e-9)
            # neither bound is trivially loose on these pages
            assert np.median(s[ok] - cen[ok]) < 5.0 and np.median(qst[ok] - s[ok]) < 50.0


def test_rival_selection_keeps_the_forced_pages():
    inputs = W.generate(W_SMALL)
    ex = Q.unit_exact(inputs, 0, 0)
    for rule in ("centroid", "quest"):
        sel = [int(p) for p in Q.rival_selection(ex, Q.rival_log_mass(inputs, 0, 0, rule))]
        assert 0 in sel and ex["n"] - 1 in sel
        assert len([p for p in sel if p >= 0]) == min(ex["k"], ex["n"])


def test_single_token_carriers_shift_one_row():
    """The peaky variant shifts one seeded token of each carrier page by
    carrier_bias along the group query direction (a unit vector), where the
    page-wide variant shifts every token: against no carriers exactly one row
    of the page moves, by carrier_bias; against the page-wide variant all the
    other rows differ by carrier_bias.  So the centroid moves by bias / B."""
    bias, B = W_SMALL.carrier_bias, W_SMALL.page_size
    tok = W.generate(W_SMALL)
    page = W.generate(W_SMALL.with_(carrier_token=False))
    none = W.generate(W_SMALL.with_(carrier_count=0))
    assert [list(c) for c in tok.carriers[0]] == [list(c) for c in page.carriers[0]]
    car = int(tok.carriers[0][0][0])
    blk = int(tok.block_table[0, car])

    def keys(x):
        return W.bf16_bits_to_f32(x.k_cache[blk, 0]).astype(np.float64)

    d_none = np.linalg.norm(keys(tok) - keys(none), axis=1)
    d_page = np.linalg.norm(keys(tok) - keys(page), axis=1)
    moved = np.nonzero(d_none > 1e-6)[0]
    assert len(moved) == 1 and abs(d_none[moved[0]] - bias) < 0.05
    assert d_page[moved[0]] < 1e-6
    others = np.delete(d_page, moved[0])
    assert others.shape == (B - 1,) and np.all(np.abs(others - bias) < 0.05)
