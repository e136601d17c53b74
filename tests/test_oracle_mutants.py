"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU)
and check that the pins catch every one of them."""
import os
import sys
import types

import pytest

from tests import oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "locks_oracle.py")

MUTANTS = {
    "no_centring": ("D = K - mu ", "D = K - 0.0 * mu "),
    "centroid_first_key": ("mu = K.mean(axis=0)", "mu = K[0]"),
    "ascending_modes": ('order = np.argsort(-w, kind="stable")', 'order = np.argsort(w, kind="stable")'),
    "basis_times_sigma": ("V[:, k] = D.T @ U[:, k] / s", "V[:, k] = D.T @ U[:, k] * s"),
    "coeff_over_sigma": ("C[:, k] = U[:, k] * s", "C[:, k] = U[:, k] / s"),
    "tail_off_by_one": ("tail = np.clip(w[r:]", "tail = np.clip(w[r + 1:]"),
    "score_scale_1_over_d": ("return (a[:, None] + p @ s.C.T) / math.sqrt(d)",
                             "return (a[:, None] + p @ s.C.T) / d"),
    "score_drops_centroid": ("return (a[:, None] + p @ s.C.T)", "return (0.0 * a[:, None] + p @ s.C.T)"),
    "score_reversed_dims": ("p = q @ s.V ", "p = q[:, ::-1] @ s.V "),
    "exact_mass_scale": ("return _lse(q @ K.T / math.sqrt(q.shape[1]), axis=-1)",
                         "return _lse(q @ K.T / q.shape[1], axis=-1)"),
    "shares_wrong_norm": ("return np.exp(scores - logz[:, None])", "return np.exp(scores - logz.mean())"),
    "group_max_not_mean": ("return np.mean(np.atleast_2d(shares), axis=0)",
                           "return np.max(np.atleast_2d(shares), axis=0)"),
    "select_smallest": ("key=lambda i: (-mbar[i], cand[i])", "key=lambda i: (mbar[i], cand[i])"),
    "tie_to_higher_index": ("key=lambda i: (-mbar[i], cand[i])", "key=lambda i: (-mbar[i], -cand[i])"),
    "forced_wrong_recent": ("forced = sorted({0, n - 1})", "forced = sorted({0, n - 2})"),
    "budget_floor": ("return -(-budget_tokens // page_size)", "return budget_tokens // page_size"),
    "sink_not_forced": ("forced = sorted({0, n - 1})", "forced = sorted({n - 1})"),
    "attend_no_scale": ("logits = q @ K.T / math.sqrt(q.shape[1])", "logits = q @ K.T"),
    "tail_page_all_tokens": ("return max(0, min(page_size, seq_len - j * page_size))", "return page_size"),
    "quant_round_half_up": ("codes = np.rint(x / scale)", "codes = np.floor(x / scale + 0.5)"),
    "quant_scale_no_qmax": ("scale = np.float32(amax / np.float32(qmax))",
                            "scale = np.float32(amax / np.float32(qmax + 1))"),
    "quant_basis_one_scale": ("v_codes[:, k], v_scales[k] = quantize_symmetric(V[:, k], INT4_QMAX)",
                              "v_codes[:, k], v_scales[k] = (quantize_symmetric(V, INT4_QMAX)[0][:, k], "
                              "quantize_symmetric(V, INT4_QMAX)[1])"),
    "quant_basis_int8": ("v_codes[:, k], v_scales[k] = quantize_symmetric(V[:, k], INT4_QMAX)",
                         "v_codes[:, k], v_scales[k] = quantize_symmetric(V[:, k], INT8_QMAX)"),
    "unit_queries_interleaved": ("q = bf16_to_f64(q_bits[b, h * G:(h + 1) * G])",
                                 "q = bf16_to_f64(q_bits[b, h::n_kv_heads])"),
    "unit_budget_floor": ("k = page_budget(budget_tokens, B)", "k = budget_tokens // B"),
    "build_partial_tail": ("n_complete = seq_len // B", "n_complete = -(-seq_len // B)"),
}


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    sys.modules["oracle_mutant"] = mod        # dataclasses look their module up here
    try:
        exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    finally:
        sys.modules.pop("oracle_mutant", None)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    mod = _mutant(*MUTANTS[name])
    caught = []
    for pin in P.FAST_PINS:
        try:
            pin(mod)
        except Exception as e:  # noqa: BLE001 -- any failure counts as caught
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin caught the planted mistake {name}"
