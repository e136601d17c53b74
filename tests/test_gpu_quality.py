"""Selection fidelity of the GPU selections on a synthetic Llama-layer
workload (Table B.1 and Table D.17 statistics of the Locks paper; see
tests/quality.py).  Asserted: what holds by construction or is proven -- the
exact selection scores 1 against itself, share-average has the largest mean
contested coverage among shared selections (Cor. 3), the per-head oracle
bounds every shared rule head by head on average.  The rest is reported."""
import numpy as np
import pytest

import workloads as W
from tests import quality as Q

pytestmark = pytest.mark.gpu

# Llama-3.1-8B layer shape, two sequences of 32K tokens, b = 2048 (k = 32)
WQ = W.get("llama32k").with_(batch=2, seed=3001)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from sparse_paged_kv_gb300 import binding, build_lib
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    binding.load_library(build_lib.build())


def _gpu_selection(inputs, summary_dtype):
    import torch
    from sparse_paged_kv_gb300 import runtime
    layer = runtime.LocksLayer.from_inputs(inputs, summary_dtype=summary_dtype)
    layer.build()
    layer.select()
    torch.cuda.synchronize()
    assert int(layer.status.cpu()[0]) == 0
    sel = layer.selected.cpu().numpy()
    del layer
    torch.cuda.empty_cache()
    return sel


def test_selection_fidelity():
    from sparse_paged_kv_gb300 import binding as Bd
    inputs = W.generate(WQ)
    w = inputs.workload
    units = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    ex = {u: Q.unit_exact(inputs, *u) for u in units}
    sels = {name: _gpu_selection(inputs, dt) for name, dt in
            (("Locks r8fp (fp32 record)", Bd.LOCKS_SUMMARY_F32),
             ("Locks r8 bf16 record", Bd.LOCKS_SUMMARY_BF16),
             ("Locks r8i4 (quantised record)", Bd.LOCKS_SUMMARY_I4))}
    rows = {"exact LSE (ceiling)": [Q.unit_stats(ex[u], ex[u]["best"]) for u in units]}
    for name, sel in sels.items():
        rows[name] = [Q.unit_stats(ex[(b, h)], sel[b, h]) for b, h in units]
    table = {name: Q.aggregate(r) for name, r in rows.items()}
    print(f"\nselection fidelity, {w.name} x{w.batch}, b = {w.budget_tokens} "
          f"(k = {ex[units[0]]['k']} of {ex[units[0]]['n']} pages)")
    for name, t in table.items():
        needle = "n/a" if t["needle"] is None else f"{100 * t['needle']:.1f}"
        print(f"  {name:32s} gamma_c {100 * t['gamma_c']:5.1f}  gamma {100 * t['gamma']:5.1f}  "
              f"recall {100 * t['recall']:5.1f}  needle {needle}")
    ceil = table["exact LSE (ceiling)"]
    assert ceil["recall"] == 1.0 and ceil["needle"] in (1.0, None)

    # Table D.17: combine rules on the exact per-head shares
    cov = {rule: np.concatenate([Q.combine_coverage(ex[u], rule) for u in units])
           for rule in ("share-average", "group-max", "group-mass", "per-head")}
    per_unit = {rule: [Q.combine_coverage(ex[u], rule) for u in units] for rule in cov}
    print("  combine rule      mean   worst    p5")
    for rule, c in cov.items():
        worst = np.mean([pu.min() for pu in per_unit[rule]])
        print(f"  {rule:15s} {c.mean():6.3f}  {worst:6.3f}  {np.percentile(c, 5):6.3f}")
    # Cor. 3: the share-average selection maximises the group-mean contested
    # coverage among shared selections of the same size
    for rule in ("group-max", "group-mass"):
        for u_sa, u_r in zip(per_unit["share-average"], per_unit[rule]):
            assert u_sa.mean() >= u_r.mean() - 1e-12
    # each head's own top set bounds any shared set on that head
    for u_sa, u_ph in zip(per_unit["share-average"], per_unit["per-head"]):
        assert np.all(u_ph >= u_sa - 1e-12)
