"""CUDA path at the full benchmark workloads, in the launch configuration the
bench times: the oracle recomputes sampled (sequence, KV head) units end to
end (build, scores, selection, sparse and dense attention), and every unit is
checked for what holds at any size (shares sum to 1, forced pages kept,
ascending unique ids, clean device status)."""
import numpy as np
import pytest

import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

FULL = ["llama32k", "long128k", "qwen16k", "1m"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from sparse_paged_kv_gb300 import binding, build_lib
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    binding.load_library(build_lib.build())


@pytest.mark.parametrize("name", FULL)
def test_full_size(name):
    import torch
    w = W.get(name)
    inputs = W.generate(w)
    last = (w.batch - 1, w.n_kv_heads - 1)
    rep, layer, snap = P.run_case(inputs, units=[(0, 0), last])
    rep.check()
    k = w.page_budget
    n = -(-w.context // w.page_size)
    sel = snap["selected"]
    shares = snap["page_share"]
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            row = [int(x) for x in sel[b, h] if x >= 0]
            assert len(row) == min(k, n)
            assert row == sorted(set(row))
            assert row[0] == 0 and row[-1] == n - 1
            s = shares[b, h, 1:n - 1]
            assert abs(s.sum() - 1.0) < 1e-3, (b, h, s.sum())
    assert np.all(np.isfinite(snap["out"])) and np.all(np.isfinite(snap["out_dense"]))
    assert snap["status"] == 0
    assert np.all(snap["build_sweeps"] <= 20)
    del layer
    torch.cuda.empty_cache()
    print(f"{name}: lse {rep.max_lse_err:.2e} out {rep.max_out_err:.2e} dense "
          f"{rep.max_dense_err:.2e} recon {rep.max_recon_rel:.2e} degenerate {rep.degenerate} "
          f"ties {rep.tie_diffs}")


def test_full_size_bf16_records():
    """llama32k with bf16 summary records, two sampled units end to end."""
    import torch
    w = W.get("llama32k")
    inputs = W.generate(w)
    rep, layer, snap = P.run_case(inputs, units=[(0, 0), (w.batch - 1, w.n_kv_heads - 1)],
                                  dense=False, summary_dtype=1)
    rep.check()
    assert snap["status"] == 0
    assert rep.max_record_err < 2e-2, rep.max_record_err
    del layer
    torch.cuda.empty_cache()
    print(f"llama32k bf16: lse {rep.max_lse_err:.2e} out {rep.max_out_err:.2e} record vs fp64 "
          f"{rep.max_record_err:.2e} ties {rep.tie_diffs}")


def test_full_size_i4_records():
    """llama32k with quantised records (int4 basis), two sampled units end to end."""
    import torch
    w = W.get("llama32k")
    inputs = W.generate(w)
    rep, layer, snap = P.run_case(inputs, units=[(0, 0), (w.batch - 1, w.n_kv_heads - 1)],
                                  dense=False, summary_dtype=2)
    rep.check()
    assert snap["status"] == 0
    del layer
    torch.cuda.empty_cache()
    print(f"llama32k i4: lse {rep.max_lse_err:.2e} out {rep.max_out_err:.2e} record vs fp64 "
          f"{rep.max_record_err:.2e} ties {rep.tie_diffs}")
