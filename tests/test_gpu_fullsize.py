"""CUDA path at the full benchmark workloads, in the launch configuration the
bench times, for every summary record type (fp32, bf16 and the quantised
int4/int8 record): the oracle recomputes sampled (sequence, KV head) units end
to end (build, scores, shares, selection, sparse and dense attention), and
every unit is checked for what holds at any size (shares sum to 1, forced
pages kept, ascending unique ids, clean device status).  bf16 and quantised
records are gated against the oracle scoring the stored records; the
quantised codes of a sample of pages are checked bit for bit against the
oracle quantiser applied to the GPU's own fp32 record of the same page."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

FULL = ["llama32k", "long128k", "qwen16k", "1m"]
DTYPES = {0: "f32", 1: "bf16", 2: "i4"}
CASES = [(name, dt) for name in FULL for dt in DTYPES]
_cache = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from sparse_paged_kv_gb300 import binding, build_lib
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    binding.load_library(build_lib.build())
    yield
    _cache.clear()


def _inputs(name):
    """Generated inputs of one workload, kept while its record types run."""
    if name not in _cache:
        _cache.clear()
        _cache[name] = W.generate(W.get(name))
    return _cache[name]


def _check_i4_codes(layer, inputs, b, h, n_pages=48):
    """Quantised codes and scales of a sample of the unit's candidate pages
    equal the oracle quantiser's on the GPU's fp32 record of the same page."""
    import torch
    from sparse_paged_kv_gb300 import binding as Bd
    w = inputs.workload
    _, cand = O.forced_and_candidates(int(inputs.seq_lens[b]), w.page_size)
    rng = np.random.default_rng(7)
    pick = np.sort(rng.choice(len(cand), size=min(n_pages, len(cand)), replace=False))
    blocks = inputs.block_table[b, [int(cand[i]) for i in pick]]
    f32 = layer.sharing_inputs(Bd.LOCKS_SUMMARY_F32)
    f32.build(torch.from_numpy(np.ascontiguousarray(blocks, dtype=np.int32)).cuda())
    torch.cuda.synchronize()
    mu32, V32, C32 = f32.host_records(blocks, h)
    raw = layer.summaries[torch.as_tensor(blocks).long().cuda(), h]
    mu_c, mu_s, v_c, v_s, c_c, c_s = Bd.unpack_i4(raw.cpu().numpy(), layer.cfg)
    r = w.rank
    for n in range(len(blocks)):
        q = O.quantize_summary(mu32[n].astype(np.float32), V32[n].astype(np.float32),
                               C32[n].astype(np.float32))
        assert np.array_equal(q.mu_codes, mu_c[n]) and q.mu_scale == mu_s[n], (b, h, n)
        assert np.array_equal(q.v_codes, v_c[n][:, :r]) and np.array_equal(q.v_scales, v_s[n][:r])
        assert np.array_equal(q.c_codes, c_c[n][:, :r]) and np.array_equal(q.c_scales, c_s[n])
    del f32


@pytest.mark.parametrize("name,dtype", CASES, ids=[f"{n}-{DTYPES[d]}" for n, d in CASES])
def test_full_size(name, dtype):
    import torch
    inputs = _inputs(name)
    w = inputs.workload
    last = (w.batch - 1, w.n_kv_heads - 1)
    rep, layer, snap = P.run_case(inputs, units=[(0, 0), last], dense=(dtype == 0),
                                  summary_dtype=dtype)
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
    assert np.all(np.isfinite(snap["out"]))
    if dtype == 0:
        assert np.all(np.isfinite(snap["out_dense"]))
    assert snap["status"] == 0
    assert np.all(snap["build_sweeps"] <= 20)
    if dtype == 1:
        assert rep.max_record_err < 2e-2, rep.max_record_err
    if dtype == 2:
        _check_i4_codes(layer, inputs, *last)
    del layer
    torch.cuda.empty_cache()
    print(f"{name} {DTYPES[dtype]}: lse {rep.max_lse_err:.2e} share abs {rep.max_share_abs:.2e} "
          f"rel {rep.max_share_rel:.2e} out {rep.max_out_err:.2e} dense {rep.max_dense_err:.2e} "
          f"recon {rep.max_recon_rel:.2e} (e_rec*gap {rep.max_recon_gap:.2e}) record "
          f"{rep.max_record_err:.2e} degenerate {rep.degenerate} ties {rep.tie_diffs}")
