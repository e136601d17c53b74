"""CUDA path against the fp64 oracle on small seeded workloads (several tiles,
ragged tails, GQA group sizes 1..8, ranks 4..16, the degenerate cases)."""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

TINY = W.get("tiny")

CASES = {
    "tiny": TINY,
    # partial tail page (n = 65), n <= k, n = k + 1, single page, empty sequence
    "ragged": TINY.with_(batch=5, seq_lens=(4096 + 37, 200, 64 * 9, 40, 0), seed=2001),
    "group1": TINY.with_(n_q_heads=2, n_kv_heads=2, seed=2002),
    "group2": TINY.with_(n_q_heads=4, n_kv_heads=2, seed=2003),
    "group8": TINY.with_(n_q_heads=16, n_kv_heads=2, seed=2004),
    "k2_forced_only": TINY.with_(budget_tokens=100, seed=2005),
    "rank4": TINY.with_(rank=4, seed=2006),
    "rank3": TINY.with_(rank=3, seed=2007),
    "rank16": TINY.with_(rank=16, seed=2008),
    # many selection chunks per unit, global component, 1% carriers
    "multichunk": TINY.with_(context=64 * 300, global_rank=16, carrier_count=None,
                             carrier_frac=0.01, budget_tokens=2048, seed=2009),
    "batch_heads": TINY.with_(batch=3, n_q_heads=16, n_kv_heads=4, context=64 * 70,
                              global_rank=16, seed=2010),
    # more than 2048 candidates: several finalize slices, merged by the last one
    "slices3": TINY.with_(context=64 * 4200 + 11, global_rank=16, carrier_count=None,
                          carrier_frac=0.01, budget_tokens=2048, seed=2014),
    # k - 2 > 32, with one and with several slices
    "k40": TINY.with_(context=64 * 300, budget_tokens=64 * 40, seed=2015),
    "k40_slices3": TINY.with_(context=64 * 4200, budget_tokens=64 * 40, global_rank=16,
                              seed=2016),
    # G = 8 with k - 2 > 32 over three slices; G = 1 over two (finalize
    # register pressure and the slice merge at the group-size extremes)
    "group8_k40_slices3": TINY.with_(n_q_heads=16, n_kv_heads=2, context=64 * 4200 + 11,
                                     budget_tokens=64 * 40, seed=2017),
    "group1_slices2": TINY.with_(n_q_heads=2, n_kv_heads=2, context=64 * 2600 + 5, seed=2018),
    # more than 16384 candidates: nine slices, the last holding 6 candidates
    # (246 winners merged by direct ranking), and seventeen at B = 16 with
    # k - 2 > 32 (over 256 winners: the merge takes the bounded top-k)
    "wide_slices2": TINY.with_(n_q_heads=4, n_kv_heads=1, context=64 * 16391 + 7,
                               global_rank=16, seed=2050),
    "b16_wide_slices3_k40": TINY.with_(page_size=16, n_q_heads=4, n_kv_heads=1,
                                       context=16 * 33000 + 9, budget_tokens=16 * 40,
                                       global_rank=16, seed=2051),
    # page size 16 (four pages per decode stage)
    "b16": TINY.with_(page_size=16, seed=2020),
    "b16_ragged": TINY.with_(page_size=16, batch=5, seq_lens=(4096 + 7, 200, 16 * 33, 9, 0),
                             seed=2021),
    "b16_rank15": TINY.with_(page_size=16, rank=15, seed=2022),
    "b16_slices2": TINY.with_(page_size=16, context=16 * 2500 + 5, global_rank=16,
                              carrier_count=None, carrier_frac=0.01, seed=2023),
    "b16_k40": TINY.with_(page_size=16, budget_tokens=16 * 40, seed=2025),
    # 80 units: three splits per unit, merged through a thread-block cluster
    "cluster_merge": TINY.with_(batch=40, context=64 * 20 + 5, seed=2030),
    "b16_cluster_merge": TINY.with_(page_size=16, batch=40, context=16 * 40 + 3, seed=2031),
    # Llama layer shape at B = 16: k = 128
    "b16_gqa4_k128": TINY.with_(page_size=16, batch=2, n_q_heads=32, n_kv_heads=8,
                                context=16384, budget_tokens=2048, global_rank=16,
                                carrier_count=None, carrier_frac=0.01, seed=2024),
    # 16 KV heads (G = 2)
    "heads16": TINY.with_(n_q_heads=32, n_kv_heads=16, context=64 * 40 + 9, seed=2040),
    # ragged sequences of several lengths sharing score CTAs, 8 KV heads
    "ragged_8heads": TINY.with_(batch=6, n_q_heads=32, n_kv_heads=8,
                              seq_lens=(64 * 200 + 3, 64 * 3, 64 * 57, 0, 64 * 130 - 1, 64 * 2 + 1),
                              global_rank=16, seed=2041),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from sparse_paged_kv_gb300 import binding, build_lib
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    binding.load_library(build_lib.build())


@pytest.mark.parametrize("name", sorted(CASES))
def test_parity(name):
    inputs = W.generate(CASES[name])
    rep, layer, snap = P.run_case(inputs)
    rep.check()
    assert rep.units == CASES[name].batch * CASES[name].n_kv_heads
    print(f"{name}: e_rec*gap {rep.max_recon_gap:.2e} lse {rep.max_lse_err:.2e} out {rep.max_out_err:.2e} dense "
          f"{rep.max_dense_err:.2e} recon {rep.max_recon_rel:.2e} sigma {rep.max_sigma_rel:.2e} "
          f"degenerate {rep.degenerate} ties {rep.tie_diffs}")


@pytest.mark.parametrize("name", ["tiny", "rank3", "rank16", "multichunk", "batch_heads"])
def test_parity_jacobi_solver(name):
    """The Jacobi solver, which a sweep cap selects at page size 64, against
    the same oracle gates as the default tridiagonal solver."""
    inputs = W.generate(CASES[name])
    rep, layer, snap = P.run_case(inputs, max_sweeps=20)
    rep.check()
    assert np.all(snap["build_sweeps"] >= 1)
    print(f"jacobi {name}: recon {rep.max_recon_rel:.2e} (e_rec*gap {rep.max_recon_gap:.2e}) "
          f"sigma {rep.max_sigma_rel:.2e} lse {rep.max_lse_err:.2e}")


BF16_CASES = ["tiny", "ragged", "group8", "rank16", "multichunk", "slices3", "k40", "b16",
              "b16_ragged"]


@pytest.mark.parametrize("name", BF16_CASES)
def test_parity_bf16_records(name):
    """bf16 summary records: selection and scores against the oracle scoring the
    stored records; decode as for fp32; record error against fp64 reported."""
    inputs = W.generate(CASES[name])
    rep, layer, snap = P.run_case(inputs, summary_dtype=1)
    rep.check()
    assert rep.units == CASES[name].batch * CASES[name].n_kv_heads
    # bf16 keeps 8 significant bits: the stored C V^T is a rounded copy
    assert rep.max_record_err < 2e-2, rep.max_record_err
    print(f"bf16 {name}: lse {rep.max_lse_err:.2e} out {rep.max_out_err:.2e} record vs fp64 "
          f"{rep.max_record_err:.2e} ties {rep.tie_diffs}")


I4_CASES = ["tiny", "ragged", "group1", "group2", "group8", "rank16", "rank3", "multichunk",
            "slices3", "k40", "b16", "b16_ragged", "b16_rank15", "cluster_merge", "batch_heads",
            "group8_k40_slices3", "heads16", "ragged_8heads", "b16_gqa4_k128",
            "b16_wide_slices3_k40"]


@pytest.mark.parametrize("name", I4_CASES)
def test_parity_i4_records(name):
    """Quantised records (int4 basis, int8 coefficients and centroid):
    selection and scores against the oracle scoring the stored codes; decode as
    for fp32; the dequantised record's distance from the fp64 summary reported."""
    inputs = W.generate(CASES[name])
    rep, layer, snap = P.run_case(inputs, summary_dtype=2)
    rep.check()
    assert rep.units == CASES[name].batch * CASES[name].n_kv_heads
    # an int4 basis keeps 4 bits: its reconstruction is a coarse copy
    assert rep.max_record_err < 0.25, rep.max_record_err
    print(f"i4 {name}: lse {rep.max_lse_err:.2e} out {rep.max_out_err:.2e} record vs fp64 "
          f"{rep.max_record_err:.2e} ties {rep.tie_diffs}")


@pytest.mark.parametrize("name", ["tiny", "rank16", "rank3", "b16"])
def test_i4_codes_equal_oracle_quantiser(name):
    """The GPU's quantised record holds exactly the oracle quantiser's codes and
    scales of the GPU's own float record (same pages, same build): every
    integer code is decided in float32 on both sides."""
    import torch
    from sparse_paged_kv_gb300 import binding as Bd, runtime
    w = CASES[name]
    inputs = W.generate(w)
    lay = {}
    for dt in (Bd.LOCKS_SUMMARY_F32, Bd.LOCKS_SUMMARY_I4):
        lay[dt] = runtime.LocksLayer.from_inputs(inputs, summary_dtype=dt)
        lay[dt].build()
    torch.cuda.synchronize()
    r = w.rank
    for b, h in [(0, 0), (w.batch - 1, w.n_kv_heads - 1)]:
        _, cand = O.forced_and_candidates(int(inputs.seq_lens[b]), w.page_size)
        blocks = inputs.block_table[b, [int(j) for j in cand]]
        mu32, V32, C32 = lay[Bd.LOCKS_SUMMARY_F32].host_records(blocks, h)
        raw = lay[Bd.LOCKS_SUMMARY_I4].summaries[torch.as_tensor(blocks).long().cuda(), h]
        mu_c, mu_s, v_c, v_s, c_c, c_s = Bd.unpack_i4(raw.cpu().numpy(), lay[Bd.LOCKS_SUMMARY_I4].cfg)
        for n in range(len(blocks)):
            q = O.quantize_summary(mu32[n].astype(np.float32), V32[n].astype(np.float32),
                                   C32[n].astype(np.float32))
            assert np.array_equal(q.mu_codes, mu_c[n]) and q.mu_scale == mu_s[n], (b, h, n)
            assert np.array_equal(q.v_codes, v_c[n][:, :r]), (b, h, n)
            assert np.array_equal(q.v_scales, v_s[n][:r]), (b, h, n)
            assert not v_c[n][:, r:].any() and not v_s[n][r:].any()
            assert np.array_equal(q.c_codes, c_c[n][:, :r]) and not c_c[n][:, r:].any()
            assert np.array_equal(q.c_scales, c_s[n]), (b, h, n)


def test_empty_sequence_outputs_zero():
    inputs = W.generate(CASES["ragged"])
    rep, layer, snap = P.run_case(inputs, units=[(4, 0), (4, 1)])
    rep.check()
    assert np.all(snap["selected"][4] == -1)
    assert np.all(snap["out"][4] == 0) and np.all(np.isneginf(snap["out_lse"][4]))


def test_repeat_calls_reuse_workspace():
    """Tickets reset themselves: the same workspace gives the same result twice."""
    import torch
    inputs = W.generate(CASES["multichunk"])
    rep, layer, snap = P.run_case(inputs, units=[(0, 0)])
    rep.check()
    for _ in range(3):
        layer.step()
        layer.dense_decode()
    torch.cuda.synchronize()
    assert np.array_equal(layer.selected.cpu().numpy(), snap["selected"])
    assert np.array_equal(layer.out.float().cpu().numpy(), snap["out"].astype(np.float32))
    assert np.array_equal(layer.out_dense.float().cpu().numpy(),
                          snap["out_dense"].astype(np.float32))


def test_bad_block_id_is_flagged_and_skipped():
    import torch
    from sparse_paged_kv_gb300 import binding as B
    inputs = W.generate(TINY.with_(seed=2011))
    rep, layer, snap = P.run_case(inputs, units=[(0, 0)], dense=False)
    rep.check()
    bt = layer.block_table.clone()
    bt[0, 5] = layer.cfg.num_blocks + 7          # outside the pool
    layer.block_table = bt
    layer.status.zero_()
    layer.step()
    layer.dense_decode()
    torch.cuda.synchronize()
    st = int(layer.status.cpu()[0])
    assert st & B.LOCKS_DEV_BAD_BLOCK_ID
    assert not st & B.LOCKS_DEV_WAIT_TIMEOUT
    assert np.all(np.isfinite(layer.out.float().cpu().numpy()))


def test_jacobi_sweep_cap_is_flagged():
    import torch
    from sparse_paged_kv_gb300 import binding as B
    inputs = W.generate(TINY.with_(seed=2012))
    from sparse_paged_kv_gb300 import runtime
    layer = runtime.LocksLayer.from_inputs(inputs)
    ids = runtime.complete_page_blocks(inputs.block_table, inputs.seq_lens, 64)[:8]
    st = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    layer.build(torch.from_numpy(ids).cuda(), status=st, max_sweeps=1)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert np.all((s >> 16) & B.LOCKS_DEV_NOT_CONVERGED)
    assert np.all((s & 0xFFFF) == 1)
    layer.build(torch.from_numpy(ids).cuda(), status=st)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert np.all((s >> 16) == 0) and np.all((s & 0xFFFF) <= 20)


def test_graph_replay_matches_eager_and_oracle():
    """A captured step replays bit-identically to the eager calls, reads q at
    replay time, and still passes the oracle gates with a new q."""
    import torch
    inputs = W.generate(CASES["batch_heads"])
    rep, layer, snap = P.run_case(inputs, dense=False, check_build=False)
    rep.check()
    graph = layer.capture_step()
    rng = np.random.default_rng(77)
    for trial in range(2):
        q_new = W.f32_to_bf16_bits(rng.standard_normal(inputs.q.shape).astype(np.float32))
        layer.q.copy_(torch.from_numpy(q_new.view(np.int16)).view(layer.q.dtype).cuda())
        graph.replay()
        torch.cuda.synchronize()
        sel_g = layer.selected.cpu().numpy().copy()
        out_g = layer.out.float().cpu().numpy().copy()
        lse_g = layer.out_lse.cpu().numpy().copy()
        layer.step()
        torch.cuda.synchronize()
        assert np.array_equal(sel_g, layer.selected.cpu().numpy())
        assert np.array_equal(out_g, layer.out.float().cpu().numpy())
        assert np.array_equal(lse_g, layer.out_lse.cpu().numpy())
        # the replayed result against the oracle on the new query
        inputs2 = dataclasses.replace(inputs, q=q_new)
        snap2 = {"selected": sel_g, "out": out_g.astype(np.float64),
                 "out_lse": lse_g.astype(np.float64)}
        rep2 = P.Report()
        w = inputs.workload
        for b, h in [(0, 0), (w.batch - 1, w.n_kv_heads - 1)]:
            res = O.run_unit(inputs2.q, inputs2.k_cache, inputs2.v_cache, inputs2.block_table,
                             inputs2.seq_lens, w.n_kv_heads, w.rank, w.budget_tokens, b, h)
            P.compare_select(layer, snap2, res, rep2)
            P.compare_sparse_decode(layer, inputs2, snap2, res, rep2)
        rep2.check()
    assert int(layer.status.cpu()[0]) == 0


@pytest.mark.parametrize("summary_dtype,context", [
    (0, 64 * 1500 + 9), (2, 64 * 1500 + 9), (0, 64 * 4200 + 11), (2, 64 * 4200 + 11),
    (0, 64 * 16391 + 7)])
def test_equal_shares_select_the_smallest_pages(context, summary_dtype):
    """With zero queries every logit is 0, so every complete page has the same
    s_hat and the same share: the selection is then decided by the tie rule
    alone (between equal shares the smaller page), i.e. pages 1 .. k-2 besides
    the forced ones.  1499 candidates in one slice, or three or nine slices
    of up to 2048, leave more equal keys above the top-K's lower bound than
    its ranking buffer holds, so the bit-by-bit search decides; the slices'
    winners are then merged through the ranking path."""
    import torch
    from sparse_paged_kv_gb300 import runtime
    w = TINY.with_(context=context, seed=2040)
    gen = W.generate(w)
    inputs = dataclasses.replace(gen, q=np.zeros_like(gen.q))
    layer = runtime.LocksLayer.from_inputs(inputs, summary_dtype=summary_dtype)
    layer.build()
    layer.select()
    torch.cuda.synchronize()
    assert int(layer.status.cpu()[0]) == 0
    sel = layer.selected.cpu().numpy()
    k = O.page_budget(w.budget_tokens, w.page_size)
    for b in range(w.batch):
        n = -(-int(inputs.seq_lens[b]) // w.page_size)
        expect = [0] + list(range(1, k - 1)) + [n - 1]
        for h in range(w.n_kv_heads):
            assert list(sel[b, h]) == expect, (b, h, list(sel[b, h]))
