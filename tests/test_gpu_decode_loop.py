"""A decode loop through the library, as an engine drives it: every step
uploads only its inputs (the query and the new token's key and value rows),
locks_append_kv writes the token into the paged cache and reports the pages it
completed, locks_build_completed summarises exactly those pages on a side
stream (section 4 "Build": one build per finalised page, off the critical
path), and the step selects and decodes.  No step copies the cache or decides
on the host which pages completed.  Every step is checked against the oracle
on a host mirror of the cache that the test keeps by itself, so page
crossings, the moving incomplete tail page and the incrementally built
summaries are all exercised; at the end the device pools and lengths must
equal the mirror bit for bit."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

# lengths chosen so that within six steps pages complete at steps 1 (B), 2
# (E), 3 (A) and 4 (D), each such page is then scored as a candidate, a
# sequence starts a new page (B), one stays inside its page (C), and a
# single-page sequence grows into a second page (D); k = 8
LOOP = W.get("tiny").with_(batch=5, seq_lens=(64 * 12 - 3, 64 * 9 - 1, 64 * 5 + 1, 60,
                                              64 * 3 - 2), headroom_pages=1, seed=4001)
LOOP16 = W.get("tiny").with_(batch=3, page_size=16, budget_tokens=128,
                             seq_lens=(16 * 20 - 2, 16 * 7 - 1, 13), headroom_pages=1, seed=4002)
STEPS = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from sparse_paged_kv_gb300 import binding, build_lib
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    binding.load_library(build_lib.build())


def _bf16(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("wl,host_lengths", [(LOOP, False), (LOOP16, False), (LOOP, True)],
                         ids=["B64", "B16", "B64-host-lengths"])
def test_decode_loop_with_page_crossings(wl, host_lengths):
    import torch
    from sparse_paged_kv_gb300 import runtime
    inputs = W.generate(wl)
    w = inputs.workload
    B, Hk = w.page_size, w.n_kv_heads
    layer = runtime.LocksLayer.from_inputs(inputs)
    layer.build()
    k_host, v_host = inputs.k_cache.copy(), inputs.v_cache.copy()
    bt_host, sl_host = inputs.block_table.copy(), inputs.seq_lens.copy()
    # the engine's part, done once: a block for every page a sequence starts
    # within the loop, written into the block table before the loop
    free = sorted(set(range(w.num_blocks)) - set(int(x) for x in bt_host.ravel() if x >= 0))
    for b in range(w.batch):
        t = int(sl_host[b])
        for j in range(-(-t // B), -(-(t + STEPS) // B)):
            bt_host[b, j] = free.pop(0)
    layer.block_table.copy_(torch.from_numpy(bt_host).cuda())
    loop = runtime.DecodeLoop(layer, host_lengths=sl_host if host_lengths else None)
    rng = np.random.default_rng(4242)
    page_lse, page_share = layer.alloc_page_lse(), layer.alloc_page_share()
    crossings, scored_new = 0, 0
    built = set()
    for step in range(STEPS):
        kv = W.f32_to_bf16_bits(rng.standard_normal((2, w.batch, Hk, w.head_dim)).astype(np.float32))
        q = W.f32_to_bf16_bits(rng.standard_normal(inputs.q.shape).astype(np.float32))
        want_done = []
        for b in range(w.batch):                    # the host mirror, kept by the test
            t = int(sl_host[b])
            blk = int(bt_host[b, t // B])
            k_host[blk, :, t % B] = kv[0, b]
            v_host[blk, :, t % B] = kv[1, b]
            sl_host[b] = t + 1
            want_done.append(blk if (t + 1) % B == 0 else -1)
        layer.q.copy_(_bf16(torch, q))
        loop.step(_bf16(torch, kv[0]), _bf16(torch, kv[1]), page_lse=page_lse,
                  page_share=page_share)
        snap = P.gpu_snapshot(layer, page_lse, page_share)
        done = loop.completed[step & 1].cpu().numpy().tolist()
        assert done == want_done, (step, done, want_done)
        assert layer.seq_lens.cpu().numpy().tolist() == sl_host.tolist()
        crossings += sum(x >= 0 for x in done)
        cur = W.LocksInputs(workload=w, q=q, k_cache=k_host, v_cache=v_host,
                            block_table=bt_host, seq_lens=sl_host, carriers=inputs.carriers)
        rep = P.Report()
        for b in range(w.batch):
            for h in range(Hk):
                res = O.run_unit(q, k_host, v_host, bt_host, sl_host, Hk, w.rank,
                                 w.budget_tokens, b, h)
                P.compare_select(layer, snap, res, rep)
                P.compare_sparse_decode(layer, cur, snap, res, rep)
                scored_new += sum(int(bt_host[b, j]) in built for j in res.sel.cand)
        assert snap["status"] == 0, hex(snap["status"])
        rep.check()
        built |= {x for x in done if x >= 0}
    loop.finish()
    torch.cuda.synchronize()
    # the summaries built in the loop, against the oracle's
    rep = P.Report()
    for b in range(w.batch):
        for h in range(Hk):
            res = O.run_unit(q, k_host, v_host, bt_host, sl_host, Hk, w.rank, w.budget_tokens,
                             b, h)
            P.compare_build(layer, cur, res, rep)
    rep.check()
    assert np.array_equal(layer.k_cache.view(torch.int16).cpu().numpy().view(np.uint16), k_host)
    assert np.array_equal(layer.v_cache.view(torch.int16).cpu().numpy().view(np.uint16), v_host)
    assert crossings >= 3 and scored_new > 0, (crossings, scored_new)
