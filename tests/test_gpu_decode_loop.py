"""A decode loop through the library, as an engine would drive it: every step
appends one token per sequence to the paged cache (allocating a block when a
sequence starts a new page), builds the summary of each page the step
completes (section 4: one build per finalised page, off the critical path),
then selects and decodes.  Every step is checked against the oracle on the
cache as it stands, so page crossings, the moving incomplete tail page and the
incrementally built summaries are all exercised."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

# lengths chosen so that within three steps: a tail page completes (A, B),
# a sequence starts a new page (B), one stays inside its page (C), and a
# single-page sequence grows (D); k = 8
LOOP = W.get("tiny").with_(batch=4, seq_lens=(64 * 12 - 3, 64 * 9 - 1, 64 * 5 + 1, 60),
                           seed=4001)
STEPS = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    from sparse_paged_kv_gb300 import binding, build_lib
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    binding.load_library(build_lib.build())


def test_decode_loop_with_page_crossings():
    import torch
    from sparse_paged_kv_gb300 import runtime
    inputs = W.generate(LOOP)
    w = inputs.workload
    B, Hk = w.page_size, w.n_kv_heads
    layer = runtime.LocksLayer.from_inputs(inputs)
    layer.build()
    k_host, v_host = inputs.k_cache.copy(), inputs.v_cache.copy()
    bt_host, sl_host = inputs.block_table.copy(), inputs.seq_lens.copy()
    free = sorted(set(range(w.num_blocks)) - set(int(x) for x in bt_host.ravel() if x >= 0))
    rng = np.random.default_rng(4242)
    page_lse, page_share = layer.alloc_page_lse(), layer.alloc_page_share()
    crossings = 0
    for step in range(STEPS):
        completed = []
        for b in range(w.batch):
            t = int(sl_host[b])
            j, slot = t // B, t % B
            if slot == 0:                               # a new page: allocate a block
                assert j < w.max_pages
                bt_host[b, j] = free.pop(0)
            blk = int(bt_host[b, j])
            kv = W.f32_to_bf16_bits(rng.standard_normal((2, Hk, w.head_dim)).astype(np.float32))
            k_host[blk, :, slot] = kv[0]
            v_host[blk, :, slot] = kv[1]
            sl_host[b] = t + 1
            if (t + 1) % B == 0:
                completed.append(blk)
        q = W.f32_to_bf16_bits(rng.standard_normal(inputs.q.shape).astype(np.float32))
        # the device copies of what changed
        layer.k_cache.copy_(torch.from_numpy(k_host.view(np.int16)).view(torch.bfloat16).cuda())
        layer.v_cache.copy_(torch.from_numpy(v_host.view(np.int16)).view(torch.bfloat16).cuda())
        layer.block_table.copy_(torch.from_numpy(bt_host).cuda())
        layer.seq_lens.copy_(torch.from_numpy(sl_host).cuda())
        layer.q.copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda())
        if completed:
            layer.build(torch.tensor(completed, dtype=torch.int32, device="cuda"))
            crossings += len(completed)
        layer.select(page_lse=page_lse, page_share=page_share)
        layer.sparse_decode()
        snap = P.gpu_snapshot(layer, page_lse, page_share)
        rep = P.Report()
        for b in range(w.batch):
            for h in range(Hk):
                res = O.run_unit(q, k_host, v_host, bt_host, sl_host, Hk, w.rank,
                                 w.budget_tokens, b, h)
                P.compare_select(layer, snap, res, rep)
                cur = W.LocksInputs(workload=w, q=q, k_cache=k_host, v_cache=v_host,
                                    block_table=bt_host, seq_lens=sl_host,
                                    carriers=inputs.carriers)
                P.compare_sparse_decode(layer, cur, snap, res, rep)
        assert snap["status"] == 0, hex(snap["status"])
        rep.check()
    assert crossings >= 2
