"""locks_select_noalloc, the selection entry point for callers that cannot
allocate device memory (a pool that owns the whole GPU, a host framework that
forbids cudaMalloc on the decode path), checked through the C ABI against
locks_select on the same inputs, on two calls in a row.

Kept in its own file, collected last, so a failure here comes after every
other test has run; it also passes alone in a fresh process (its first call
does the per-device set-up)."""
import ctypes

import numpy as np
import pytest

import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


def _layer(w):
    from sparse_paged_kv_gb300 import runtime
    inputs = W.generate(w)
    layer = runtime.LocksLayer.from_inputs(inputs)
    layer.build()
    return layer


def _noalloc(lib, layer, sel, lse, share, status):
    import torch
    return lib.locks_select_noalloc(
        ctypes.byref(layer.cfg.c()), layer.q.data_ptr(), layer.summaries.data_ptr(),
        layer.block_table.data_ptr(), layer.seq_lens.data_ptr(), layer.budget, sel.data_ptr(),
        lse.data_ptr(), share.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_select_on_two_calls_in_a_row():
    import torch
    from sparse_paged_kv_gb300 import binding as B
    from sparse_paged_kv_gb300 import build_lib
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = B.load_library(build_lib.build())
    tiny = W.get("tiny")
    cases = [tiny.with_(context=64 * 300, global_rank=16, carrier_count=None, carrier_frac=0.01,
                        budget_tokens=2048, seed=3101),
             tiny.with_(batch=3, seq_lens=(4096 + 37, 64 * 9, 200), seed=3102)]
    for w in cases:
        layer = _layer(w)
        ref_lse, ref_share = layer.alloc_page_lse(), layer.alloc_page_share()
        layer.select(page_lse=ref_lse, page_share=ref_share)
        torch.cuda.synchronize()
        ref_sel = layer.selected.cpu().numpy()
        sel = torch.full_like(layer.selected, -7)
        lse, share = layer.alloc_page_lse(), layer.alloc_page_share()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, layer, sel, lse, share, status) == B.LOCKS_OK
        torch.cuda.synchronize()
        assert int(status.cpu()[0]) == 0
        assert np.array_equal(sel.cpu().numpy(), ref_sel)
        a, b = lse.cpu().numpy(), ref_lse.cpu().numpy()
        assert np.array_equal(np.isnan(a), np.isnan(b))
        m = ~np.isnan(b)
        assert np.abs(a[m] - b[m]).max() <= P.LSE_TOL
        a, b = share.cpu().numpy(), ref_share.cpu().numpy()
        m = ~np.isnan(b)
        assert np.abs(a[m] - b[m]).max() <= P.TIE_TOL


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from sparse_paged_kv_gb300 import binding as B
    from sparse_paged_kv_gb300 import build_lib
    lib = B.load_library(build_lib.build())
    big = B.LocksConfig(batch=64, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=64, rank=8,
                        max_pages=16384, num_blocks=1 << 20)
    fake = 0x10000    # never dereferenced: the size check comes first
    rc = lib.locks_select_noalloc(ctypes.byref(big.c()), fake, fake, fake, fake, 2048, fake,
                                  None, None, None, None)
    assert rc == B.LOCKS_ERR_WORKSPACE
