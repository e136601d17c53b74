"""The seeded input generator: determinism, layout and the key recipe (no GPU)."""
import math

import numpy as np

import workloads as W


def test_deterministic_and_layout():
    w = W.get("tiny")
    a, b = W.generate(w), W.generate(w, threads=1)
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.v_cache, b.v_cache),
                 (a.block_table, b.block_table)):
        assert np.array_equal(x, y)
    assert a.k_cache.shape == (w.num_blocks, w.n_kv_heads, w.page_size, w.head_dim)
    assert a.q.shape == (w.batch, w.n_q_heads, w.head_dim)
    n = w.context // w.page_size
    row = a.block_table[0, :n]
    assert len(set(row.tolist())) == n and row.min() >= 0 and row.max() < w.num_blocks
    # unused blocks are NaN
    unused = sorted(set(range(w.num_blocks)) - set(row.tolist()))
    assert len(unused) == w.spare_blocks
    assert np.all(a.k_cache[unused] == 0x7FC0)
    assert [len(c) for c in a.carriers[0]] == [3, 3]
    for c in a.carriers[0]:
        assert c.min() >= 1 and c.max() <= n - 2


def test_ragged_tail_is_nan_and_table_padded():
    w = W.get("tiny").with_(batch=2, seq_lens=(4096 + 37, 200))
    x = W.generate(w)
    B = w.page_size
    n0 = math.ceil((4096 + 37) / B)
    tail = x.block_table[0, n0 - 1]
    assert np.all(x.k_cache[tail, :, 37:] == 0x7FC0)
    assert not np.any(x.k_cache[tail, :, :37] == 0x7FC0)
    assert np.all(x.block_table[1, math.ceil(200 / B):] == -1)
    assert x.seq_lens.tolist() == [4096 + 37, 200]


def test_key_recipe_is_page_local_low_rank():
    """Rank-8-plus-noise pages: rank 8 captures almost all centred energy, and
    carrier pages are shifted along the group query direction."""
    w = W.get("tiny")
    x = W.generate(w)
    keys = W.bf16_bits_to_f32(x.k_cache[x.block_table[0, 10], 0]).astype(np.float64)
    D = keys - keys.mean(axis=0)
    sv = np.linalg.svd(D, compute_uv=False) ** 2
    assert sv[:8].sum() / sv.sum() > 0.97
    assert np.std(keys) > 0.3
    q = W.bf16_bits_to_f32(x.q[0, :4]).astype(np.float64).sum(axis=0)
    qh = q / np.linalg.norm(q)
    car = x.carriers[0][0][0]
    kc = W.bf16_bits_to_f32(x.k_cache[x.block_table[0, car], 0]).astype(np.float64)
    assert kc.mean(axis=0) @ qh > 0.4           # shifted by 0.5 along q_hat


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], dtype=np.float32)
    bits = W.f32_to_bf16_bits(v)
    back = W.bf16_bits_to_f32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0                        # tie -> even
    assert back[2] == 1.0 + 4 * 2 ** -8          # tie -> even (up)
    assert back[3] == -2.5


def test_unit_subset_matches_full_workload():
    """Generating only some (sequence, KV head) units gives those units the
    bytes they have in the full workload and leaves every other page NaN."""
    w = W.get("tiny")
    full = W.generate(w)
    part = W.generate(w, units=[(0, 1)])
    blk = full.block_table[0, :w.max_pages]
    assert np.array_equal(full.k_cache[blk, 1], part.k_cache[blk, 1])
    assert np.array_equal(full.v_cache[blk, 1], part.v_cache[blk, 1])
    assert np.array_equal(full.q, part.q)
    assert np.array_equal(full.carriers[0][1], part.carriers[0][1])
    assert (part.k_cache[blk, 0] == 0x7FC0).all() and (part.v_cache[blk, 0] == 0x7FC0).all()
