"""Seeded synthetic inputs for a Locks decode step.

The generator writes the arrays both sides consume -- the query batch, the
paged bf16 key/value pools, the block table and the sequence lengths -- as
plain NumPy arrays (bf16 held as its uint16 bit pattern).  It draws every
number from NumPy's PCG64 in float64, so the same seed gives the same bytes on
every platform, and rounds each value to bf16 once (round to nearest even).

Layout of the pools: ``[num_blocks][n_kv_heads][page_size][head_dim]``; the
logical page ``j`` of sequence ``b`` lives in physical block
``block_table[b, j]``, a seeded random permutation of the pool, so page
gathering is real.  Slots of a partially filled tail page, unused blocks and
unused block-table entries hold NaN keys/values and ``-1`` ids, so a reader
that touches anything outside the valid tokens is caught.

Key recipe per (sequence, KV head), page by page:
  k = A_p G_p  (A_p: B x 8, G_p: 8 x d, entries N(0,1)/sqrt(8))
    + noise * N(0,1)
    + Z_t H    (shared global rank-16 part, Z: T x 16, H: 16 x d, N(0,1)/4)
    + 0.5 * q_hat on every key of a carrier page,
where q_hat is the unit vector of the sum of the GQA group's queries.  With
``carrier_token`` only one seeded token of each carrier page gets the shift
(``carrier_bias`` * q_hat), so the page's centroid barely moves.  Values and
queries are N(0,1).

Nothing in this module computes any part of the Locks method.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

from .configs import LocksWorkload

BF16_NAN = np.uint16(0x7FC0)
CHUNK_PAGES = 128            # pages per independent RNG stream inside a unit


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class LocksInputs:
    workload: LocksWorkload
    q: np.ndarray            # uint16 [batch][n_q_heads][head_dim]
    k_cache: np.ndarray      # uint16 [num_blocks][n_kv_heads][page_size][head_dim]
    v_cache: np.ndarray      # uint16 same shape
    block_table: np.ndarray  # int32 [batch][max_pages]
    seq_lens: np.ndarray     # int32 [batch]
    carriers: List[List[np.ndarray]]   # carrier logical pages per [b][h_kv]

    @property
    def nbytes(self) -> int:
        return self.q.nbytes + self.k_cache.nbytes + self.v_cache.nbytes


def _seed(w: LocksWorkload, *key: int) -> np.random.SeedSequence:
    return np.random.SeedSequence(entropy=w.seed, spawn_key=tuple(int(k) for k in key))


def _candidate_pages(n_pages: int, seq_len: int, page_size: int) -> np.ndarray:
    """Complete pages other than the first and the last page."""
    n_complete = seq_len // page_size
    hi = min(n_pages - 1, n_complete)        # exclusive upper bound
    return np.arange(1, hi, dtype=np.int64) if hi > 1 else np.zeros(0, dtype=np.int64)


def _gen_unit(w: LocksWorkload, b: int, h: int, seq_len: int, q_hat: np.ndarray,
              k_out: np.ndarray, v_out: np.ndarray, blocks: np.ndarray) -> np.ndarray:
    """Fill keys/values of one (sequence, KV head); return its carrier pages."""
    B, d = w.page_size, w.head_dim
    n_pages = math.ceil(seq_len / B)
    unit = b * w.n_kv_heads + h
    rng = np.random.Generator(np.random.PCG64(_seed(w, 1, unit, 0)))

    cand = _candidate_pages(n_pages, seq_len, B)
    if w.carrier_count is not None:
        n_car = min(len(cand), w.carrier_count)
    else:
        n_car = min(len(cand), math.ceil(w.carrier_frac * len(cand)))
    carriers = np.sort(rng.choice(cand, size=n_car, replace=False)) if n_car else np.zeros(0, np.int64)
    is_carrier = np.zeros(n_pages, dtype=bool)
    is_carrier[carriers] = True
    token_of = None
    if w.carrier_token and n_car:               # the one shifted token of each carrier page
        token_of = np.full(n_pages, -1, dtype=np.int64)
        token_of[carriers] = rng.integers(0, B, size=n_car)

    gr = w.global_rank
    H = rng.standard_normal((gr, d)) / math.sqrt(gr) if gr else None
    lr = w.local_rank

    for c0 in range(0, n_pages, CHUNK_PAGES):
        c1 = min(n_pages, c0 + CHUNK_PAGES)
        n = c1 - c0
        crng = np.random.Generator(np.random.PCG64(_seed(w, 1, unit, 1 + c0 // CHUNK_PAGES)))
        A = crng.standard_normal((n, B, lr)) / math.sqrt(lr)
        G = crng.standard_normal((n, lr, d)) / math.sqrt(lr)
        keys = np.matmul(A, G)
        keys += w.noise * crng.standard_normal((n, B, d))
        if gr:
            Z = crng.standard_normal((n * B, gr)) / math.sqrt(gr)
            keys += (Z @ H).reshape(n, B, d)
        car = is_carrier[c0:c1]
        if car.any():
            if token_of is None:
                keys[car] += w.carrier_bias * q_hat
            else:
                for p in np.nonzero(car)[0]:
                    keys[p, token_of[c0 + p]] += w.carrier_bias * q_hat
        vals = crng.standard_normal((n, B, d))
        kb = f32_to_bf16_bits(keys)
        vb = f32_to_bf16_bits(vals)
        # invalid slots of a partial tail page stay NaN
        last_valid = seq_len - (n_pages - 1) * B
        if c1 == n_pages and last_valid < B:
            kb[-1, last_valid:] = BF16_NAN
            vb[-1, last_valid:] = BF16_NAN
        phys = blocks[c0:c1]
        k_out[phys, h] = kb
        v_out[phys, h] = vb
    return carriers


def generate(w: LocksWorkload, threads: Optional[int] = None,
             units: Optional[Sequence[Tuple[int, int]]] = None) -> LocksInputs:
    """Generate the inputs of workload ``w`` (deterministic in ``w.seed``).

    ``units`` limits the keys and values filled to the listed (sequence, KV
    head) pairs; every other page of the pools stays NaN.  Each unit draws
    from its own streams, so a listed unit gets exactly the bytes it has in
    the full workload."""
    assert w.n_q_heads % w.n_kv_heads == 0
    lens = w.lengths()
    B, d, Hk, Hq = w.page_size, w.head_dim, w.n_kv_heads, w.n_q_heads
    G = w.group
    maxp = w.max_pages

    q_rng = np.random.Generator(np.random.PCG64(_seed(w, 0, 0)))
    q = f32_to_bf16_bits(q_rng.standard_normal((w.batch, Hq, d)))
    q32 = bf16_bits_to_f32(q).astype(np.float64)

    p_rng = np.random.Generator(np.random.PCG64(_seed(w, 0, 1)))
    perm = p_rng.permutation(w.num_blocks).astype(np.int32)
    block_table = np.full((w.batch, maxp), -1, dtype=np.int32)
    for b, t in enumerate(lens):
        n = math.ceil(t / B)
        block_table[b, :n] = perm[b * maxp: b * maxp + n]

    k_cache = np.full((w.num_blocks, Hk, B, d), BF16_NAN, dtype=np.uint16)
    v_cache = np.full((w.num_blocks, Hk, B, d), BF16_NAN, dtype=np.uint16)

    jobs = []
    want = None if units is None else {(int(b), int(h)) for b, h in units}
    for b, t in enumerate(lens):
        if t <= 0:
            continue
        n = math.ceil(t / B)
        for h in range(Hk):
            if want is not None and (b, h) not in want:
                continue
            s = q32[b, h * G:(h + 1) * G].sum(axis=0)
            q_hat = s / max(np.linalg.norm(s), 1e-30)
            jobs.append((b, h, t, q_hat, block_table[b, :n].astype(np.int64)))

    carriers: List[List[np.ndarray]] = [[np.zeros(0, np.int64)] * Hk for _ in range(w.batch)]
    nthreads = threads or min(len(jobs) or 1, os.cpu_count() or 1)

    def run(job):
        b, h, t, q_hat, blocks = job
        return b, h, _gen_unit(w, b, h, t, q_hat, k_cache, v_cache, blocks)

    if nthreads <= 1 or len(jobs) <= 1:
        results = [run(j) for j in jobs]
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            results = list(ex.map(run, jobs))
    for b, h, car in results:
        carriers[b][h] = car

    return LocksInputs(workload=w, q=q, k_cache=k_cache, v_cache=v_cache,
                       block_table=block_table,
                       seq_lens=np.asarray(lens, dtype=np.int32), carriers=carriers)
