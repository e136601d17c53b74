"""The C-ABI library on the host: it builds, loads, exports every symbol the
header declares, and rejects bad arguments before launching anything (no GPU)."""
import ctypes
import os
import re

import pytest

from sparse_paged_kv_gb300 import binding as B
from sparse_paged_kv_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "locks.h")


@pytest.fixture(scope="module")
def lib():
    path = build_lib.build()
    return B.load_library(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(locks_[a-z_0-9]+)\s*\(", src)))


def cfg(**kw):
    base = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=64, rank=8,
                max_pages=64, num_blocks=200, summary_dtype=B.LOCKS_SUMMARY_F32)
    base.update(kw)
    return B.LocksConfig(**base)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert lib.locks_abi_version() == 1


def test_struct_layout_matches_header(lib):
    assert ctypes.sizeof(B.locks_cfg_t) == 9 * 4
    src = open(HEADER).read()
    body = re.search(r"typedef struct locks_cfg \{(.*?)\} locks_cfg_t;", src, re.S).group(1)
    fields = re.findall(r"int32_t\s+(\w+);", body)
    assert fields == [f[0] for f in B.locks_cfg_t._fields_]


def test_record_bytes(lib):
    assert B.summary_record_bytes(cfg()) == ((8 + 1) * 128 + 8 * 64) * 4 == 6656
    assert B.summary_record_bytes(cfg(summary_dtype=B.LOCKS_SUMMARY_BF16)) == 3328
    assert B.summary_record_bytes(cfg(rank=3)) == ((4 + 1) * 128 + 4 * 64) * 4
    assert B.summary_record_bytes(cfg(rank=15)) == ((16 + 1) * 128 + 16 * 64) * 4
    assert B.summary_record_bytes(cfg(head_dim=64)) == 0          # unsupported
    assert B.summary_record_bytes(cfg(page_size=16)) == ((8 + 1) * 128 + 8 * 16) * 4 == 5120
    assert B.summary_record_bytes(cfg(page_size=16, rank=15)) == ((16 + 1) * 128 + 16 * 16) * 4
    assert B.summary_record_bytes(cfg(page_size=32)) == 0
    assert B.summary_record_bytes(cfg(n_q_heads=6, n_kv_heads=2)) == 0   # G = 3
    for c in (cfg(), cfg(summary_dtype=B.LOCKS_SUMMARY_BF16), cfg(rank=15), cfg(head_dim=64)):
        assert lib.locks_summary_bytes(ctypes.byref(c.c())) == B.summary_record_bytes(c)


def test_workspace_sizes_grow_with_shape(lib):
    a = B.select_workspace_bytes(cfg(), 512)
    b = B.select_workspace_bytes(cfg(batch=4), 512)
    assert 0 < a < b
    s = B.decode_workspace_bytes(cfg(), 8)
    d = B.decode_workspace_bytes(cfg(), 64)
    assert 0 < s <= d
    assert B.decode_workspace_bytes(cfg(), -1) == 0
    assert 0 < B.select_workspace_bytes(cfg(page_size=16), 512)
    assert 0 < B.decode_workspace_bytes(cfg(page_size=16), 32)


FAKE = 0x10000   # never dereferenced: every call below returns before a launch


def _select(lib, c, budget=512, ws_bytes=1 << 30, **over):
    args = dict(q=FAKE, summ=FAKE, bt=FAKE, sl=FAKE, sel=FAKE, ws=FAKE)
    args.update(over)
    return lib.locks_select(ctypes.byref(c.c()), args["q"], args["summ"], args["bt"], args["sl"],
                            budget, args["sel"], None, None, args["ws"], ws_bytes, None, None)


def test_headline_shape_sizes(lib):
    """The 1M-token layer (one sequence, 32/8 heads, 16384 pages): the select
    workspace holds s_hat for every (unit, page, head) plus the partials, the
    slice winners and the tickets, a few MB; the quantised record is 1456
    bytes at r = 8, B = 64."""
    c = cfg(batch=1, n_q_heads=32, n_kv_heads=8, max_pages=16384, num_blocks=16384 + 8)
    ws = B.select_workspace_bytes(c, 2048)
    assert 8 * 16384 * 4 * 4 <= ws < 16 * 2 ** 20
    assert B.decode_workspace_bytes(c, 32) > 0
    assert B.summary_record_bytes(cfg(summary_dtype=B.LOCKS_SUMMARY_I4)) == 1456


def test_select_validation(lib):
    assert _select(lib, cfg(), budget=64) == B.LOCKS_ERR_INVALID_ARG        # k = 1
    assert _select(lib, cfg(), budget=0) == B.LOCKS_ERR_INVALID_ARG
    assert _select(lib, cfg(), ws_bytes=16) == B.LOCKS_ERR_WORKSPACE
    assert _select(lib, cfg(), q=None) == B.LOCKS_ERR_INVALID_ARG
    assert _select(lib, cfg(head_dim=96)) == B.LOCKS_ERR_UNSUPPORTED
    assert _select(lib, cfg(page_size=32)) == B.LOCKS_ERR_UNSUPPORTED     # B in {64, 16}
    assert _select(lib, cfg(rank=17)) == B.LOCKS_ERR_UNSUPPORTED
    assert _select(lib, cfg(n_q_heads=7)) == B.LOCKS_ERR_INVALID_ARG
    assert _select(lib, cfg(summary_dtype=5)) == B.LOCKS_ERR_INVALID_ARG
    assert _select(lib, cfg(), budget=64 * 300) == B.LOCKS_ERR_UNSUPPORTED   # k > 256
    assert _select(lib, cfg(batch=0)) == B.LOCKS_OK                       # nothing to do
    assert lib.locks_select(None, FAKE, FAKE, FAKE, FAKE, 512, FAKE, None, None, FAKE, 1 << 30,
                            None, None) == B.LOCKS_ERR_INVALID_ARG


def test_supported_shape_limits(lib):
    """The header's shape limits: G a power of two up to 8, page ids below
    2^24, record indices below 2^31; a negative batch is invalid."""
    assert _select(lib, cfg(n_q_heads=12, n_kv_heads=4)) == B.LOCKS_ERR_UNSUPPORTED   # G = 3
    assert _select(lib, cfg(n_q_heads=32, n_kv_heads=2)) == B.LOCKS_ERR_UNSUPPORTED   # G = 16
    assert _select(lib, cfg(max_pages=1 << 24)) == B.LOCKS_ERR_UNSUPPORTED
    assert _select(lib, cfg(num_blocks=1 << 30, n_kv_heads=2)) == B.LOCKS_ERR_UNSUPPORTED
    assert _select(lib, cfg(batch=-1)) == B.LOCKS_ERR_INVALID_ARG
    for c in (cfg(max_pages=1 << 24), cfg(n_q_heads=12, n_kv_heads=4), cfg(batch=-1)):
        assert lib.locks_summary_record_bytes(ctypes.byref(c.c())) == 0
        assert lib.locks_select_workspace_bytes(ctypes.byref(c.c()), 512) == 0
        assert lib.locks_decode_workspace_bytes(ctypes.byref(c.c()), 8) == 0
    # just inside the limits
    assert lib.locks_summary_record_bytes(ctypes.byref(cfg(max_pages=(1 << 24) - 1).c())) > 0
    assert lib.locks_summary_record_bytes(ctypes.byref(cfg(n_q_heads=16, n_kv_heads=2).c())) > 0


def test_decode_rejects_unaligned_pools(lib):
    """The decode reads K and V through tensor maps, whose base must be
    16-byte aligned; a misaligned pool is refused before any launch."""
    c = cfg()
    ws = B.decode_workspace_bytes(c, 8)
    odd = FAKE + 8
    assert lib.locks_sparse_decode(ctypes.byref(c.c()), FAKE, odd, FAKE, FAKE, FAKE, FAKE, 8,
                                   FAKE, None, FAKE, ws, None, None) == B.LOCKS_ERR_INVALID_ARG
    assert lib.locks_dense_decode(ctypes.byref(c.c()), FAKE, FAKE, odd, FAKE, FAKE, FAKE, None,
                                  FAKE, B.decode_workspace_bytes(c, c.max_pages), None,
                                  None) == B.LOCKS_ERR_INVALID_ARG


def test_decode_and_build_validation(lib):
    c = cfg()
    ws = B.decode_workspace_bytes(c, 8)
    assert lib.locks_sparse_decode(ctypes.byref(c.c()), FAKE, FAKE, FAKE, FAKE, FAKE, None, 8,
                                   FAKE, None, FAKE, ws, None, None) == B.LOCKS_ERR_INVALID_ARG
    assert lib.locks_sparse_decode(ctypes.byref(c.c()), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8,
                                   FAKE, None, FAKE, ws - 1, None, None) == B.LOCKS_ERR_WORKSPACE
    assert lib.locks_dense_decode(ctypes.byref(c.c()), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                  FAKE, 16, None, None) == B.LOCKS_ERR_WORKSPACE
    assert lib.locks_dense_decode(ctypes.byref(cfg(batch=0).c()), FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, None, FAKE, 0, None, None) == B.LOCKS_OK
    assert lib.locks_build_summaries(ctypes.byref(c.c()), FAKE, FAKE, -1, FAKE, None, None, 0,
                                     None) == B.LOCKS_ERR_INVALID_ARG
    assert lib.locks_build_summaries(ctypes.byref(c.c()), FAKE, FAKE, 0, FAKE, None, None, 0,
                                     None) == B.LOCKS_OK
    assert lib.locks_build_summaries(ctypes.byref(c.c()), None, FAKE, 4, FAKE, None, None, 0,
                                     None) == B.LOCKS_ERR_INVALID_ARG


def test_append_and_completed_build_validation(lib):
    """locks_append_kv moves rows as 16-byte words: null or misaligned
    pointers are refused before any launch; an empty batch does nothing.
    locks_build_completed validates like locks_build_summaries."""
    c = cfg()
    cc = ctypes.byref(c.c())
    assert lib.locks_append_kv(cc, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                               None) == B.LOCKS_ERR_INVALID_ARG
    assert lib.locks_append_kv(cc, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                               None) == B.LOCKS_ERR_INVALID_ARG
    for i in range(4):
        args = [FAKE] * 4
        args[i] = FAKE + 8
        assert lib.locks_append_kv(cc, *args, FAKE, FAKE, None, None,
                                   None) == B.LOCKS_ERR_INVALID_ARG, i
    assert lib.locks_append_kv(ctypes.byref(cfg(batch=0).c()), FAKE, FAKE, FAKE, FAKE, FAKE,
                               FAKE, None, None, None) == B.LOCKS_OK
    assert lib.locks_append_kv(ctypes.byref(cfg(page_size=32).c()), FAKE, FAKE, FAKE, FAKE, FAKE,
                               FAKE, None, None, None) == B.LOCKS_ERR_UNSUPPORTED
    assert lib.locks_build_completed(cc, FAKE, FAKE, -1, FAKE, None, None, 0,
                                     None) == B.LOCKS_ERR_INVALID_ARG
    assert lib.locks_build_completed(cc, FAKE, FAKE, 0, FAKE, None, None, 0, None) == B.LOCKS_OK
    assert lib.locks_build_completed(cc, FAKE, None, 4, FAKE, None, None, 0,
                                     None) == B.LOCKS_ERR_INVALID_ARG


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, 99):
        assert isinstance(lib.locks_status_string(code), bytes)


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(B.LocksLibraryMissing):
        B.load_library(str(tmp_path / "missing.so"))


def test_unpack_records_layout():
    import numpy as np
    c = cfg(rank=8)
    R, d, Bp = 8, 128, 64
    mu = np.arange(d, dtype=np.float32)
    V = np.random.default_rng(0).standard_normal((d, R)).astype(np.float32)
    C = np.random.default_rng(1).standard_normal((Bp, R)).astype(np.float32)
    W = np.concatenate([mu[None], V.T], axis=0).reshape(-1)
    C4 = C.reshape(Bp, R // 4, 4).transpose(1, 0, 2).reshape(-1)
    raw = np.concatenate([W, C4]).view(np.uint8)
    m2, V2, C2 = B.unpack_records(raw[None], c)
    assert np.array_equal(m2[0], mu) and np.array_equal(V2[0], V) and np.array_equal(C2[0], C)


def test_unpack_i4_layout(lib):
    """The quantised record layout documented in locks.h, packed here by hand
    from its description, unpacks to the codes and scales it was packed from."""
    import numpy as np
    for rank, Bp in ((8, 64), (16, 16), (3, 64)):
        c = cfg(summary_dtype=B.LOCKS_SUMMARY_I4, rank=rank, page_size=Bp)
        R, d = c.rank_cap, c.head_dim
        KK = (R + 7) // 8
        nbytes = B.summary_record_bytes(c)
        hdr = ((R + 1) * 4 + 15) // 16 * 16
        assert nbytes == hdr + 64 * R + 128 + 8 * Bp * KK + 4 * Bp
        rng = np.random.default_rng(3 + rank)
        v = rng.integers(-7, 8, (d, R))
        mu = rng.integers(-127, 128, d)
        cc = rng.integers(-127, 128, (Bp, R))
        vs = rng.random(R).astype(np.float32)
        cs = rng.random(Bp).astype(np.float32)
        rec = np.zeros(nbytes, np.uint8)
        rec[:4 * R] = vs.view(np.uint8)
        rec[4 * R:4 * R + 4] = np.float32(0.25).reshape(1).view(np.uint8)
        words = np.zeros((R, 4, 4), np.uint32)
        for k in range(R):
            for t in range(4):
                for j in range(4):
                    w = 0
                    for h in range(2):                  # k-step 2j + h
                        c0 = 16 * (2 * j + h) + 2 * t
                        w |= int(v[c0, k] + 8) << (4 * (2 * h))
                        w |= int(v[c0 + 1, k] + 8) << (4 * (2 * h + 4))
                        w |= int(v[c0 + 8, k] + 8) << (4 * (2 * h + 1))
                        w |= int(v[c0 + 9, k] + 8) << (4 * (2 * h + 5))
                    words[k, t, j] = w
        rec[hdr:hdr + 64 * R] = words.reshape(-1).view(np.uint8)
        for l in range(32):
            g, t = l >> 2, l & 3
            for e, off in enumerate((0, 1, 8, 9)):
                rec[hdr + 64 * R + 4 * l + e] = mu[16 * g + 2 * t + off] + 128
        base = hdr + 64 * R + 128
        for m in range(Bp // 16):
            for kk in range(KK):
                for l in range(32):
                    g, t = l >> 2, l & 3
                    for e, (di, dk) in enumerate(((0, 0), (0, 1), (8, 0), (8, 1))):
                        k = 8 * kk + 2 * t + dk
                        val = cc[16 * m + g + di, k] if k < R else 0
                        rec[base + ((m * KK + kk) * 32 + l) * 4 + e] = val + 128
        rec[base + 8 * Bp * KK:] = cs.view(np.uint8)
        mu_c, mu_s, v_c, v_s, c_c, c_s = B.unpack_i4(rec[None], c)
        assert np.array_equal(mu_c[0], mu) and float(mu_s[0]) == 0.25
        assert np.array_equal(v_c[0], v) and np.array_equal(v_s[0], vs)
        assert np.array_equal(c_c[0], cc) and np.array_equal(c_s[0], cs)
        m_, V, C = B.unpack_records(rec[None], c)
        assert np.allclose(V[0], (v * vs[None, :])[:, :rank])
        assert np.allclose(C[0], (cc * cs[:, None])[:, :rank])
        assert np.allclose(m_[0], mu * 0.25)
