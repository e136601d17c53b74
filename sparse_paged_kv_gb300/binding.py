"""Thin Python binding of libsparse_paged_kv (include/locks.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of the shared library.  Device buffers are torch CUDA tensors (or raw
device pointers given as ints); streams default to torch's current stream.
The functions carry the C names.  Importing this module does not need a GPU;
calling a kernel entry point does, and a missing library raises
``LocksLibraryMissing`` -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional, Tuple

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libsparse_paged_kv.so")

LOCKS_OK = 0
LOCKS_ERR_INVALID_ARG = -1
LOCKS_ERR_UNSUPPORTED = -2
LOCKS_ERR_WORKSPACE = -3
LOCKS_ERR_CUDA = -4

LOCKS_DEV_BAD_BLOCK_ID = 0x1
LOCKS_DEV_WAIT_TIMEOUT = 0x2
LOCKS_DEV_NOT_CONVERGED = 0x4
LOCKS_DEV_BAD_PAGE_ID = 0x8
LOCKS_DEV_BAD_SEQ_LEN = 0x10

LOCKS_SUMMARY_F32 = 0
LOCKS_SUMMARY_BF16 = 1
LOCKS_SUMMARY_I4 = 2


class LocksLibraryMissing(RuntimeError):
    pass


class LocksError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} returned {code} ({msg})")
        self.code = code


class locks_cfg_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "n_q_heads", "n_kv_heads", "head_dim", "page_size", "rank", "max_pages",
        "num_blocks", "summary_dtype")]


@dataclass(frozen=True)
class LocksConfig:
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    rank: int
    max_pages: int
    num_blocks: int
    summary_dtype: int = LOCKS_SUMMARY_F32

    def c(self) -> locks_cfg_t:
        return locks_cfg_t(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim,
                           self.page_size, self.rank, self.max_pages, self.num_blocks,
                           self.summary_dtype)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def rank_cap(self) -> int:
        return 4 if self.rank <= 4 else (8 if self.rank <= 8 else 16)

    def page_budget(self, budget_tokens: int) -> int:
        return -(-budget_tokens // self.page_size)

    @staticmethod
    def from_workload(w, summary_dtype: int = LOCKS_SUMMARY_F32) -> "LocksConfig":
        return LocksConfig(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                           head_dim=w.head_dim, page_size=w.page_size, rank=w.rank,
                           max_pages=w.max_pages, num_blocks=w.num_blocks,
                           summary_dtype=summary_dtype)


_lib = None

_P = ctypes.c_void_p
_SIGS = {
    "locks_summary_record_bytes": (ctypes.c_size_t, [ctypes.POINTER(locks_cfg_t)]),
    "locks_summary_bytes": (ctypes.c_size_t, [ctypes.POINTER(locks_cfg_t)]),
    "locks_select_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(locks_cfg_t), ctypes.c_int32]),
    "locks_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(locks_cfg_t), ctypes.c_int32]),
    "locks_build_summaries": (ctypes.c_int, [ctypes.POINTER(locks_cfg_t), _P, _P, ctypes.c_int32,
                                             _P, _P, _P, ctypes.c_int32, _P]),
    "locks_select": (ctypes.c_int, [ctypes.POINTER(locks_cfg_t), _P, _P, _P, _P, ctypes.c_int32,
                                    _P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "locks_sparse_decode": (ctypes.c_int, [ctypes.POINTER(locks_cfg_t), _P, _P, _P, _P, _P, _P,
                                           ctypes.c_int32, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "locks_dense_decode": (ctypes.c_int, [ctypes.POINTER(locks_cfg_t), _P, _P, _P, _P, _P, _P, _P,
                                          _P, ctypes.c_size_t, _P, _P]),
    "locks_select_noalloc": (ctypes.c_int, [ctypes.POINTER(locks_cfg_t), _P, _P, _P, _P,
                                            ctypes.c_int32, _P, _P, _P, _P, _P]),
    "locks_append_kv": (ctypes.c_int, [ctypes.POINTER(locks_cfg_t), _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P]),
    "locks_build_completed": (ctypes.c_int, [ctypes.POINTER(locks_cfg_t), _P, _P, ctypes.c_int32,
                                             _P, _P, _P, ctypes.c_int32, _P]),
    "locks_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "locks_abi_version": (ctypes.c_int, []),
}


def load_library(path: Optional[str] = None):
    """Load (once) and return the ctypes handle of libsparse_paged_kv."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise LocksLibraryMissing(
            f"{p} not found: build it with `python -m sparse_paged_kv_gb300.build_lib` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("device tensor expected")
    if not x.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int):
    if rc != LOCKS_OK:
        raise LocksError(fn, rc, load_library().locks_status_string(rc).decode())


def summary_record_bytes(cfg: LocksConfig) -> int:
    return int(load_library().locks_summary_record_bytes(ctypes.byref(cfg.c())))


def select_workspace_bytes(cfg: LocksConfig, budget_tokens: int) -> int:
    return int(load_library().locks_select_workspace_bytes(ctypes.byref(cfg.c()), budget_tokens))


def decode_workspace_bytes(cfg: LocksConfig, n_pages: int) -> int:
    return int(load_library().locks_decode_workspace_bytes(ctypes.byref(cfg.c()), n_pages))


# --------------------------------------------------------------------------
# entry points (C names)
# --------------------------------------------------------------------------
def locks_build_summaries(cfg: LocksConfig, k_cache, block_ids, summaries, tail_energy=None,
                          status=None, max_sweeps: int = 0, stream=None) -> None:
    n_blocks = block_ids.numel() if not isinstance(block_ids, int) else None
    if n_blocks is None:
        raise ValueError("block_ids must be a tensor")
    rc = load_library().locks_build_summaries(
        ctypes.byref(cfg.c()), _ptr(k_cache), _ptr(block_ids), int(n_blocks), _ptr(summaries),
        _ptr(tail_energy), _ptr(status), int(max_sweeps), _stream(stream))
    _check("locks_build_summaries", rc)


def locks_append_kv(cfg: LocksConfig, k_new, v_new, k_cache, v_cache, block_table, seq_lens,
                    completed=None, status=None, stream=None) -> None:
    rc = load_library().locks_append_kv(
        ctypes.byref(cfg.c()), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), _ptr(seq_lens), _ptr(completed), _ptr(status), _stream(stream))
    _check("locks_append_kv", rc)


def locks_build_completed(cfg: LocksConfig, k_cache, completed, summaries, tail_energy=None,
                          status=None, max_sweeps: int = 0, stream=None) -> None:
    rc = load_library().locks_build_completed(
        ctypes.byref(cfg.c()), _ptr(k_cache), _ptr(completed), int(completed.numel()),
        _ptr(summaries), _ptr(tail_energy), _ptr(status), int(max_sweeps), _stream(stream))
    _check("locks_build_completed", rc)


def locks_select(cfg: LocksConfig, q, summaries, block_table, seq_lens, budget_tokens: int,
                 selected, workspace, page_lse=None, page_share=None, status=None,
                 workspace_bytes: Optional[int] = None, stream=None) -> None:
    wsb = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    rc = load_library().locks_select(
        ctypes.byref(cfg.c()), _ptr(q), _ptr(summaries), _ptr(block_table), _ptr(seq_lens),
        int(budget_tokens), _ptr(selected), _ptr(page_lse), _ptr(page_share), _ptr(workspace),
        int(wsb), _ptr(status), _stream(stream))
    _check("locks_select", rc)


def locks_select_noalloc(cfg: LocksConfig, q, summaries, block_table, seq_lens,
                         budget_tokens: int, selected, page_lse=None, page_share=None,
                         status=None, stream=None) -> None:
    """locks_select without a workspace: the scratch is a fixed device array
    inside the library (for callers that cannot allocate device memory)."""
    rc = load_library().locks_select_noalloc(
        ctypes.byref(cfg.c()), _ptr(q), _ptr(summaries), _ptr(block_table), _ptr(seq_lens),
        int(budget_tokens), _ptr(selected), _ptr(page_lse), _ptr(page_share), _ptr(status),
        _stream(stream))
    _check("locks_select_noalloc", rc)


def locks_sparse_decode(cfg: LocksConfig, q, k_cache, v_cache, block_table, seq_lens, selected,
                        k: int, out, workspace, out_lse=None, status=None,
                        workspace_bytes: Optional[int] = None, stream=None) -> None:
    wsb = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    rc = load_library().locks_sparse_decode(
        ctypes.byref(cfg.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(selected), int(k), _ptr(out), _ptr(out_lse), _ptr(workspace),
        int(wsb), _ptr(status), _stream(stream))
    _check("locks_sparse_decode", rc)


def locks_dense_decode(cfg: LocksConfig, q, k_cache, v_cache, block_table, seq_lens, out,
                       workspace, out_lse=None, status=None,
                       workspace_bytes: Optional[int] = None, stream=None) -> None:
    wsb = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    rc = load_library().locks_dense_decode(
        ctypes.byref(cfg.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(out), _ptr(out_lse), _ptr(workspace), int(wsb), _ptr(status),
        _stream(stream))
    _check("locks_dense_decode", rc)


# --------------------------------------------------------------------------
# host-side view of the summary record layout (see locks.h)
# --------------------------------------------------------------------------
def unpack_i4(raw, cfg: LocksConfig) -> Tuple:
    """Codes (unbiased int32) and scales of quantised records [..., record_bytes]
    (fragment-order layout in locks.h): mu_codes [..., d], mu_scale [...],
    v_codes [..., d, R], v_scales [..., R], c_codes [..., B, R], c_scales [..., B]."""
    import numpy as np
    d, B, R = cfg.head_dim, cfg.page_size, cfg.rank_cap
    KK = (R + 7) // 8
    raw = np.asarray(raw, dtype=np.uint8)
    lead = raw.shape[:-1]
    hdr = ((R + 1) * 4 + 15) // 16 * 16
    off_mq = hdr + 64 * R
    off_cq = off_mq + 128
    off_cs = off_cq + 8 * B * KK

    def f32(a, b):
        return np.ascontiguousarray(raw[..., a:b]).view(np.float32)

    head = f32(0, 4 * (R + 1))
    v_scales, mu_scale = head[..., :R], head[..., R]
    t = np.arange(4)
    # basis: word [k][t][j], nibble n -> (k-step 2j + (n & 3) // 2, column offset)
    words = np.ascontiguousarray(raw[..., hdr:off_mq]).view(np.uint32).reshape(*lead, R, 4, 4)
    v_codes = np.zeros((*lead, d, R), dtype=np.int32)
    for n in range(8):
        nib = ((words >> np.uint32(4 * n)) & np.uint32(15)).astype(np.int32) - 8   # [..., k, t, j]
        step = 2 * np.arange(4)[None, :] + ((n & 3) // 2)                            # [t?, j]
        off = (8 if (n & 1) else 0) + (1 if n >= 4 else 0)
        cols = 16 * step + 2 * t[:, None] + off                                       # [t, j]
        v_codes[..., cols, :] = np.moveaxis(nib, -3, -1)
    # centroid: lane l = 4g + t -> columns 16g + 2t + (0, 1, 8, 9)
    mb = raw[..., off_mq:off_cq].reshape(*lead, 8, 4, 4).astype(np.int32) - 128
    mu_codes = np.zeros((*lead, d), dtype=np.int32)
    g = np.arange(8)[:, None]
    for e, off in enumerate((0, 1, 8, 9)):
        mu_codes[..., 16 * g + 2 * t[None, :] + off] = mb[..., e]
    # coefficients: cq[m][kk][l] bytes = (16m+g, 8kk+2t), (16m+g, +1), (16m+g+8, 8kk+2t), (.., +1)
    cb = raw[..., off_cq:off_cs].reshape(*lead, B // 16, KK, 8, 4, 4).astype(np.int32) - 128
    c_full = np.zeros((*lead, B, 8 * KK), dtype=np.int32)
    m = np.arange(B // 16)[:, None, None, None]
    kk = np.arange(KK)[None, :, None, None]
    gg = np.arange(8)[None, None, :, None]
    tt = np.arange(4)[None, None, None, :]
    for e, (di, dk) in enumerate(((0, 0), (0, 1), (8, 0), (8, 1))):
        c_full[..., 16 * m + gg + di, 8 * kk + 2 * tt + dk] = cb[..., e]
    c_codes = c_full[..., :R]
    c_scales = f32(off_cs, off_cs + 4 * B)
    return mu_codes, mu_scale, v_codes, v_scales, c_codes, c_scales


def unpack_records(raw, cfg: LocksConfig) -> Tuple:
    """Split host record bytes [..., record_bytes] into (mu, V, C) float64 arrays
    (a quantised record is dequantised: code times its group's scale).

    mu: [..., d]; V: [..., d, rank] (basis columns); C: [..., B, rank]."""
    import numpy as np
    d, B, R = cfg.head_dim, cfg.page_size, cfg.rank_cap
    raw = np.asarray(raw)
    lead = raw.shape[:-1]
    if cfg.summary_dtype == LOCKS_SUMMARY_I4:
        mu_c, mu_s, v_c, v_s, c_c, c_s = unpack_i4(raw, cfg)
        mu = mu_c * mu_s.astype(np.float64)[..., None]
        V = v_c * v_s.astype(np.float64)[..., None, :]
        C = c_c * c_s.astype(np.float64)[..., :, None]
        return mu, V[..., :cfg.rank], C[..., :cfg.rank]
    if cfg.summary_dtype == LOCKS_SUMMARY_F32:
        x = raw.view(np.float32).astype(np.float64)
    else:
        x = (raw.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    W = x[..., :(R + 1) * d].reshape(*lead, R + 1, d)
    C4 = x[..., (R + 1) * d:(R + 1) * d + R * B].reshape(*lead, R // 4, B, 4)
    C = np.moveaxis(C4, -3, -2).reshape(*lead, B, R)
    mu = W[..., 0, :]
    V = np.swapaxes(W[..., 1:, :], -1, -2)
    return mu, V[..., :cfg.rank], C[..., :cfg.rank]
