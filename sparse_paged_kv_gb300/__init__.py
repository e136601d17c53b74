"""sparse_paged_kv_gb300 -- the Locks decode-attention hot path on GB300 (sm_103a).

The compute lives in ``lib/libsparse_paged_kv.so`` (hand-written CUDA behind the
C ABI of ``include/locks.h``); ``binding`` marshals torch tensors into it and
``runtime`` bundles the buffers of one decode layer.
"""
from .binding import (LOCKS_SUMMARY_BF16, LOCKS_SUMMARY_F32, LocksConfig, LocksError,  # noqa: F401
                      LocksLibraryMissing, load_library, locks_build_summaries,
                      locks_dense_decode, locks_select, locks_sparse_decode, unpack_records)
