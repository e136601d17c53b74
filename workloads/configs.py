"""Named synthetic decode workloads for the Locks hot path.

Each workload fixes the shapes of one attention layer at decode time (batch,
query/KV heads, head dimension, page size B, context T, summary rank r, token
budget b) and the recipe of its synthetic keys: per page a rank-8 product
A_p G_p with A_p, G_p ~ N(0,1)/sqrt(8), isotropic noise, optionally a shared
global rank-16 component, and a few "carrier" pages whose keys are shifted by
0.5 times the unit direction of the GQA group's summed query (or, with
carrier_token, a single token of each carrier page shifted by carrier_bias:
a "peaky" needle that moves the page centroid by only 1/B of that).

The shapes follow the layer shapes of the models the Locks paper evaluates on
(Llama-3.1-8B: 32 query / 8 KV heads; Qwen3-4B: 32 / 8; head_dim 128) and its
budget regime ("Locks: Page-Local Compact Key Summaries for Efficient
Long-Context Decoding", section 2 for the budget b and k = ceil(b/B); section 5.3
and Table C.9 for the 16K..1M contexts). Real model traces and datasets are not
used; these synthetic workloads stand in for them.

This module holds no arithmetic of the method itself.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class LocksWorkload:
    """Shapes and key-generator recipe of one synthetic decode workload."""

    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    context: int                      # tokens per sequence (all rows equal unless seq_lens given)
    rank: int                         # summary rank r
    budget_tokens: int                # per-(sequence, KV head) token budget b
    noise: float = 0.05               # std of the isotropic key noise
    local_rank: int = 8               # rank of the per-page A_p G_p component
    global_rank: int = 0              # rank of the shared per-(sequence, KV head) component (0 = none)
    carrier_count: Optional[int] = None   # carriers per (sequence, KV head); overrides carrier_frac
    carrier_frac: float = 0.0         # fraction of candidate pages made carriers (rounded up)
    carrier_bias: float = 0.5         # shift of every key of a carrier page along the group query direction
    carrier_token: bool = False       # shift one (seeded) token of each carrier page instead of every key
    seed: int = 1000
    seq_lens: Optional[Tuple[int, ...]] = None   # ragged per-sequence lengths (overrides context)
    spare_blocks: int = 3             # unused physical blocks in the pool (filled with NaN)
    headroom_pages: int = 0           # block-table entries (and blocks) per sequence beyond its
                                      # length, for pages a decode loop will start
    description: str = field(default="", compare=False)

    # ---- derived sizes -------------------------------------------------
    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def lengths(self) -> Tuple[int, ...]:
        if self.seq_lens is not None:
            assert len(self.seq_lens) == self.batch
            return tuple(int(x) for x in self.seq_lens)
        return (self.context,) * self.batch

    @property
    def max_pages(self) -> int:
        return max(1, max(math.ceil(t / self.page_size) for t in self.lengths())) + \
            self.headroom_pages

    @property
    def page_budget(self) -> int:
        """k = ceil(b / B)."""
        return math.ceil(self.budget_tokens / self.page_size)

    @property
    def num_blocks(self) -> int:
        return self.batch * self.max_pages + self.spare_blocks

    def with_(self, **kw) -> "LocksWorkload":
        return replace(self, **kw)


# The five workloads, smallest first.  "tiny" is the case the oracle finishes in
# seconds; "llama32k" is the single-GPU decode-step workload the bench times.
TINY = LocksWorkload(
    name="tiny", batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=64,
    context=4096, rank=8, budget_tokens=512, noise=0.05, global_rank=0,
    carrier_count=3, seed=1000,
    description="batch 1, 8/2 heads, d 128, B 64, T 4096, r 8, b 512, 3 carriers")

LLAMA32K = LocksWorkload(
    name="llama32k", batch=8, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=64,
    context=32768, rank=8, budget_tokens=2048, noise=0.05, global_rank=16,
    carrier_frac=0.01, seed=1001,
    description="Llama-3.1-8B layer shape, batch 8, T 32768, r 8, b 2048, 1% carriers")

LONG128K = LocksWorkload(
    name="long128k", batch=4, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=64,
    context=131072, rank=8, budget_tokens=2048, noise=0.05, global_rank=16,
    carrier_frac=0.01, seed=1002,
    description="Llama-3.1-8B layer shape, batch 4, T 131072, r 8, b 2048")

QWEN16K = LocksWorkload(
    name="qwen16k", batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=64,
    context=16384, rank=8, budget_tokens=256, noise=0.1, global_rank=16,
    carrier_frac=0.005, seed=1003,
    description="Qwen3-4B layer shape, batch 16, T 16384, r 8, b 256, noise 0.1, 0.5% carriers")

ONE_M = LocksWorkload(
    name="1m", batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=64,
    context=1048576, rank=8, budget_tokens=2048, noise=0.05, global_rank=16,
    carrier_frac=0.01, seed=1004,
    description="Llama-3.1-8B layer shape, batch 1, T 1048576 (~4 GiB bf16 KV), r 8, b 2048")

CONFIGS = {w.name: w for w in (TINY, LLAMA32K, LONG128K, QWEN16K, ONE_M)}
ORDER = ("tiny", "llama32k", "long128k", "qwen16k", "1m")


def get(name: str) -> LocksWorkload:
    return CONFIGS[name]
