"""Device buffers of one Locks decode layer, held in torch CUDA tensors.

``LocksLayer`` owns the paged K/V pools, the block table, the summary pool and
the workspaces of one attention layer and calls the C-ABI entry points on
them.  PyTorch only provides memory and streams; every step runs in the
library's kernels.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from . import binding as B


def complete_page_blocks(block_table: np.ndarray, seq_lens: np.ndarray, page_size: int) -> np.ndarray:
    """Physical blocks of every complete page (host arrays in, int32 out)."""
    out = []
    for b, t in enumerate(seq_lens.tolist()):
        n_complete = int(t) // page_size
        out.append(block_table[b, :n_complete])
    return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)


class LocksLayer:
    def __init__(self, cfg: B.LocksConfig, budget_tokens: int, device: str = "cuda"):
        import torch
        self.torch = torch
        self.cfg = cfg
        self.budget = int(budget_tokens)
        self.k = cfg.page_budget(self.budget)
        self.device = device
        d = device
        self.rec_bytes = B.summary_record_bytes(cfg)
        if self.rec_bytes == 0:
            raise B.LocksError("locks_summary_record_bytes", B.LOCKS_ERR_UNSUPPORTED, "unsupported cfg")
        self.summaries = torch.zeros((cfg.num_blocks, cfg.n_kv_heads, self.rec_bytes),
                                     dtype=torch.uint8, device=d)
        self.ws_select = torch.zeros(max(1, B.select_workspace_bytes(cfg, self.budget)),
                                     dtype=torch.uint8, device=d)
        self.ws_sparse = torch.zeros(max(1, B.decode_workspace_bytes(cfg, self.k)),
                                     dtype=torch.uint8, device=d)
        self.ws_dense = torch.zeros(max(1, B.decode_workspace_bytes(cfg, cfg.max_pages)),
                                    dtype=torch.uint8, device=d)
        self.selected = torch.full((cfg.batch, cfg.n_kv_heads, self.k), -1, dtype=torch.int32, device=d)
        self.out = torch.zeros((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.bfloat16, device=d)
        self.out_lse = torch.zeros((cfg.batch, cfg.n_q_heads), dtype=torch.float32, device=d)
        self.out_dense = torch.zeros_like(self.out)
        self.out_dense_lse = torch.zeros_like(self.out_lse)
        self.status = torch.zeros(1, dtype=torch.int32, device=d)
        self.q = self.k_cache = self.v_cache = self.block_table = self.seq_lens = None

    # ---- inputs -------------------------------------------------------------
    def load_inputs(self, inputs) -> "LocksLayer":
        """Copy seeded host inputs (workloads.LocksInputs) into device memory."""
        torch = self.torch
        d = self.device

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(d).view(torch.bfloat16)

        self.q = bf16(inputs.q)
        self.k_cache = bf16(inputs.k_cache)
        self.v_cache = bf16(inputs.v_cache)
        self.block_table = torch.from_numpy(inputs.block_table).to(d)
        self.seq_lens = torch.from_numpy(inputs.seq_lens).to(d)
        self.host_block_table = inputs.block_table
        self.host_seq_lens = inputs.seq_lens
        return self

    @classmethod
    def from_inputs(cls, inputs, summary_dtype: int = B.LOCKS_SUMMARY_F32,
                    budget_tokens: Optional[int] = None) -> "LocksLayer":
        w = inputs.workload
        cfg = B.LocksConfig.from_workload(w, summary_dtype)
        return cls(cfg, w.budget_tokens if budget_tokens is None else budget_tokens).load_inputs(inputs)

    def sharing_inputs(self, summary_dtype: int) -> "LocksLayer":
        """A layer over the same device inputs (q, K/V pools, block table,
        sequence lengths) with its own summary pool of another record type."""
        cfg = dataclasses.replace(self.cfg, summary_dtype=int(summary_dtype))
        other = LocksLayer(cfg, self.budget, self.device)
        for name in ("q", "k_cache", "v_cache", "block_table", "seq_lens", "host_block_table",
                     "host_seq_lens"):
            setattr(other, name, getattr(self, name))
        return other

    # ---- calls ----------------------------------------------------------------
    def build(self, block_ids=None, tail_energy=None, status=None, max_sweeps: int = 0):
        torch = self.torch
        if block_ids is None:
            ids = complete_page_blocks(self.host_block_table, self.host_seq_lens, self.cfg.page_size)
            block_ids = torch.from_numpy(ids).to(self.device)
        if block_ids.numel() == 0:
            return block_ids
        B.locks_build_summaries(self.cfg, self.k_cache, block_ids, self.summaries,
                                tail_energy=tail_energy, status=status, max_sweeps=max_sweeps)
        return block_ids

    def select(self, page_lse=None, page_share=None, stream=None):
        B.locks_select(self.cfg, self.q, self.summaries, self.block_table, self.seq_lens,
                       self.budget, self.selected, self.ws_select, page_lse=page_lse,
                       page_share=page_share, status=self.status, stream=stream)

    def sparse_decode(self, stream=None):
        B.locks_sparse_decode(self.cfg, self.q, self.k_cache, self.v_cache, self.block_table,
                              self.seq_lens, self.selected, self.k, self.out, self.ws_sparse,
                              out_lse=self.out_lse, status=self.status, stream=stream)

    def dense_decode(self, stream=None):
        B.locks_dense_decode(self.cfg, self.q, self.k_cache, self.v_cache, self.block_table,
                             self.seq_lens, self.out_dense, self.ws_dense,
                             out_lse=self.out_dense_lse, status=self.status, stream=stream)

    def step(self, stream=None):
        """One sparse decode step: selection, then attention over the selected pages."""
        self.select(stream=stream)
        self.sparse_decode(stream=stream)

    def capture_step(self):
        """A CUDA graph of one sparse decode step (selection, then attention)
        over this layer's buffers.  replay() runs it on the current stream and
        reads q, seq_lens and block_table as they are at replay time.  The
        step runs once outside the capture first, so one-time launch set-up
        (kernel attributes, the cluster-size query) never happens inside it."""
        torch = self.torch
        cur = torch.cuda.current_stream(self.device)
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            self.step()
        cur.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.step()
        return graph

    def append(self, k_new, v_new, completed=None, stream=None):
        """Write each sequence's new token (k_new, v_new: bf16 [batch][H_kv][d]
        on the device) at position seq_lens[b], advance seq_lens, and store in
        `completed` (int32 [batch]) the block of each page the token completed
        (-1 for none)."""
        B.locks_append_kv(self.cfg, k_new, v_new, self.k_cache, self.v_cache, self.block_table,
                          self.seq_lens, completed=completed, status=self.status, stream=stream)

    def build_completed(self, completed, status=None, stream=None):
        """Summaries of the blocks listed in `completed` (entries < 0 skipped)."""
        B.locks_build_completed(self.cfg, self.k_cache, completed, self.summaries, status=status,
                                stream=stream)

    # ---- diagnostics ------------------------------------------------------------
    def host_records(self, blocks, h: int):
        """(mu, V, C) of the given physical blocks for KV head h (float64, host)."""
        raw = self.summaries[self.torch.as_tensor(np.asarray(blocks), device=self.device).long(), h]
        return B.unpack_records(raw.cpu().numpy(), self.cfg)

    def alloc_page_lse(self):
        c = self.cfg
        return self.torch.full((c.batch, c.n_q_heads, c.max_pages), float("nan"),
                               dtype=self.torch.float32, device=self.device)

    def alloc_page_share(self):
        c = self.cfg
        return self.torch.full((c.batch, c.n_kv_heads, c.max_pages), float("nan"),
                               dtype=self.torch.float32, device=self.device)


class DecodeLoop:
    """Decode steps of one layer as an engine runs them, with no host round
    trip: each step appends the new token (current stream), builds the
    summary of any page that token completed on a side stream, then selects
    and decodes.  A page completed at step s becomes a selection candidate at
    step s + 1, so its build overlaps step s's selection and decode, and step
    s + 1's selection waits for it (section 4 "Build": one build per
    finalised page, off the critical path).  Two `completed` buffers
    alternate, so a step's append never overwrites the list the previous
    step's build may still be reading."""

    def __init__(self, layer: LocksLayer, host_lengths=None):
        """host_lengths: optional int array of the sequences' current lengths
        as the caller tracks them (an engine knows them: it allocates a block
        for each page a sequence starts).  With them, a step in which no
        sequence completes a page launches no build; which blocks are built
        is still decided on the device, from the `completed` list."""
        import torch
        self.torch = torch
        self.layer = layer
        self.side = torch.cuda.Stream(device=layer.device)
        self.completed = [torch.full((layer.cfg.batch,), -1, dtype=torch.int32,
                                     device=layer.device) for _ in range(2)]
        self.appended = torch.cuda.Event()
        self.built = None             # event: the previous step's build is done
        self.steps = 0
        self.host_lengths = None if host_lengths is None else np.array(host_lengths, dtype=np.int64)

    def step(self, k_new, v_new, page_lse=None, page_share=None):
        torch = self.torch
        L = self.layer
        cur = torch.cuda.current_stream(L.device)
        done = self.completed[self.steps & 1]
        L.append(k_new, v_new, completed=done, stream=cur)
        crosses = True
        if self.host_lengths is not None:
            crosses = bool(((self.host_lengths + 1) % L.cfg.page_size == 0).any())
            self.host_lengths += 1
        built = None
        if crosses:
            self.appended.record(cur)
            self.side.wait_event(self.appended)
            L.build_completed(done, stream=self.side)
            built = torch.cuda.Event()
            built.record(self.side)
        if self.built is not None:
            cur.wait_event(self.built)
        self.built = built
        L.select(page_lse=page_lse, page_share=page_share, stream=cur)
        L.sparse_decode(stream=cur)
        self.steps += 1

    def finish(self):
        """Make the current stream wait for the last step's build."""
        if self.built is not None:
            self.torch.cuda.current_stream(self.layer.device).wait_event(self.built)
