"""GPU-vs-oracle comparison helpers (used by the -m gpu tests and the smoke check).

Gates (fp32 summaries, bf16 KV with fp32 accumulation):
  * reconstructed page scores s_hat: 1e-3 absolute;
  * selected page sets: identical, except pages whose oracle averaged share is
    within 1e-5 of the oracle's (k-2)-th (last selected) candidate share;
  * attention outputs: 2e-2 absolute (bf16 output), lse 1e-3 absolute; the
    sparse output is compared with the oracle attending the GPU's selected set,
    so a legitimate tie-window difference cannot fail it;
  * build: the projector-invariant reconstruction C V^T within
    max(1e-4, 2e-5 * sigma_1^2 / (sigma_r^2 - sigma_{r+1}^2)) of max|D| -- the
    rank-r subspace is fixed only up to the spectral gap (Cor. 1), and an fp32
    solve perturbs it by about (fp32 roundoff x sigma_1^2) / gap (Davis-Kahan) --
    the top-r sigma^2 (= squared column norms of C) within 1e-4 of sigma_1^2,
    V^T V = I within max(1e-4, 4e-6 sigma_1^2 / (sigma_k sigma_l)) -- the
    solve's 1e-6 residual, amplified by v_k = D^T u_k / sigma_k for small kept
    modes -- tau within 1e-4 of the Gram trace.
Pages whose relative spectral gap (sigma_r^2 - sigma_{r+1}^2) / sigma_1^2 is
below 1e-4 have no unique rank-r subspace (Cor. 1) and are excluded from the
score and reconstruction gates; they are counted.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Tuple

import numpy as np

import oracle as O

LSE_TOL = 1e-3
OUT_TOL = 2e-2
OUT_LSE_TOL = 1e-3
TIE_TOL = 1e-5
# averaged shares m_bar, element by element: within the tie window in absolute
# terms, and within the relative change that the s_hat gate allows -- every
# s_hat within LSE_TOL moves log Z by at most LSE_TOL too, so each share
# exp(s_hat - log Z) by at most a factor e^{2 LSE_TOL}, and so their mean;
# 1e-5 more covers the float32 exponentials and sums
SHARE_ABS_TOL = TIE_TOL
SHARE_REL_TOL = math.expm1(2 * LSE_TOL) + 1e-5
RECON_TOL = 1e-4
RECON_GAP_COEF = 2e-5
SIGMA_TOL = 1e-4
ORTHO_TOL = 1e-4
# a symmetric eigensolve stopped at an off-diagonal residual e*|A| fixes the
# basis columns v_k = D^T u_k / sigma_k of modes k, l only to about
# e * sigma_1^2 / (sigma_k sigma_l) (first-order perturbation); the build stops
# at e = 1e-6, and the gate allows four times that
ORTHO_RESID_COEF = 4e-6
TAU_TOL = 1e-4
DEGENERATE_GAP = 1e-4


@dataclass
class Report:
    units: int = 0
    pages: int = 0
    degenerate: int = 0
    tie_diffs: int = 0
    max_lse_err: float = 0.0
    max_out_err: float = 0.0
    max_dense_err: float = 0.0
    max_recon_rel: float = 0.0
    max_sigma_rel: float = 0.0
    max_record_err: float = 0.0
    max_share_abs: float = 0.0
    max_share_rel: float = 0.0
    # largest e_rec * gap over the gated pages: the coefficient the
    # reconstruction gate max(RECON_TOL, RECON_GAP_COEF / gap) actually needed
    max_recon_gap: float = 0.0
    failures: List[str] = field(default_factory=list)

    def fail(self, msg):
        self.failures.append(msg)

    def check(self):
        assert not self.failures, "\n".join(self.failures[:20])


def degenerate(s: O.PageSummary, r: int) -> bool:
    if len(s.sigma2) <= r or s.sigma2[0] <= 0:
        return False
    return (s.sigma2[r - 1] - s.sigma2[r]) / s.sigma2[0] < DEGENERATE_GAP


def gpu_snapshot(layer, page_lse=None, page_share=None):
    """Copy the GPU outputs of one step to host numpy arrays."""
    import torch
    torch.cuda.synchronize()
    snap = {
        "selected": layer.selected.cpu().numpy(),
        "out": layer.out.float().cpu().numpy().astype(np.float64),
        "out_lse": layer.out_lse.cpu().numpy().astype(np.float64),
        "out_dense": layer.out_dense.float().cpu().numpy().astype(np.float64),
        "out_dense_lse": layer.out_dense_lse.cpu().numpy().astype(np.float64),
        "status": int(layer.status.cpu().numpy()[0]),
    }
    if page_lse is not None:
        snap["page_lse"] = page_lse.cpu().numpy().astype(np.float64)
    if page_share is not None:
        snap["page_share"] = page_share.cpu().numpy().astype(np.float64)
    return snap


def compare_build(layer, inputs, res: O.UnitResult, rep: Report, tail=None, status=None,
                  block_index=None):
    """GPU summary records of one unit against the oracle's page summaries."""
    b, h = res.b, res.h
    r = layer.cfg.rank
    pages = sorted(res.summaries)
    if not pages:
        return
    blocks = inputs.block_table[b, pages]
    mu, V, C = layer.host_records(blocks, h)
    for n_, j in enumerate(pages):
        s = res.summaries[j]
        keys = O.page_keys(inputs.k_cache, inputs.block_table, b, h, j, layer.cfg.page_size)
        D = keys - keys.mean(axis=0)
        scale = np.abs(D).max()
        if np.abs(mu[n_] - s.mu).max() > 1e-6 * max(1.0, np.abs(s.mu).max()):
            rep.fail(f"mu b{b} h{h} p{j}")
        sig_gpu = (C[n_] ** 2).sum(axis=0)
        sig_ref = np.where(np.arange(r) < s.kept, s.sigma2[:r], 0.0)
        e_sig = np.abs(sig_gpu - sig_ref).max() / s.sigma2[0]
        rep.max_sigma_rel = max(rep.max_sigma_rel, e_sig)
        if e_sig > SIGMA_TOL:
            rep.fail(f"sigma2 b{b} h{h} p{j}: {e_sig:.2e}")
        kept = sig_gpu > 0
        VtV = V[n_][:, kept].T @ V[n_][:, kept]
        sk = np.sqrt(np.maximum(sig_gpu[kept], 1e-300))
        o_tol = np.maximum(ORTHO_TOL, ORTHO_RESID_COEF * s.sigma2[0] / np.outer(sk, sk))
        o_err = np.abs(VtV - np.eye(kept.sum()))
        if (o_err > o_tol).any():
            rep.fail(f"orthonormal b{b} h{h} p{j}: {o_err.max():.2e} "
                     f"(allowed {o_tol[np.unravel_index(np.argmax(o_err / o_tol), o_err.shape)]:.2e})")
        if degenerate(s, r):
            rep.degenerate += 1
            continue
        rec_gpu = C[n_] @ V[n_].T
        rec_ref = s.C @ s.V.T
        e_rec = np.abs(rec_gpu - rec_ref).max() / scale
        rep.max_recon_rel = max(rep.max_recon_rel, e_rec)
        gap = (s.sigma2[r - 1] - s.sigma2[r]) / s.sigma2[0] if len(s.sigma2) > r else 1.0
        rep.max_recon_gap = max(rep.max_recon_gap, e_rec * gap)
        tol = max(RECON_TOL, RECON_GAP_COEF / gap)
        if e_rec > tol:
            rep.fail(f"reconstruction b{b} h{h} p{j}: {e_rec:.2e} (relative gap {gap:.2e})")
        if tail is not None and block_index is not None:
            t_gpu = float(tail[block_index[blocks[n_]], h])
            trace = float(np.trace(D @ D.T))
            if abs(t_gpu - s.tau) > TAU_TOL * trace:
                rep.fail(f"tau b{b} h{h} p{j}: {t_gpu} vs {s.tau}")


def compare_select(layer, snap, res: O.UnitResult, rep: Report):
    b, h = res.b, res.h
    G = layer.cfg.group
    sel = res.sel
    rep.units += 1
    rep.pages += len(sel.cand)
    degen = {int(j) for j in sel.cand if degenerate(res.summaries[int(j)], layer.cfg.rank)}
    if "page_lse" in snap and len(sel.cand):
        g_lse = snap["page_lse"][b, h * G:(h + 1) * G][:, sel.cand]
        err = np.abs(g_lse - sel.scores)
        mask = np.array([int(j) not in degen for j in sel.cand])
        if mask.any():
            e = err[:, mask].max()
            rep.max_lse_err = max(rep.max_lse_err, e)
            if not np.isfinite(e) or e > LSE_TOL:
                rep.fail(f"s_hat b{b} h{h}: max err {e:.3e}")
    if "page_share" in snap and len(sel.cand):
        sh = snap["page_share"][b, h][sel.cand]
        if abs(sh.sum() - 1.0) > 1e-4:
            rep.fail(f"shares b{b} h{h} sum to {sh.sum()}")
        if not degen:                     # a degenerate page's s_hat is not gated
            err = np.abs(sh - sel.mbar)
            rel = float((err / np.maximum(sel.mbar, 1e-30)).max())
            rep.max_share_abs = max(rep.max_share_abs, float(err.max()))
            rep.max_share_rel = max(rep.max_share_rel, rel)
            if not np.isfinite(err.max()) or err.max() > SHARE_ABS_TOL or rel > SHARE_REL_TOL:
                rep.fail(f"shares b{b} h{h}: max abs err {err.max():.3e}, rel {rel:.3e}")
    got = [int(x) for x in snap["selected"][b, h] if x >= 0]
    want = [int(x) for x in sel.selected]
    if got != sorted(got) or len(set(got)) != len(got):
        rep.fail(f"selected b{b} h{h} not ascending/unique: {got}")
    if len(got) != len(want):
        rep.fail(f"selected b{b} h{h}: {len(got)} pages, oracle {len(want)}")
        return
    diff = set(got) ^ set(want)
    if diff:
        idx = {int(j): i for i, j in enumerate(sel.cand)}
        chosen = [j for j in want if j in idx]
        thr = min(sel.mbar[idx[j]] for j in chosen) if chosen else 0.0
        for j in diff:
            if j not in idx or abs(sel.mbar[idx[j]] - thr) > TIE_TOL:
                rep.fail(f"selected b{b} h{h}: page {j} differs outside the tie window "
                         f"(got {got}, oracle {want})")
                return
        rep.tie_diffs += len(diff) // 2


def compare_sparse_decode(layer, inputs, snap, res: O.UnitResult, rep: Report):
    b, h = res.b, res.h
    G = layer.cfg.group
    got = [int(x) for x in snap["selected"][b, h] if x >= 0]
    q = O.bf16_to_f64(inputs.q[b, h * G:(h + 1) * G])
    o, lse = O.attend_pages(q, inputs.k_cache, inputs.v_cache, inputs.block_table,
                            int(inputs.seq_lens[b]), b, h, got)
    g_o = snap["out"][b, h * G:(h + 1) * G]
    g_l = snap["out_lse"][b, h * G:(h + 1) * G]
    e = np.abs(g_o - o).max() if o.size else 0.0
    rep.max_out_err = max(rep.max_out_err, e)
    if not np.isfinite(e) or e > OUT_TOL:
        rep.fail(f"sparse out b{b} h{h}: {e:.3e}")
    if np.isneginf(lse).any() or np.isneginf(g_l).any():
        if not np.array_equal(np.isneginf(lse), np.isneginf(g_l)):
            rep.fail(f"sparse lse b{b} h{h}: -inf mismatch")
    elif np.abs(g_l - lse).max() > OUT_LSE_TOL:
        rep.fail(f"sparse lse b{b} h{h}: {np.abs(g_l - lse).max():.3e}")


def compare_dense_decode(layer, inputs, snap, res: O.UnitResult, rep: Report):
    b, h = res.b, res.h
    G = layer.cfg.group
    g_o = snap["out_dense"][b, h * G:(h + 1) * G]
    g_l = snap["out_dense_lse"][b, h * G:(h + 1) * G]
    e = np.abs(g_o - res.o_dense).max()
    rep.max_dense_err = max(rep.max_dense_err, e)
    if not np.isfinite(e) or e > OUT_TOL:
        rep.fail(f"dense out b{b} h{h}: {e:.3e}")
    if np.isneginf(res.lse_dense).any() or np.isneginf(g_l).any():
        if not np.array_equal(np.isneginf(res.lse_dense), np.isneginf(g_l)):
            rep.fail(f"dense lse b{b} h{h}: -inf mismatch")
    elif np.abs(g_l - res.lse_dense).max() > OUT_LSE_TOL:
        rep.fail(f"dense lse b{b} h{h}: {np.abs(g_l - res.lse_dense).max():.3e}")


def records_as_summaries(layer, inputs, b: int, h: int):
    """The GPU-stored records of one unit's candidate pages as oracle page
    summaries (values upcast exactly to fp64).  A bf16 record is a rounded
    copy of the spectral summary, so its selection and score gates take the
    oracle scoring the stored record itself; only mu, V and C enter a score."""
    w = inputs.workload
    _, cand = O.forced_and_candidates(int(inputs.seq_lens[b]), w.page_size)
    if len(cand) == 0:
        return {}
    pages = [int(j) for j in cand]
    mu, V, C = layer.host_records(inputs.block_table[b, pages], h)
    out = {}
    for i, j in enumerate(pages):
        sig = (C[i] ** 2).sum(axis=0)
        out[j] = O.PageSummary(mu=mu[i], V=V[i], C=C[i], sigma2=sig, tau=0.0,
                               kept=int((sig > 0).sum()))
    return out


def record_error(layer, inputs, b: int, h: int, fp64) -> float:
    """Max over the unit's pages of |C V^T (stored) - C V^T (fp64)| / max|D|:
    how far a reduced-precision record is from the fp64 summary (a measurement,
    not a gate)."""
    w = inputs.workload
    pages = sorted(fp64)
    if not pages:
        return 0.0
    _, V, C = layer.host_records(inputs.block_table[b, pages], h)
    err = 0.0
    for i, j in enumerate(pages):
        s = fp64[j]
        if degenerate(s, w.rank):
            continue                      # no unique rank-r subspace to compare
        keys = O.page_keys(inputs.k_cache, inputs.block_table, b, h, j, w.page_size)
        scale = np.abs(keys - keys.mean(axis=0)).max()
        err = max(err, float(np.abs(C[i] @ V[i].T - s.C @ s.V.T).max() / scale))
    return err


def run_case(inputs, units=None, dense=True, check_build=True, summary_dtype=0, max_sweeps=0):
    """Build, select, sparse- and dense-decode on the GPU; compare the given
    units (default: all) with the oracle.  Returns (report, layer, snapshot).

    summary_dtype 1 (bf16 records) or 2 (quantised records): the build is
    measured, not gated (report.max_record_err), and selection/scores are
    gated against the oracle scoring the GPU-stored records.

    max_sweeps > 0 builds with the Jacobi solver and that sweep cap (at page
    size 64 the default is the tridiagonal solver)."""
    import torch
    from sparse_paged_kv_gb300 import runtime
    w = inputs.workload
    layer = runtime.LocksLayer.from_inputs(inputs, summary_dtype=summary_dtype)
    ids = runtime.complete_page_blocks(inputs.block_table, inputs.seq_lens, w.page_size)
    ids_t = torch.from_numpy(ids).cuda()
    tail = torch.full((max(1, len(ids)), w.n_kv_heads), float("nan"), device="cuda")
    bstat = torch.zeros((max(1, len(ids)), w.n_kv_heads), dtype=torch.int32, device="cuda")
    layer.build(ids_t, tail_energy=tail, status=bstat, max_sweeps=max_sweeps)
    page_lse = layer.alloc_page_lse()
    page_share = layer.alloc_page_share()
    layer.select(page_lse=page_lse, page_share=page_share)
    layer.sparse_decode()
    if dense:
        layer.dense_decode()
    snap = gpu_snapshot(layer, page_lse, page_share)
    bstat_h = bstat.cpu().numpy()
    tail_h = tail.cpu().numpy()
    rep = Report()
    if snap["status"] != 0:
        rep.fail(f"device status {snap['status']:#x}")
    if len(ids) and ((bstat_h >> 16) != 0).any():
        rep.fail(f"build status flags {np.unique(bstat_h >> 16)}")
    block_index = {int(x): i for i, x in enumerate(ids)}
    if units is None:
        units = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    for b, h in units:
        stored = records_as_summaries(layer, inputs, b, h) if summary_dtype != 0 else None
        res = O.run_unit(inputs.q, inputs.k_cache, inputs.v_cache, inputs.block_table,
                         inputs.seq_lens, w.n_kv_heads, w.rank, w.budget_tokens, b, h, dense=dense,
                         summaries=stored)
        if check_build and summary_dtype != 0:
            fp64 = O.build_unit(inputs.k_cache, inputs.block_table, int(inputs.seq_lens[b]), b, h,
                                w.rank)
            rep.max_record_err = max(rep.max_record_err, record_error(layer, inputs, b, h, fp64))
        elif check_build:
            compare_build(layer, inputs, res, rep, tail=tail_h, block_index=block_index)
        compare_select(layer, snap, res, rep)
        compare_sparse_decode(layer, inputs, snap, res, rep)
        if dense:
            compare_dense_decode(layer, inputs, snap, res, rep)
    snap["build_sweeps"] = (bstat_h & 0xFFFF) if len(ids) else np.zeros(0)
    return rep, layer, snap
