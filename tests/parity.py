"""Helpers for the GPU-vs-oracle parity tests.

Inputs come from ``synth`` (seeded); expected values only from ``oracle``.
Decision margins: a float decision is compared bit-exactly only when the
oracle's value sits far enough from the boundary that fp32 rounding on the GPU
cannot flip it; otherwise the GPU result is checked for validity (it must be a
result the rule could give under some resolution of the near-tie).

Margins used (derived from the fp32 error of each quantity):
* threshold tests (conf vs tau, tau_low, tau_high, bulk_conf): |c - t| >= 1e-3
* CAP conflict test: |D_ij - gamma| >= 1e-3
* DepGA sign test: |S_k| >= 1e-3 for every k up to the first negative
* orderings that can change a greedy result (conf order of conflicting CAP
  pairs, DAPD key order of tau-adjacent pairs, the top-1/top-2 gap of a
  fallback, the pool cut): relative gap >= ORDER_TOL.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from brute import is_independent, is_maximal

ORDER_TOL = 1e-5
THRESH_TOL = 1e-3
ATOL = 1e-4
RTOL = 1e-4

TORCH_DT = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}


def to_torch(arr: np.ndarray, code: int, device) -> torch.Tensor:
    if code == synth.F32:
        return torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device)
    return t.view(TORCH_DT[code])


class DeviceWorkload:
    """Device copies of a synth.Workload; attention is laid out full size
    [B, L, H, N, N] with the block submatrix scattered in (zeros elsewhere)."""

    def __init__(self, w: synth.Workload, device="cuda", compact_attn=False):
        cfg = w.cfg
        self.w = w
        self.cfg = cfg
        self.cur = to_torch(w.cur, cfg.logit_dtype, device)
        self.prev = to_torch(w.prev, cfg.logit_dtype, device)
        self.masked = torch.from_numpy(w.masked).to(device)
        self.row_index = None
        if cfg.masked_count >= 0:
            ri = np.nonzero(w.masked.reshape(-1))[0].astype(np.int32)
            self.row_index = torch.from_numpy(ri).to(device)
        self.attn = None
        self.block_start = cfg.block_start
        if w.attn is not None:
            sub = to_torch(w.attn, cfg.attn_dtype, device)
            if compact_attn:
                self.attn = sub
                self.block_start = 0
            else:
                B, L, H, blk, _ = sub.shape
                N, bs = cfg.seq_len, cfg.block_start
                full = torch.zeros((B, L, H, N, N), dtype=sub.dtype, device=device)
                full[:, :, :, bs:bs + blk, bs:bs + blk] = sub
                self.attn = full


def row_index_np(w: synth.Workload):
    if w.cfg.masked_count < 0:
        return None
    return np.nonzero(w.masked.reshape(-1))[0].astype(np.int32)


def oracle_stats(w: synth.Workload):
    cfg = w.cfg
    code = None if cfg.logit_dtype == synth.F32 else cfg.logit_dtype
    return oracle.row_stats(w.cur, w.prev, dtype=code, row_index=row_index_np(w), n_out=cfg.batch * cfg.blk)


def gpu_stats(dw: DeviceWorkload, status=None):
    import diffusion_decoding_token_gb300 as dlm
    n = dw.cur.shape[0]
    out = dlm.RowStats(*[torch.zeros(n, dtype=dt, device=dw.cur.device) for dt in
                         (torch.int32, torch.float32, torch.float32, torch.float32, torch.float32, torch.float32)])
    return dlm.row_stats(dw.cur, dw.prev, row_index=dw.row_index, out=out, status=status)


def close(g, o, atol=ATOL, rtol=RTOL):
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    return np.abs(g - o) <= atol + rtol * np.abs(o)


# ------------------------------------------------------------------ margins
def _fallback_gap_ok(c, masked):
    cm = np.sort(c[masked.astype(bool)])[::-1]
    return len(cm) < 2 or (cm[0] - cm[1]) >= ORDER_TOL * max(abs(cm[0]), 1e-30)


def threshold_margin_ok(c, masked, tau):
    m = masked.astype(bool)
    if np.any(np.abs(c[m] - tau) < THRESH_TOL):
        return False
    if not np.any(c[m] > tau):
        return _fallback_gap_ok(c, masked)
    return True


def boundary_margin_ok(score):
    neg = np.nonzero(score < 0)[0]
    kstar = int(neg[0]) if len(neg) else len(score)
    upto = score[:min(kstar + 1, len(score))]
    return not np.any(np.abs(upto) < THRESH_TOL)


def cap_margin_ok(cfg, c, masked, D, pool, pool_n, scope, conf_tol=THRESH_TOL):
    """``conf_tol``: margin of the tau_low test (f32 logits may use the
    row-stats parity tolerance, 1e-4, instead of THRESH_TOL)."""
    m = masked.astype(bool).copy()
    m[scope:] = False
    for t in (cfg.tau_low,):
        if np.any(np.abs(c[m] - t) < conf_tol):
            return False
    p = [int(x) for x in pool[:pool_n]]
    if not p:
        cm = c.copy()
        cm[~m] = -np.inf
        return _fallback_gap_ok(np.where(m, c, -np.inf), m.astype(np.uint8)) if m.any() else True
    cand = np.nonzero(m & (c >= cfg.tau_low))[0]
    if len(cand) > cfg.p_max:
        srt = np.sort(c[cand])[::-1]
        if (srt[cfg.p_max - 1] - srt[cfg.p_max]) < ORDER_TOL * srt[cfg.p_max - 1]:
            return False
    for a in p:
        for b in p:
            if a < b:
                if abs(D[a, b] - cfg.gamma) < THRESH_TOL:
                    return False
                if D[a, b] > cfg.gamma and abs(c[a] - c[b]) < ORDER_TOL * max(c[a], c[b]):
                    return False
    return True


def dapd_margin_ok(cfg, c, masked, s, dtilde, order_mode=0, key_tol=ORDER_TOL):
    m = masked.astype(bool)
    M = int(m.sum())
    if np.float32(M) < np.float32(cfg.bulk_frac) * np.float32(cfg.blk):
        return threshold_margin_ok(c, masked, cfg.bulk_conf)
    nodes = np.nonzero(m)[0]
    S = s[np.ix_(nodes, nodes)]
    if np.any(np.abs(S - cfg.tau_edge) < 1e-9 * max(cfg.tau_edge, 1e-30)):
        return False
    adj = (S > np.float32(cfg.tau_edge)) & ~np.eye(len(nodes), dtype=bool)
    key = dtilde[nodes] * (1.0 if order_mode else c[nodes])
    ii, jj = np.nonzero(np.triu(adj, 1))
    if len(ii):
        gap = np.abs(key[ii] - key[jj]) / np.maximum(np.maximum(np.abs(key[ii]), np.abs(key[jj])), 1e-300)
        if np.any(gap < key_tol):
            return False
    return True


# -------------------------------------------------------------- validity
def greedy_valid(adj, sel, order_key, universe, tol):
    """sel is independent, maximal, and every left-out node has a kept
    neighbour not ranked clearly after it."""
    if not is_independent(adj, sel) or not is_maximal(adj, sel, universe):
        return False
    for v in universe:
        if v in sel:
            continue
        if not any(adj[v, u] and order_key[u] >= order_key[v] * (1 - tol) for u in sel):
            return False
    return True
