"""Helpers for the GPU-vs-oracle parity tests.

Inputs come from ``synth`` (seeded); expected values only from ``oracle``.

Decision margins.  A floating-point value that decides an integer outcome (a
threshold test, an order between two positions) is compared bit for bit only
when the oracle's value sits far enough from the boundary that the GPU's fp32
arithmetic cannot flip it:

* every threshold-type test -- conf against tau, tau_low, tau_high and the
  late-phase 0.9; the CAP conflict score D_ij against gamma; the DAPD score
  s_ij against tau; the DepGA score S_k against 0 up to the first negative --
  must clear ``MARGIN`` = 1e-3 (absolute);
* every order comparison that can change a greedy result -- the confidence
  order of two conflicting CAP pool members of one tier, the DAPD key order of
  two tau-adjacent nodes, the top-1/top-2 gap of a fallback, the pool cut --
  must clear a relative gap of ``order_margin(cfg, rule)``: 1e-3, except on
  the stress graph workload, where 256 positions with about 150 planted
  conflicts and 1100 tau-edges make a 1e-3 gap unreachable (a sequence
  clears it with probability about e^-20).  There each rule's gap is set
  from the error of the values it orders: CAP orders confidences near 1,
  whose fp32 error is ~1e-7 (the sum S = 1 + eps is quantised at 1.2e-7),
  so its gap is 1e-5; DAPD orders d~ * conf over all positions, and the
  GPU's fp32 confidence carries up to ~3e-6 relative error where many
  logits share the mass, so its gap is 1e-4.  Both stay 10x or more above
  the error the pipeline test measures.

``screen`` draws a workload and redraws every sequence that misses a margin
(``Workload.replace_sequence`` with the next attempt number, up to
``MAX_ATTEMPTS``), then fails loudly.  On a screened workload every decision
of every sequence is compared exactly.

For unscreened draws, ``*_outcomes`` enumerate every result the rule can give
when each ambiguous decision (inside ``MARGIN`` for threshold tests, inside
``FP32_ORDER_BAND`` for orders) is resolved either way; the GPU's result must
be one of them.  A greedy maximal independent set depends only on which end
of each edge comes first, so an order ambiguity is a flip of that edge's
orientation (acyclic resolutions only).
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
import torch

import oracle
import synth

MARGIN = 1e-3
ORDER_MARGIN = 1e-3
FP32_ORDER_BAND = 1e-5
MAX_ATTEMPTS = 64
RULES = ("threshold", "boundary", "cap", "dapd")
ORDER_MARGIN_BY_WORKLOAD = {"stress_graph": {"cap": 1e-5, "dapd": 1e-4}}
ATOL = 1e-4
RTOL = 1e-4
MAX_AMBIGUOUS = 14

# kept for the driver tests: the older names of the two margins
THRESH_TOL = MARGIN
ORDER_TOL = FP32_ORDER_BAND

TORCH_DT = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}
GOLDEN_ATTEMPTS = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "screened_attempts.json")


def order_margin(cfg, rule: str) -> float:
    return ORDER_MARGIN_BY_WORKLOAD.get(cfg.name, {}).get(rule, ORDER_MARGIN)


def order_margins(cfg) -> dict:
    return {r: order_margin(cfg, r) for r in RULES}


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


def _code(cfg):
    return None if cfg.logit_dtype == synth.F32 else cfg.logit_dtype


def oracle_stats(w: synth.Workload):
    cfg = w.cfg
    return oracle.row_stats(w.cur, w.prev, dtype=_code(cfg), row_index=row_index_np(w), n_out=cfg.batch * cfg.blk)


def oracle_stats_seq(w: synth.Workload, b: int):
    """Oracle row statistics of sequence b alone ([blk] arrays)."""
    cfg = w.cfg
    blk = cfg.blk
    sl = slice(b * blk, (b + 1) * blk)
    ri = None
    if cfg.masked_count >= 0:
        ri = np.nonzero(w.masked[b])[0].astype(np.int32)
    return oracle.row_stats(w.cur[sl], w.prev[sl], dtype=_code(cfg), row_index=ri, n_out=blk)


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


def _near_rel(a, b, tol):
    return abs(a - b) < tol * max(abs(a), abs(b), 1e-300)


def _f32(x):
    return float(np.float32(x))


# ------------------------------------------------------------ the rules' ambiguities
def _top_near(c, cand, tol):
    """Candidates whose confidence is within ``tol`` (relative) of the best
    one: the possible fallbacks (the oracle takes the first of them)."""
    if not len(cand):
        return []
    best = max(float(c[i]) for i in cand)
    return [int(i) for i in cand if _near_rel(float(c[i]), best, tol)]


def threshold_outcome_check(c, masked, t, sel, margin=MARGIN, order_tol=FP32_ORDER_BAND):
    """Is ``sel`` a result of the threshold rule (c > t, top-1 fallback) under
    some resolution of the decisions within the bands?  Returns (ok, unique)."""
    m = np.nonzero(masked)[0]
    if not len(m):
        return (not np.any(sel)), True
    near = {int(i) for i in m if abs(c[i] - t) < margin}
    clear = {int(i) for i in m if c[i] - t >= margin}
    s = {int(i) for i in np.nonzero(sel)[0]}
    fb = set(_top_near(c, m, order_tol))
    unique = not near and (bool(clear) or len(fb) == 1)
    if clear:
        return (clear <= s <= clear | near), unique
    if s and s <= near:                       # some near-threshold positions resolved above
        return True, unique
    return (len(s) == 1 and s <= fb), unique  # nothing above: one fallback position


def threshold_margin_failures(c, masked, t, margin=MARGIN, order_tol=ORDER_MARGIN):
    m = np.nonzero(masked)[0]
    if not len(m):
        return []
    f = [f"conf {c[i]:.6f} of position {i} within {margin} of {t}" for i in m if abs(c[i] - t) < margin]
    if not any(c[i] > t for i in m) and len(_top_near(c, m, order_tol)) > 1:
        f.append("fallback top-1/top-2 near tie")
    return f


def boundary_range(score, L_min, margin=MARGIN):
    """Range [lo, hi] of the first-negative index k* that fp32 rounding of the
    scores can give: every S_k before lo is at least ``margin`` above 0, and
    S_hi is at least ``margin`` below it (hi = L_window when no such k)."""
    Lw = len(score)
    lo = next((k for k in range(Lw) if score[k] < margin), Lw)
    hi = next((k for k in range(Lw) if score[k] <= -margin), Lw)
    clip = lambda k: min(max(k, L_min), Lw)  # noqa: E731
    return clip(lo), clip(hi)


def boundary_margin_failures(score, margin=MARGIN):
    neg = np.nonzero(score < 0)[0]
    kstar = int(neg[0]) if len(neg) else len(score)
    upto = score[:min(kstar + 1, len(score))]
    return [f"S_{k} = {v:.2e} within {margin} of 0" for k, v in enumerate(upto) if abs(v) < margin]


def _greedy_dag(nodes, edges, before):
    """Greedy maximal independent set when each edge (u, v) is oriented by
    ``before(u, v)`` (True: u first).  None if the orientation has a cycle."""
    idx = {v: k for k, v in enumerate(nodes)}
    indeg = [0] * len(nodes)
    out = [[] for _ in nodes]
    for u, v in edges:
        a, b = (u, v) if before(u, v) else (v, u)
        out[idx[a]].append(idx[b])
        indeg[idx[b]] += 1
    ready = sorted(k for k in range(len(nodes)) if indeg[k] == 0)
    kept, blocked, seen = set(), set(), 0
    while ready:
        k = ready.pop()
        seen += 1
        if k not in blocked:
            kept.add(nodes[k])
            blocked.update(out[k])
        for j in out[k]:
            indeg[j] -= 1
            if indeg[j] == 0:
                ready.append(j)
    return frozenset(kept) if seen == len(nodes) else None


def cap_ambiguities(cfg, c, masked, D, scope, margin=MARGIN, order_tol=ORDER_MARGIN):
    """Ambiguous decisions of CAP on one sequence.  ``c``: oracle confidences
    (fp64); ``D``: oracle D_ij over every candidate pair (NaN elsewhere),
    from a pool taken down to tau_low - margin so that near-threshold
    candidates have scores.  Returns a dict of the determined parts and the
    lists of ambiguous items."""
    cand = [i for i in range(min(scope, len(c))) if masked[i]]
    member = {i: _f32(c[i]) >= cfg.tau_low for i in cand}
    amb_member = [i for i in cand if abs(c[i] - cfg.tau_low) < margin]
    pool_any = [i for i in cand if member[i] or i in amb_member]
    tier = {i: _f32(c[i]) >= cfg.tau_high for i in pool_any}
    amb_tier = [i for i in pool_any if abs(c[i] - cfg.tau_high) < margin]
    edges, amb_edge, amb_orient = [], [], []
    for a, b in itertools.combinations(pool_any, 2):
        d = D[a, b]
        if np.isnan(d):
            continue
        conflict = _f32(d) > cfg.gamma
        near = abs(d - cfg.gamma) < margin
        if conflict or near:
            edges.append((a, b))
            if near:
                amb_edge.append((a, b))
            same_tier_possible = tier[a] == tier[b] or a in amb_tier or b in amb_tier
            if same_tier_possible and _near_rel(c[a], c[b], order_tol):
                amb_orient.append((a, b))
    pool_n = sum(1 for i in cand if member[i])
    cut_amb = False
    if pool_n + len([i for i in amb_member if not member[i]]) > cfg.p_max:
        srt = sorted((float(c[i]) for i in pool_any), reverse=True)
        k = cfg.p_max
        cut_amb = bool(amb_member) or (len(srt) > k and _near_rel(srt[k - 1], srt[k], order_tol))
    fallback = _top_near(c, cand, order_tol)
    amb_fallback = (pool_n == 0 or bool(amb_member)) and len(fallback) > 1
    return dict(cand=cand, member=member, tier=tier, edges=edges, amb_member=amb_member, amb_tier=amb_tier,
                amb_edge=amb_edge, amb_orient=amb_orient, cut_amb=cut_amb, fallback=fallback,
                amb_fallback=amb_fallback)


def cap_margin_failures(cfg, c, masked, D, scope, margin=MARGIN, order_tol=ORDER_MARGIN):
    a = cap_ambiguities(cfg, c, masked, D, scope, margin, order_tol)
    f = [f"CAP: {len(a[k])} {k}" for k in ("amb_member", "amb_tier", "amb_edge", "amb_orient") if a[k]]
    if a["cut_amb"]:
        f.append("CAP: pool cut near tie")
    if a["amb_fallback"]:
        f.append("CAP: fallback near tie")
    return f


def cap_outcomes(cfg, c, masked, D, scope, margin=MARGIN, order_tol=FP32_ORDER_BAND):
    """Every CAP selection (as a frozenset of positions) that some resolution
    of the ambiguous decisions gives."""
    a = cap_ambiguities(cfg, c, masked, D, scope, margin, order_tol)
    assert not a["cut_amb"], "an ambiguous pool cut is not enumerated"
    items = ([("m", i) for i in a["amb_member"]] + [("t", i) for i in a["amb_tier"]] +
             [("e", e) for e in a["amb_edge"]] + [("o", e) for e in a["amb_orient"]])
    assert len(items) <= MAX_AMBIGUOUS, f"{len(items)} ambiguous CAP decisions"
    c32 = {i: _f32(c[i]) for i in a["cand"]}
    outs = set()
    for bits in itertools.product((False, True), repeat=len(items)):
        flip = {it: bit for it, bit in zip(items, bits)}
        member = {i: a["member"][i] ^ flip.get(("m", i), False) for i in a["cand"]}
        tier = {i: a["tier"][i] ^ flip.get(("t", i), False) for i in a["tier"]}
        pool = sorted((i for i in a["cand"] if member[i]), key=lambda i: (-c32[i], i))[:cfg.p_max]
        if not pool:
            outs.update(frozenset([j]) for j in (a["fallback"] if len(a["fallback"]) else []))
            continue
        ps = set(pool)
        edges = [e for e in a["edges"] if e[0] in ps and e[1] in ps and not flip.get(("e", e), False)]

        def before(u, v, tier=tier, flip=flip):
            first = (not tier[u], -c32[u], u) < (not tier[v], -c32[v], v)
            return first ^ flip.get(("o", (u, v) if u < v else (v, u)), False)

        s = _greedy_dag(pool, edges, before)
        if s is not None:
            outs.add(s)
    return outs


def dapd_ambiguities(cfg, c, masked, s, dtilde, order_mode=0, margin=MARGIN, order_tol=ORDER_MARGIN):
    """Ambiguous decisions of the DAPD graph path on one sequence (oracle s,
    d~ in fp64; the kernel decides the edge test and key order exactly)."""
    nodes = [int(i) for i in np.nonzero(masked)[0]]
    key = {i: float(dtilde[i]) * (1.0 if order_mode else float(c[i])) for i in nodes}
    tau = _f32(cfg.tau_edge)                 # the call passes tau as a float
    edges, amb_edge, amb_orient = [], [], []
    for a, b in itertools.combinations(nodes, 2):
        v = s[a, b]
        near = abs(v - tau) < margin
        if v > tau or near:
            edges.append((a, b))
            if near:
                amb_edge.append((a, b))
            if _near_rel(key[a], key[b], order_tol):
                amb_orient.append((a, b))
    return dict(nodes=nodes, key=key, edges=edges, amb_edge=amb_edge, amb_orient=amb_orient)


def dapd_late(cfg, masked):
    M = int(np.sum(masked))
    return np.float32(M) < np.float32(cfg.bulk_frac) * np.float32(cfg.blk)


def dapd_margin_failures(cfg, c, masked, s, dtilde, order_mode=0, margin=MARGIN, order_tol=ORDER_MARGIN):
    if dapd_late(cfg, masked):
        return threshold_margin_failures(c, masked, cfg.bulk_conf, margin, order_tol)
    a = dapd_ambiguities(cfg, c, masked, s, dtilde, order_mode, margin, order_tol)
    return [f"DAPD: {len(a[k])} {k}" for k in ("amb_edge", "amb_orient") if a[k]]


def dapd_outcomes(cfg, c, masked, s, dtilde, order_mode=0, margin=MARGIN, order_tol=FP32_ORDER_BAND):
    """Every DAPD graph-path selection some resolution of the ambiguous
    decisions gives (the late phase is checked by threshold_outcome_check)."""
    a = dapd_ambiguities(cfg, c, masked, s, dtilde, order_mode, margin, order_tol)
    items = [("e", e) for e in a["amb_edge"]] + [("o", e) for e in a["amb_orient"]]
    assert len(items) <= MAX_AMBIGUOUS, f"{len(items)} ambiguous DAPD decisions"
    key = a["key"]
    outs = set()
    for bits in itertools.product((False, True), repeat=len(items)):
        flip = {it: bit for it, bit in zip(items, bits)}
        edges = [e for e in a["edges"] if not flip.get(("e", e), False)]

        def before(u, v, flip=flip):
            first = (-key[u], u) < (-key[v], v)
            return first ^ flip.get(("o", (u, v) if u < v else (v, u)), False)

        r = _greedy_dag(a["nodes"], edges, before)
        if r is not None:
            outs.add(r)
    return outs


# ------------------------------------------------------------------ screening
def sequence_decisions(w: synth.Workload, b: int, st: dict) -> dict:
    """The oracle's rules on sequence b alone, from its statistics ``st``."""
    cfg = w.cfg
    blk = cfg.blk
    m = w.masked[b:b + 1]
    c = st["conf"]
    out = {}
    scope = None
    if "boundary" in cfg.rules:
        bl, sc = oracle.depcap_boundary(st["kl"][None], st["entropy"][None], cfg.lam, cfg.L_min)
        out["boundary"] = (int(bl[0]), sc[0])
        if cfg.name.startswith("depcap_window"):
            scope = bl
    if "cap" in cfg.rules:
        am = np.where(st["argmax"] < 0, 0, st["argmax"])[None]
        sl = slice(b * blk, (b + 1) * blk)
        args = (w.cur[sl], am, c[None], st["lse"][None], m)
        r = oracle.cap_select(*args, cfg.tau_low, cfg.tau_high, cfg.gamma, cfg.p_max, scope_len=scope,
                              dtype=_code(cfg))
        # D_ij over every candidate of the whole block, down to tau_low - margin
        wide = oracle.cap_select(*args, cfg.tau_low - MARGIN, cfg.tau_high, cfg.gamma, blk, dtype=_code(cfg))
        out["cap"] = (r, wide["D"][0], blk if scope is None else int(scope[0]))
    if "dapd" in cfg.rules:
        code = None if cfg.attn_dtype == synth.F32 else cfg.attn_dtype
        out["dapd"] = oracle.dapd(w.attn[b:b + 1], m, c[None], cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0,
                                  dtype=code)
    return out


def sequence_margin_failures(w: synth.Workload, b: int, st: dict, dec: dict | None = None,
                             margins: dict | None = None) -> list:
    """Why sequence b misses the decision margins (empty: it clears them).
    ``margins``: the order margin per rule (default order_margins(cfg))."""
    cfg = w.cfg
    dec = sequence_decisions(w, b, st) if dec is None else dec
    om = dict(order_margins(cfg), **(margins or {}))
    c, m = st["conf"], w.masked[b]
    f = []
    if "threshold" in cfg.rules:
        f += threshold_margin_failures(c, m, cfg.tau, MARGIN, om["threshold"])
    if "boundary" in cfg.rules:
        f += boundary_margin_failures(dec["boundary"][1])
    if "cap" in cfg.rules:
        _, Dw, scope = dec["cap"]
        f += cap_margin_failures(cfg, c, m, Dw, scope, MARGIN, om["cap"])
    if "dapd" in cfg.rules:
        r = dec["dapd"]
        f += dapd_margin_failures(cfg, c, m, r["s"][0], r["dtilde"][0], 0, MARGIN, om["dapd"])
    return f


def _load_attempts(cfg, seed):
    try:
        with open(GOLDEN_ATTEMPTS) as fh:
            rec = json.load(fh).get(f"{cfg.name}:{cfg.boost_mode}:{seed}")
    except (OSError, ValueError):
        return None
    if rec and len(rec["attempts"]) == cfg.batch and rec.get("order_margins") == order_margins(cfg):
        return np.asarray(rec["attempts"], np.int64)
    return None


def screen(cfg, seed: int, attempts=None, use_stored=True, log=None, margins=None):
    """A workload whose every sequence clears the decision margins.

    Starts from ``attempts`` (or the stored table written by
    tests/golden/make_screened_attempts.py, or all zeros), checks each
    sequence against the oracle, and redraws the failing ones with the next
    attempt number until they clear; fails after MAX_ATTEMPTS attempts.
    ``margins`` overrides order margins per rule (unit tests whose two sides
    order the same fp32 values need none).  Returns (workload, oracle
    statistics of the whole batch)."""
    if isinstance(cfg, str):
        cfg = synth.CONFIGS[cfg]
    if attempts is None and use_stored and not margins:
        attempts = _load_attempts(cfg, seed)
    w = synth.make(cfg, seed, attempts)
    B, blk = cfg.batch, cfg.blk
    o = oracle_stats(w)
    for b in range(B):
        while True:
            st = {k: v[b * blk:(b + 1) * blk] for k, v in o.items()}
            fails = sequence_margin_failures(w, b, st, margins=margins)
            if not fails:
                break
            nxt = int(w.attempts[b]) + 1
            if nxt >= MAX_ATTEMPTS:
                raise AssertionError(f"{cfg.name} sequence {b}: no draw of {MAX_ATTEMPTS} clears the decision "
                                     f"margins (last: {fails[:3]})")
            if log is not None:
                log.append((b, nxt - 1, fails[:3]))
            w.replace_sequence(b, nxt)
            st = oracle_stats_seq(w, b)
            for k in o:
                o[k][b * blk:(b + 1) * blk] = st[k]
    return w, o


def screen_decode(cfg, seed: int, run_twin, sequence_ok):
    """A multi-step decoding problem whose every sequence's oracle decode
    clears the margins at every step.  ``run_twin(problem)`` decodes the whole
    batch on the oracle side; ``sequence_ok(twin, b)`` says whether sequence
    b's steps all clear.  Sequences decode independently, so the failing
    ones are redrawn (next attempt number) and the batch is decoded again;
    fails after MAX_ATTEMPTS attempts.  Returns (problem, twin)."""
    attempts = np.zeros(cfg.batch, np.int64)
    for _ in range(MAX_ATTEMPTS):
        prob = synth.decode_problem(cfg, seed, attempts)
        twin = run_twin(prob)
        bad = [b for b in range(cfg.batch) if not sequence_ok(twin, b)]
        if not bad:
            return prob, twin
        attempts[bad] += 1
    raise AssertionError(f"{cfg.name}: sequences {bad} have no draw of {MAX_ATTEMPTS} that clears the margins")
