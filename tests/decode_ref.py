"""Oracle-side twin of the synthetic decode driver (tests only): the same
stand-in model in numpy fp32, the oracle's row statistics and rules, the same
commit.  Returns the per-step selections and the oracle values needed for
margin checks."""
import numpy as np

import oracle

PRM_DEFAULT = dict(tau=0.9, factor_f=1.0, topk_k=2, tau_low=0.8, tau_high=0.95, gamma=-16.0, tau_edge=0.05,
                   bulk_conf=0.9, bulk_frac=0.5)


def model_logits(problem, logits, masked):
    cfg = problem["cfg"]
    B, blk = cfg.batch, cfg.blk
    adj = problem["links"].astype(np.int32)
    deg = np.maximum(adj.sum(-1), 1).astype(np.float32).reshape(-1)
    decoded = (masked == 0).astype(np.int32)
    cnt = (adj * decoded[:, None, :]).sum(-1).reshape(-1)
    s = cnt.astype(np.float32) / deg
    c0 = np.float32(problem["c0"])
    zt = (c0 + problem["u"]).astype(np.float32).reshape(-1) + np.float32(cfg.kappa) * s
    zd = c0 + problem["v"].reshape(-1) * (np.float32(1.0) - s)
    rows = np.arange(B * blk)
    logits[rows, problem["target"].reshape(-1)] = zt
    logits[rows, problem["decoy"].reshape(-1)] = zd


def oracle_step(problem, masked, rule, prm):
    """One step from the given mask: the model, the oracle's row statistics
    and rule.  Returns (selected, stats) with the rule's extra outputs."""
    cfg = problem["cfg"]
    B, blk = cfg.batch, cfg.blk
    logits = problem["base"].copy()
    model_logits(problem, logits, masked)
    o = oracle.row_stats(logits)
    conf = o["conf"].reshape(B, blk)
    if rule == "threshold":
        sel, _ = oracle.select_threshold(conf, masked, prm["tau"])
    elif rule == "factor":
        sel, _ = oracle.select_factor(conf, masked, prm["factor_f"])
    elif rule == "topk":
        sel, _ = oracle.select_topk(conf, masked, prm["topk_k"])
    elif rule == "cap":
        r = oracle.cap_select(logits, o["argmax"].reshape(B, blk), conf, o["lse"].reshape(B, blk), masked,
                              prm["tau_low"], prm["tau_high"], prm["gamma"], blk)
        sel = r["selected"]
        o["cap"] = r
    else:
        r = oracle.dapd(problem["attn"], masked, conf, prm["tau_edge"], prm["bulk_conf"], prm["bulk_frac"],
                        dtype=oracle.F16)
        sel = r["selected"]
        o["dapd"] = r
    return sel, o


def oracle_decode(problem, rule, max_steps, prm):
    """The whole decode on the oracle side: per-step selections, the step's
    (stats, mask) and the committed tokens."""
    cfg = problem["cfg"]
    B, blk = cfg.batch, cfg.blk
    masked = np.ones((B, blk), np.uint8)
    tok = np.full((B, blk), -1, np.int64)
    log, stats = [], []
    for _ in range(max_steps):
        if masked.sum() == 0:
            break
        sel, o = oracle_step(problem, masked, rule, prm)
        stats.append((o, masked.copy()))
        log.append(sel.copy())
        tok = np.where(sel > 0, o["argmax"].reshape(B, blk), tok)
        masked = masked * (1 - sel)
    return log, stats, tok


# ---------------------------------------------------------------------------
# DepCap block loop (DepCap, "Methodology"): the oracle side of
# DepCapDecoder.  The problem's cfg.blk is the generation length N.
# ---------------------------------------------------------------------------
DEPCAP_DEFAULT = dict(L_max=32, lam=1.2, L_min=8, smooth_w=1, norm_mode=0, tau_low=0.8, tau_high=0.95, gamma=-16.0)


def full_logits(problem, masked):
    lg = problem["base"].copy()
    model_logits(problem, lg, masked)
    return lg


def depcap_step(problem, state, prm):
    """One step of the block loop from ``state`` (masked [B,N], cursor [B],
    blen [B] (0 = pick a block), cold [B], snap_masked [B,N]: the mask at the
    forward pass that became the sequence's snapshot, or None before the
    first).  Returns dict(need, new_len, score, blen, sel, pos, stats, cap)."""
    cfg = problem["cfg"]
    B, N, Lm = cfg.batch, cfg.blk, prm["L_max"]
    masked, cursor = state["masked"], state["cursor"]
    cur = full_logits(problem, masked)
    pos = np.minimum(cursor[:, None] + np.arange(Lm)[None, :], N - 1)
    rows = (np.arange(B)[:, None] * N + pos).reshape(-1)
    prev = np.empty((B * Lm, cfg.vocab), np.float32)
    snap_all = masked.copy()       # a sequence's rows depend on its own mask only
    have = np.zeros(B, bool)
    for b in range(B):
        if state["snap_masked"][b] is not None:
            snap_all[b], have[b] = state["snap_masked"][b], True
    snap = full_logits(problem, snap_all) if have.any() else cur
    for b in range(B):
        src = snap if have[b] else cur
        prev[b * Lm:(b + 1) * Lm] = src[rows[b * Lm:(b + 1) * Lm]]
    win = cur[rows]
    o = oracle.row_stats(win, prev)
    window_len = np.clip(N - cursor, 0, Lm)
    active = cursor < N
    need = active & (state["blen"] == 0)
    new_len, score = oracle.depcap_boundary(o["kl"].reshape(B, Lm), o["entropy"].reshape(B, Lm), prm["lam"],
                                            prm["L_min"], prm["smooth_w"], prm["norm_mode"],
                                            cold_start=state["cold"], window_len=window_len)
    blen = np.where(need, new_len, state["blen"])
    in_block = np.arange(Lm)[None, :] < blen[:, None]
    mwin = (np.take_along_axis(masked, pos, 1) * in_block).astype(np.uint8)
    r = oracle.cap_select(win, o["argmax"].reshape(B, Lm), o["conf"].reshape(B, Lm), o["lse"].reshape(B, Lm),
                          mwin, prm["tau_low"], prm["tau_high"], prm["gamma"], Lm, scope_len=blen)
    return dict(need=need, new_len=new_len, score=score, blen=blen, sel=r["selected"], pos=pos, stats=o, cap=r,
                mwin=mwin, window_len=window_len)


def depcap_commit(state, out, tok):
    """Commit a step's selection (given as ``out``'s sel/pos/blen/need) into
    ``state`` and ``tok``; returns the new state."""
    B = len(state["cursor"])
    masked = state["masked"].copy()
    snap = list(state["snap_masked"])
    for b in range(B):
        if out["need"][b]:
            snap[b] = state["masked"][b].copy()
        for k in np.nonzero(out["sel"][b])[0]:
            p = out["pos"][b, k]
            masked[b, p] = 0
            tok[b, p] = out["argmax"][b, k]
    cursor, blen = state["cursor"].copy(), out["blen"].copy()
    for b in range(B):
        if cursor[b] < masked.shape[1] and blen[b] > 0 and not masked[b, cursor[b]:cursor[b] + blen[b]].any():
            cursor[b] += blen[b]
            blen[b] = 0
    cold = state["cold"] * (1 - out["need"].astype(np.uint8))
    return dict(masked=masked, cursor=cursor, blen=blen, cold=cold, snap_masked=snap)


def depcap_initial(problem):
    cfg = problem["cfg"]
    B, N = cfg.batch, cfg.blk
    return dict(masked=np.ones((B, N), np.uint8), cursor=np.zeros(B, np.int64), blen=np.zeros(B, np.int64),
                cold=np.ones(B, np.uint8), snap_masked=[None] * B)


def depcap_decode(problem, prm=DEPCAP_DEFAULT, max_steps=None, trace=None):
    """The whole block loop on the oracle side.  Returns (steps [B], tok,
    blocks: per sequence the list of (start, length)); ``trace``, a list,
    receives (state before the step, the step's outputs) per step."""
    cfg = problem["cfg"]
    B, N = cfg.batch, cfg.blk
    state = depcap_initial(problem)
    tok = np.full((B, N), -1, np.int64)
    steps = np.zeros(B, np.int64)
    blocks = [[] for _ in range(B)]
    for _ in range(max_steps or N):
        if (state["cursor"] >= N).all():
            break
        out = depcap_step(problem, state, prm)
        steps += state["cursor"] < N
        for b in np.nonzero(out["need"])[0]:
            blocks[b].append((int(state["cursor"][b]), int(out["blen"][b])))
        out["argmax"] = out["stats"]["argmax"].reshape(B, prm["L_max"])
        if trace is not None:
            trace.append((state, out))
        state = depcap_commit(state, out, tok)
    return steps, tok, blocks


# ---------------------------------------------------------------------------
# Revocable decoding (COVER page): the oracle side of SyntheticDecoder's
# "revocable" rule.
# ---------------------------------------------------------------------------
REVOCABLE_DEFAULT = dict(tau_replace=0.9, tau_draft=0.9, draft_budget=0, w_unc=1.0, w_infl=1.0, w_drift=1.0,
                         pi=1.0, cooldown=1, remask_budget=2)


def revocable_decode(problem, max_steps, prm=REVOCABLE_DEFAULT):
    """Returns (trace, state): per step dict(masked, conf, argmax, kl, infl,
    outcome, seed_before, last_seed_before, remasks_before, tok_before) and the
    final state."""
    cfg = problem["cfg"]
    B, blk = cfg.batch, cfg.blk
    state = oracle.revocable_init(B, blk)
    prev = problem["base"].copy()
    trace = []
    for t in range(max_steps):
        if state["masked"].sum() == 0:
            break
        cur = full_logits(problem, state["masked"])
        o = oracle.row_stats(cur, prev)
        prev = cur
        infl = oracle.attention_influence(problem["attn"], state["masked"], dtype=oracle.F16)
        rec = dict(masked=state["masked"].copy(), seed=state["seed"].copy(), last_seed=state["last_seed"].copy(),
                   remasks=state["remasks"].copy(), tok=state["tok"].copy(), last_tok=state["last_tok"].copy(),
                   conf=o["conf"].reshape(B, blk), argmax=o["argmax"].reshape(B, blk), kl=o["kl"].reshape(B, blk),
                   infl=infl)
        r = oracle.revocable_step(o["argmax"].reshape(B, blk), o["conf"].reshape(B, blk), state, t,
                                  influence=infl, drift=o["kl"].reshape(B, blk), **prm)
        rec["outcome"] = r["outcome"]
        trace.append(rec)
    return trace, state
