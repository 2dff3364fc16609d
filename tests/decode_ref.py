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
