"""The multi-step synthetic decode driver on the GPU against its oracle twin.
The decoding problems are screened (parity.screen_decode): every sequence's
oracle decode clears the decision margins of parity.py at every step, so the
two decode independently and must agree on every step of every sequence;
invariants (progress, termination, commits) on every rule; the whole decode
replayed as one CUDA graph equals the eager run."""
import numpy as np
import pytest

import synth
from decode_ref import PRM_DEFAULT, oracle_decode
from parity import (MARGIN, ORDER_MARGIN, cap_margin_failures, dapd_margin_failures, screen_decode,
                    threshold_margin_failures)

pytestmark = pytest.mark.gpu

PRM = PRM_DEFAULT
CFG = synth.DecodeConfig(batch=8, blk=32, vocab=2048)


def _margin_ok(rule, o, masked, sel, b):
    """True when every decision of sequence b in this oracle step clears the
    parity margins (1e-3 on threshold tests, a relative 1e-3 on orders)."""
    blk = CFG.blk
    c = o["conf"].reshape(CFG.batch, blk)[b]
    m = masked[b]
    if m.sum() == 0:
        return True
    if rule == "threshold":
        return not threshold_margin_failures(c, m, PRM["tau"])
    if rule in ("factor", "topk"):
        cm = np.sort(c[m > 0])[::-1].astype(np.float32)
        n = int(sel[b].sum())
        if n < len(cm) and (cm[n - 1] - cm[n]) < ORDER_MARGIN * cm[n - 1]:
            return False
        if rule == "factor":
            lhs = np.arange(2, len(cm) + 2, dtype=np.float32) * (np.float32(1) - cm)
            return not np.any(np.abs(lhs - np.float32(PRM["factor_f"])) < MARGIN)
        return True
    if rule == "cap":
        r = o["cap"]
        scfg = synth.scaled(synth.CONFIGS["tiny"], tau_low=PRM["tau_low"], gamma=PRM["gamma"], p_max=blk)
        return not cap_margin_failures(scfg, c, m, r["D"][b], blk)
    r = o["dapd"]
    scfg = synth.scaled(synth.CONFIGS["tiny"], tau_edge=PRM["tau_edge"], blk=blk)
    return not dapd_margin_failures(scfg, c, m, r["s"][b], r["dtilde"][b])


def _sequence_ok(rule):
    def ok(twin, b):
        olog, ostats, _ = twin
        return all(_margin_ok(rule, o, m, olog[k], b) for k, (o, m) in enumerate(ostats) if m[b].sum() > 0)
    return ok


@pytest.mark.parametrize("rule", ["threshold", "factor", "topk", "cap", "dapd"])
def test_driver_matches_oracle_twin(rule):
    """GPU and oracle decode the screened problem independently; every step
    of every sequence agrees, and so do the final tokens and step counts."""
    from diffusion_decoding_token_gb300.driver import SyntheticDecoder
    prob, (olog, ostats, otok) = screen_decode(CFG, 17, lambda p: oracle_decode(p, rule, CFG.blk, PRM),
                                               _sequence_ok(rule))
    dec = SyntheticDecoder(prob, rule, **PRM)
    glog = []
    res = dec.run(log=glog)
    assert res["status"] == 0
    compared = 0
    for b in range(CFG.batch):
        for k, (o, m) in enumerate(ostats):
            if m[b].sum() == 0:
                break
            assert k < len(glog), (b, k)
            np.testing.assert_array_equal(glog[k][b], olog[k][b], err_msg=f"sequence {b} step {k}")
            compared += 1
        np.testing.assert_array_equal(res["tokens"][b], otok[b])
        assert res["steps"][b] == sum(1 for _, m in ostats if m[b].sum() > 0)
    # invariants on the GPU run alone: progress on every active sequence, commits only at masked positions
    masked = np.ones((CFG.batch, CFG.blk), np.uint8)
    for k, g in enumerate(glog):
        active = masked.sum(-1) > 0
        assert np.all(g.sum(-1)[active] >= 1) and not np.any(g & (1 - masked)), f"step {k}"
        masked = masked * (1 - g)
    assert masked.sum() == 0 and res["unfinished"] == 0
    assert (res["steps"] <= CFG.blk).all() and (res["steps"] >= 1).all()
    print(f"{rule}: mean steps {res['mean_steps']:.2f}, error rate {res['error_rate']:.3f}, "
          f"sequence-steps compared {compared} (all), redrawn sequences {int((prob['attempts'] > 0).sum())}")


@pytest.mark.parametrize("rule", ["threshold", "topk", "cap", "dapd", "revocable"])
def test_whole_decode_graph_equals_eager_run(rule):
    from diffusion_decoding_token_gb300.driver import SyntheticDecoder
    prob = synth.decode_problem(CFG, seed=23)
    a = SyntheticDecoder(prob, rule, **PRM).run()
    dec = SyntheticDecoder(prob, rule, **PRM)
    b = dec.run(graph=True)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_array_equal(a["steps"], b["steps"])
    dec.reset()
    c = dec.run(graph=True)                      # a replay from the reset state repeats the decode
    np.testing.assert_array_equal(c["tokens"], b["tokens"])


# A threshold decision (REPLACE, drafting) is compared when the oracle's value
# clears the threshold by MARGIN, a seed-score ranking when the k-th and
# (k+1)-th scores are MARGIN apart (the score's fp32 error from the GPU's
# confidence, influence and KL is far below it).
CONF_TOL = MARGIN
SCORE_TOL = MARGIN


def _revocable_margin_ok(rec, b, prm):
    """Every decision of sequence b in this oracle step clears the margins."""
    c, m = rec["conf"][b], rec["masked"][b]
    if m.sum() == 0:
        return True
    verified = (rec["seed"][b] > 0) & (m == 0) & (rec["argmax"][b] != rec["tok"][b])
    if np.any(np.abs(c[verified] - prm["tau_replace"]) < CONF_TOL):
        return False
    if np.any(np.abs(c[m > 0] - prm["tau_draft"]) < CONF_TOL):
        return False
    cand = np.sort(c[(m > 0) & (c > prm["tau_draft"])])[::-1]
    if len(cand) == 0 and not _gap_ok(np.sort(c[m > 0])[::-1], 1):
        return False
    if prm["draft_budget"] > 0 and not _gap_ok(cand, prm["draft_budget"]):
        return False
    # the next seeds: the k-th and (k+1)-th best scores must be apart
    out = rec["outcome"][b]
    masked_after = ((m > 0) & (out != 1)) | (out == 4)
    remasks = rec["remasks"][b] + (out == 4)
    t = rec["t"]
    elig = ~masked_after & (t - rec["last_seed"][b] > prm["cooldown"]) & (remasks < prm["remask_budget"])
    score = prm["w_unc"] * (1 - c) + prm["w_infl"] * rec["infl"][b] - prm["w_drift"] * rec["kl"][b]
    s = np.sort(score[elig])[::-1]
    n = len(s)
    k = min(n, int(np.ceil(np.float32(np.sqrt(np.float32(n))) * np.float32(prm["pi"]))))
    return not (0 < k < n and s[k - 1] - s[k] < SCORE_TOL)


def _gap_ok(sorted_desc, cut):
    return not (0 < cut < len(sorted_desc) and
                sorted_desc[cut - 1] - sorted_desc[cut] < ORDER_MARGIN * abs(sorted_desc[cut - 1]))


def test_revocable_driver_matches_oracle_twin():
    """GPU and oracle decode the screened problem independently; the outcome
    codes of every step of every sequence agree, and so do the final tokens."""
    from decode_ref import REVOCABLE_DEFAULT, revocable_decode
    from diffusion_decoding_token_gb300.driver import SyntheticDecoder

    def twin(p):
        otrace, ostate = revocable_decode(p, 3 * CFG.blk, REVOCABLE_DEFAULT)
        for k, rec in enumerate(otrace):
            rec["t"] = k
        return otrace, ostate

    def ok(tw, b):
        return all(_revocable_margin_ok(rec, b, REVOCABLE_DEFAULT) for rec in tw[0] if rec["masked"][b].sum() > 0)

    prob, (otrace, ostate) = screen_decode(CFG, 29, twin, ok)
    dec = SyntheticDecoder(prob, "revocable", **PRM)
    assert dec.max_steps == 3 * CFG.blk
    glog = []
    res = dec.run(log=glog)
    assert res["status"] == 0 and res["unfinished"] == 0
    compared = 0
    for b in range(CFG.batch):
        for k, rec in enumerate(otrace):
            if rec["masked"][b].sum() == 0:
                break
            assert k < len(glog), (b, k)
            np.testing.assert_array_equal(glog[k][b], rec["outcome"][b], err_msg=f"sequence {b} step {k}")
            compared += 1
        np.testing.assert_array_equal(res["tokens"][b], ostate["tok"][b])
        assert res["steps"][b] == sum(1 for rec in otrace if rec["masked"][b].sum() > 0)
    # the revisions fix decoys: fewer wrong tokens than the plain threshold rule
    thr = SyntheticDecoder(prob, "threshold", **PRM).run()
    print(f"revocable: mean steps {res['mean_steps']:.2f}, error rate {res['error_rate']:.3f} "
          f"(threshold {thr['error_rate']:.3f}), revisions {res['revisions']}, remasks {res['remasks']}, "
          f"flip-flops {res['flipflops']}, sequence-steps compared {compared} (all)")
    assert res["error_rate"] <= thr["error_rate"]
