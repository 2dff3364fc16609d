"""The multi-step synthetic decode driver on the GPU against its oracle twin:
the two decode independently and every sequence's steps agree up to its first
decision inside the margins of parity.py; invariants (progress, termination, commits)
on every rule; the whole decode replayed as one CUDA graph equals the eager
run."""
import numpy as np
import pytest

import synth
from decode_ref import PRM_DEFAULT, oracle_decode
from parity import ORDER_TOL, THRESH_TOL, cap_margin_ok, dapd_margin_ok, threshold_margin_ok

pytestmark = pytest.mark.gpu

PRM = PRM_DEFAULT
CFG = synth.DecodeConfig(batch=8, blk=32, vocab=2048)


def _margin_ok(rule, o, masked, sel, b):
    """True when every decision of sequence b in this oracle step clears the
    parity margins."""
    blk = CFG.blk
    c = o["conf"].reshape(CFG.batch, blk)[b]
    m = masked[b]
    if m.sum() == 0:
        return True
    if rule == "threshold":
        return threshold_margin_ok(c, m, PRM["tau"])
    if rule in ("factor", "topk"):
        cm = np.sort(c[m > 0])[::-1].astype(np.float32)
        n = int(sel[b].sum())
        if n < len(cm) and (cm[n - 1] - cm[n]) < ORDER_TOL * cm[n - 1]:
            return False
        if rule == "factor":
            lhs = np.arange(2, len(cm) + 2, dtype=np.float32) * (np.float32(1) - cm)
            return not np.any(np.abs(lhs - np.float32(PRM["factor_f"])) < THRESH_TOL)
        return True
    if rule == "cap":
        r = o["cap"]
        scfg = synth.scaled(synth.CONFIGS["tiny"], tau_low=PRM["tau_low"], gamma=PRM["gamma"], p_max=blk)
        return cap_margin_ok(scfg, c, m, r["D"][b], r["pool"][b], r["pool_n"][b], blk, conf_tol=CONF_TOL)
    r = o["dapd"]
    scfg = synth.scaled(synth.CONFIGS["tiny"], tau_edge=PRM["tau_edge"], blk=blk)
    return dapd_margin_ok(scfg, c, m, r["s"][b], r["dtilde"][b])


@pytest.mark.parametrize("rule", ["threshold", "factor", "topk", "cap", "dapd"])
def test_driver_matches_oracle_twin(rule):
    """GPU and oracle decode independently; each sequence is compared step by
    step until its first step with a decision inside the margins, and its
    final tokens and step count when it never had one."""
    from diffusion_decoding_token_gb300.driver import SyntheticDecoder
    prob = synth.decode_problem(CFG, seed=17)
    dec = SyntheticDecoder(prob, rule, **PRM)
    glog = []
    res = dec.run(log=glog)
    assert res["status"] == 0
    olog, ostats, otok = oracle_decode(prob, rule, CFG.blk, PRM)
    compared = total = whole = 0
    for b in range(CFG.batch):
        clean = True
        for k, (o, m) in enumerate(ostats):
            if m[b].sum() == 0:
                break
            total += 1
            if not clean or not _margin_ok(rule, o, m, olog[k], b):
                clean = False
                continue
            assert k < len(glog), (b, k)
            np.testing.assert_array_equal(glog[k][b], olog[k][b], err_msg=f"sequence {b} step {k}")
            compared += 1
        if clean:
            whole += 1
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
    assert compared >= 0.75 * total and whole >= CFG.batch // 2
    print(f"{rule}: mean steps {res['mean_steps']:.2f}, error rate {res['error_rate']:.3f}, "
          f"sequence-steps compared {compared}/{total}, whole sequences {whole}")


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


# The driver's logits are f32: GPU confidences and KL are within the row-stats
# parity tolerance (1e-4 absolute + relative) of the oracle's, so a threshold
# decision is compared when the oracle's value is at least that far from the
# threshold, and a score ranking when neighbouring scores are at least the sum
# of the terms' tolerances apart.
CONF_TOL = 1e-4
SCORE_TOL = 5e-4


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
    return not (0 < cut < len(sorted_desc) and sorted_desc[cut - 1] - sorted_desc[cut] < ORDER_TOL)


def test_revocable_driver_matches_oracle_twin():
    """GPU and oracle decode independently; each sequence is compared step by
    step (outcome codes) until its first step with a decision inside the
    margins, and its final tokens when it never had one."""
    from decode_ref import REVOCABLE_DEFAULT, revocable_decode
    from diffusion_decoding_token_gb300.driver import SyntheticDecoder
    prob = synth.decode_problem(CFG, seed=29)
    dec = SyntheticDecoder(prob, "revocable", **PRM)
    glog = []
    res = dec.run(log=glog)
    assert res["status"] == 0 and res["unfinished"] == 0
    otrace, ostate = revocable_decode(prob, dec.max_steps, REVOCABLE_DEFAULT)
    for k, rec in enumerate(otrace):
        rec["t"] = k
    compared = total = whole = 0
    for b in range(CFG.batch):
        clean = True
        for k, rec in enumerate(otrace):
            if rec["masked"][b].sum() == 0:
                break
            total += 1
            if not clean or not _revocable_margin_ok(rec, b, REVOCABLE_DEFAULT):
                clean = False
                continue
            assert k < len(glog), (b, k)
            np.testing.assert_array_equal(glog[k][b], rec["outcome"][b], err_msg=f"sequence {b} step {k}")
            compared += 1
        if clean:
            whole += 1
            np.testing.assert_array_equal(res["tokens"][b], ostate["tok"][b])
            assert res["steps"][b] == sum(1 for rec in otrace if rec["masked"][b].sum() > 0)
    assert compared >= 0.6 * total and whole >= CFG.batch // 2
    # the revisions fix decoys: fewer wrong tokens than the plain threshold rule
    thr = SyntheticDecoder(prob, "threshold", **PRM).run()
    print(f"revocable: mean steps {res['mean_steps']:.2f}, error rate {res['error_rate']:.3f} "
          f"(threshold {thr['error_rate']:.3f}), revisions {res['revisions']}, remasks {res['remasks']}, "
          f"flip-flops {res['flipflops']}, compared {compared}/{total}, whole sequences {whole}")
    assert res["error_rate"] <= thr["error_rate"]
