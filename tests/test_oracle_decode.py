"""The oracle twin of the multi-step decode driver: the stand-in model's
closed forms and the loop's invariants (progress, termination, commits)."""
import dataclasses

import numpy as np
import pytest

import synth
from decode_ref import PRM_DEFAULT, model_logits, oracle_decode

CFG = synth.DecodeConfig(batch=3, blk=16, vocab=256)


def test_model_closed_forms():
    prob = synth.decode_problem(CFG, seed=5)
    B, blk = CFG.batch, CFG.blk
    rows = np.arange(B * blk)
    t, d = prob["target"].reshape(-1), prob["decoy"].reshape(-1)
    c0 = np.float32(prob["c0"])
    lg = prob["base"].copy()
    model_logits(prob, lg, np.ones((B, blk), np.uint8))            # nothing decoded: s = 0
    np.testing.assert_array_equal(lg[rows, t], c0 + prob["u"].reshape(-1))
    np.testing.assert_array_equal(lg[rows, d], c0 + prob["v"].reshape(-1))
    model_logits(prob, lg, np.zeros((B, blk), np.uint8))           # all decoded: s = 1 where deg > 0
    has = prob["links"].reshape(B * blk, blk).any(-1)
    np.testing.assert_allclose(lg[rows, t][has], (c0 + prob["u"].reshape(-1) + np.float32(CFG.kappa))[has], rtol=1e-6)
    np.testing.assert_array_equal(lg[rows, d][has], np.full(has.sum(), c0, np.float32))
    other = np.ones_like(lg, bool)
    other[rows, t] = other[rows, d] = False
    np.testing.assert_array_equal(lg[other], prob["base"][other])   # background untouched


def test_background_mass_constant():
    # c0 = ln(V - 1) + sigma^2/2 is the expected log of the summed exp of V - 1
    # N(0, sigma^2) logits (lognormal mean)
    cfg = dataclasses.replace(CFG, vocab=4096, batch=2)
    prob = synth.decode_problem(cfg, seed=1)
    lse = np.log(np.exp(prob["base"].astype(np.float64)).sum(-1))
    assert abs(lse.mean() - float(prob["c0"])) < 0.05


@pytest.mark.parametrize("rule", ["threshold", "factor", "topk", "cap", "dapd"])
def test_decode_invariants(rule):
    prob = synth.decode_problem(CFG, seed=9)
    log, stats, tok = oracle_decode(prob, rule, CFG.blk, PRM_DEFAULT)
    masked = np.ones((CFG.batch, CFG.blk), np.uint8)
    for sel, (o, m) in zip(log, stats):
        np.testing.assert_array_equal(m, masked)
        assert not np.any(sel & (1 - masked))                 # only masked positions are chosen
        active = masked.sum(-1) > 0
        assert np.all(sel.sum(-1)[active] >= 1)               # progress on every active sequence
        masked = masked * (1 - sel)
    assert masked.sum() == 0 and len(log) <= CFG.blk          # termination
    am = [o["argmax"].reshape(CFG.batch, CFG.blk) for o, _ in stats]
    for b in range(CFG.batch):                                # each token is the argmax at its commit step
        for i in range(CFG.blk):
            k = next(k for k, s in enumerate(log) if s[b, i])
            assert tok[b, i] == am[k][b, i]
    if rule == "topk":
        assert len(log) == -(-CFG.blk // PRM_DEFAULT["topk_k"])


def test_no_decoy_no_errors():
    cfg = dataclasses.replace(CFG, v_hi=1e-6, u_lo=3.0)
    prob = synth.decode_problem(cfg, seed=3)
    for rule in ("threshold", "factor", "topk", "cap", "dapd"):
        _, _, tok = oracle_decode(prob, rule, cfg.blk, PRM_DEFAULT)
        np.testing.assert_array_equal(tok, prob["target"])


def test_decoys_hurt_parallel_rules_more():
    # one token per step commits each position after more of its neighbours
    # are decoded than a confidence threshold does: fewer decoys win
    cfg = dataclasses.replace(synth.DecodeConfig(), batch=8, blk=32, vocab=1024)
    prob = synth.decode_problem(cfg, seed=11)
    err = {}
    for rule, k in (("topk", 1), ("threshold", None)):
        prm = dict(PRM_DEFAULT, topk_k=1)
        _, _, tok = oracle_decode(prob, rule, cfg.blk, prm)
        err[rule] = float((tok != prob["target"]).mean())
    assert err["topk"] < err["threshold"]


def test_depcap_loop_invariants():
    from decode_ref import DEPCAP_DEFAULT, depcap_decode
    cfg = synth.DecodeConfig(name="depcap_loop", batch=3, blk=96, vocab=256, band=10, p_link=0.01)
    prob = synth.decode_problem(cfg, seed=5)
    prm = dict(DEPCAP_DEFAULT, L_max=32, L_min=4)
    steps, tok, blocks = depcap_decode(prob, prm)
    assert (tok >= 0).all()
    for b in range(cfg.batch):
        starts = [s for s, _ in blocks[b]]
        ends = [s + n for s, n in blocks[b]]
        assert starts[0] == 0 and ends[-1] == cfg.blk and starts[1:] == ends[:-1]     # contiguous tiling
        assert blocks[b][0][1] == prm["L_min"]                                       # cold start
        for s, n in blocks[b]:
            assert min(prm["L_min"], cfg.blk - s) <= n <= min(prm["L_max"], cfg.blk - s)
        assert len(blocks[b]) <= steps[b] <= cfg.blk
    assert len({n for bl in blocks for _, n in bl}) > 2
