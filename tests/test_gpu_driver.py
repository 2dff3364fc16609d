"""The multi-step synthetic decode driver on the GPU against its oracle twin:
every GPU step equals the oracle step taken from the same mask, sequence by
sequence where the decisions clear the margins of parity.py; invariants (progress, termination, commits)
on every rule; the whole decode replayed as one CUDA graph equals the eager
run."""
import numpy as np
import pytest

import synth
from decode_ref import PRM_DEFAULT, oracle_step
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
        return cap_margin_ok(scfg, c, m, r["D"][b], r["pool"][b], r["pool_n"][b], blk)
    r = o["dapd"]
    scfg = synth.scaled(synth.CONFIGS["tiny"], tau_edge=PRM["tau_edge"], blk=blk)
    return dapd_margin_ok(scfg, c, m, r["s"][b], r["dtilde"][b])


@pytest.mark.parametrize("rule", ["threshold", "factor", "topk", "cap", "dapd"])
def test_driver_matches_oracle_twin(rule):
    """Each GPU step against the oracle's step taken from the same mask (the
    GPU trajectory's), sequence by sequence where the margins hold; every
    committed token is the oracle's argmax at its commit step."""
    from diffusion_decoding_token_gb300.driver import SyntheticDecoder
    prob = synth.decode_problem(CFG, seed=17)
    dec = SyntheticDecoder(prob, rule, **PRM)
    glog = []
    res = dec.run(log=glog)
    assert res["status"] == 0
    masked = np.ones((CFG.batch, CFG.blk), np.uint8)
    tok = np.full((CFG.batch, CFG.blk), -1, np.int64)
    compared = total = 0
    for k, g in enumerate(glog):
        osel, o = oracle_step(prob, masked, rule, PRM)
        active = masked.sum(-1) > 0
        assert np.all(g.sum(-1)[active] >= 1) and not np.any(g & (1 - masked)), f"step {k}"
        for b in np.nonzero(active)[0]:
            total += 1
            if _margin_ok(rule, o, masked, osel, b):
                np.testing.assert_array_equal(g[b], osel[b], err_msg=f"step {k} sequence {b}")
                compared += 1
        tok = np.where(g > 0, o["argmax"].reshape(CFG.batch, CFG.blk), tok)
        masked = masked * (1 - g)
    assert masked.sum() == 0 and res["unfinished"] == 0
    np.testing.assert_array_equal(res["tokens"], tok)
    assert compared >= 0.75 * total
    assert (res["steps"] <= CFG.blk).all() and (res["steps"] >= 1).all()
    print(f"{rule}: mean steps {res['mean_steps']:.2f}, error rate {res['error_rate']:.3f}, "
          f"sequence-steps compared {compared}/{total}")


@pytest.mark.parametrize("rule", ["threshold", "topk", "cap", "dapd"])
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
