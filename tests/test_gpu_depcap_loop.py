"""DepCap's block loop on the GPU (DepCapDecoder: row stats of the window
rows, read in place through a row index, against the snapshot; the ragged
DepGA-Block boundary; CAP within the block through the same row index)
against the oracle's loop, which gathers the window rows itself.  The
problem is screened (parity.screen_decode) so that every sequence's oracle
loop clears the decision margins at every step: the two run independently
and agree on every step of every sequence.  Also the loop's invariants, and
the whole decode replayed as one CUDA graph equals the eager run."""
import numpy as np
import pytest

import synth
from decode_ref import DEPCAP_DEFAULT, depcap_decode
from parity import boundary_margin_failures, cap_margin_failures, screen_decode

pytestmark = pytest.mark.gpu

CFG = synth.DecodeConfig(name="depcap_loop", batch=4, blk=128, vocab=1024, band=10, p_link=0.01)
PRM = dict(DEPCAP_DEFAULT, L_max=32, L_min=4, lam=1.2)


def _decoder(prob):
    from diffusion_decoding_token_gb300.driver import DepCapDecoder
    return DepCapDecoder(prob, **PRM)


def _step_margin_ok(state, out, b, scfg):
    """The boundary (when the sequence picks a block) and CAP decisions of
    sequence b in this oracle step clear the margins of parity.py."""
    if out["need"][b] and state["snap_masked"][b] is not None:
        wl = int(out["window_len"][b])
        if boundary_margin_failures(out["score"][b, :wl]):
            return False
    conf = out["stats"]["conf"].reshape(len(out["need"]), -1)
    return not cap_margin_failures(scfg, conf[b], out["mwin"][b], out["cap"]["D"][b], int(out["blen"][b]))


def _twin(prob):
    otrace = []
    osteps, otok, oblocks = depcap_decode(prob, PRM, trace=otrace)
    return otrace, osteps, otok, oblocks


def _sequence_ok(twin, b):
    scfg = synth.scaled(synth.CONFIGS["tiny"], tau_low=PRM["tau_low"], gamma=PRM["gamma"], p_max=PRM["L_max"])
    return all(_step_margin_ok(state, out, b, scfg) for state, out in twin[0] if state["cursor"][b] < CFG.blk)


def test_depcap_loop_matches_oracle():
    """GPU and oracle run the loop independently on the screened problem;
    every step of every sequence (cursor, block length, selection) agrees,
    and so do the tokens, step counts and block counts."""
    prob, (otrace, osteps, otok, oblocks) = screen_decode(CFG, 5, _twin, _sequence_ok)
    res = _decoder(prob).run(trace=True)
    assert res["status"] == 0 and res["unfinished"] == 0
    B, N, Lm = CFG.batch, CFG.blk, PRM["L_max"]
    compared = 0
    for b in range(B):
        for k, (state, out) in enumerate(otrace):
            if state["cursor"][b] >= N:
                break
            g = res["trace"][k]
            assert g["cursor"][b] == state["cursor"][b] and bool(g["need"][b]) == bool(out["need"][b]), (b, k)
            assert g["blen"][b] == out["blen"][b], (b, k)
            np.testing.assert_array_equal(g["sel"][b], out["sel"][b], err_msg=f"sequence {b} step {k}")
            compared += 1
        np.testing.assert_array_equal(res["tokens"][b], otok[b])
        assert res["steps"][b] == osteps[b] and res["n_blocks"][b] == len(oblocks[b])
    # the loop's invariants on the GPU trace alone
    for b in range(B):
        start, blen, lens = 0, 0, []
        for k, t in enumerate(res["trace"]):
            if t["cursor"][b] >= N:
                assert start + blen == N
                break
            if t["need"][b]:                                            # a new block starts where the last ended
                assert t["cursor"][b] == start + blen, (b, k)
                start, blen = int(t["cursor"][b]), int(t["blen"][b])
                wl = min(Lm, N - start)
                assert min(PRM["L_min"], wl) <= blen <= wl
                lens.append(blen)
            else:
                assert t["cursor"][b] == start and t["blen"][b] == blen, (b, k)
            assert t["sel"][b].any() and not np.any(t["sel"][b][blen:])   # progress, inside the block
        assert lens[0] == PRM["L_min"] and len(set(lens)) > 1
    print(f"depcap loop: mean steps {res['mean_steps']:.1f}, blocks {res['n_blocks'].tolist()}, "
          f"steps compared {compared} (all), redrawn sequences {int((prob['attempts'] > 0).sum())}, "
          f"error rate {res['error_rate']:.3f}")


def test_depcap_whole_decode_graph_equals_eager():
    prob = synth.decode_problem(CFG, seed=6)
    a = _decoder(prob).run()
    dec = _decoder(prob)
    b = dec.run(graph=True)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_array_equal(a["steps"], b["steps"])
    np.testing.assert_array_equal(a["n_blocks"], b["n_blocks"])
    dec.reset()
    c = dec.run(graph=True)
    np.testing.assert_array_equal(c["tokens"], b["tokens"])
