"""DepCap's block loop on the GPU (DepCapDecoder: row stats against the
snapshot, the ragged DepGA-Block boundary, CAP within the block) against the
oracle's step from the same state, step by step, where the decisions clear
the margins of parity.py; invariants of the loop; the whole decode replayed
as one CUDA graph equals the eager run."""
import numpy as np
import pytest

import synth
from decode_ref import DEPCAP_DEFAULT, depcap_step
from parity import boundary_margin_ok, cap_margin_ok

pytestmark = pytest.mark.gpu

CFG = synth.DecodeConfig(name="depcap_loop", batch=4, blk=128, vocab=1024, band=10, p_link=0.01)
PRM = dict(DEPCAP_DEFAULT, L_max=32, L_min=4, lam=1.2)


def _decoder(prob):
    from diffusion_decoding_token_gb300.driver import DepCapDecoder
    return DepCapDecoder(prob, **PRM)


def test_depcap_loop_matches_oracle_steps():
    prob = synth.decode_problem(CFG, seed=5)
    res = _decoder(prob).run(trace=True)
    assert res["status"] == 0 and res["unfinished"] == 0
    B, N, Lm = CFG.batch, CFG.blk, PRM["L_max"]
    snap = [None] * B
    seen = np.zeros(B, bool)
    tok = np.full((B, N), -1, np.int64)
    n_len = n_len_ok = n_cap = n_cap_ok = 0
    lens = []
    for k, t in enumerate(res["trace"]):
        need = t["need"].astype(bool)
        state = dict(masked=t["masked"], cursor=t["cursor"].astype(np.int64),
                     blen=np.where(need, 0, t["blen"]).astype(np.int64), cold=(~seen).astype(np.uint8),
                     snap_masked=snap)
        out = depcap_step(prob, state, PRM, blen_override=t["blen"].astype(np.int64))
        for b in np.nonzero(need)[0]:
            n_len += 1
            wl = int(out["window_len"][b])
            assert min(PRM["L_min"], wl) <= t["blen"][b] <= wl, (k, b)
            if not seen[b] or boundary_margin_ok(out["score"][b, :wl]):
                assert t["blen"][b] == out["new_len"][b], (k, b)
                n_len_ok += 1
            lens.append(int(t["blen"][b]))
        conf = out["stats"]["conf"].reshape(B, Lm)
        scfg = synth.scaled(synth.CONFIGS["tiny"], tau_low=PRM["tau_low"], gamma=PRM["gamma"], p_max=Lm)
        for b in range(B):
            if t["cursor"][b] >= N:
                assert not t["sel"][b].any()
                continue
            n_cap += 1
            if cap_margin_ok(scfg, conf[b], out["mwin"][b], out["cap"]["D"][b], out["cap"]["pool"][b],
                             out["cap"]["pool_n"][b], int(t["blen"][b])):
                np.testing.assert_array_equal(t["sel"][b], out["sel"][b], err_msg=f"step {k} sequence {b}")
                n_cap_ok += 1
            assert t["sel"][b].any()                                   # progress
            am = out["stats"]["argmax"].reshape(B, Lm)[b]
            for j in np.nonzero(t["sel"][b])[0]:
                tok[b, out["pos"][b, j]] = am[j]
        for b in np.nonzero(need)[0]:
            snap[b] = t["masked"][b].copy()
            seen[b] = True
    np.testing.assert_array_equal(res["tokens"], tok)                  # every commit is the oracle's argmax
    assert n_len_ok >= 0.8 * n_len and n_cap_ok >= 0.8 * n_cap
    assert len(set(lens)) > 2                                          # the boundary really varies
    assert (res["n_blocks"] >= N // Lm).all()
    print(f"depcap loop: mean steps {res['mean_steps']:.1f}, blocks {res['n_blocks'].tolist()}, "
          f"lengths compared {n_len_ok}/{n_len}, CAP steps compared {n_cap_ok}/{n_cap}, "
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
