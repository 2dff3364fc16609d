"""The parity harness itself (CPU): the margin screen, and the enumeration of
admissible results that checks unscreened draws.

* With no decision inside the margins, the enumerated result is the oracle's
  own selection (the greedy over edge orientations reproduces the oracle's
  scan), for CAP and DAPD on screened workloads.
* A planted near tie admits both resolutions, a clear gap only one.
* The screen returns workloads on which every sequence clears the margins,
  redrawing the sequences that do not.
"""
import numpy as np
import pytest

import oracle
import synth
from parity import (FP32_ORDER_BAND, MARGIN, _greedy_dag, boundary_range, cap_outcomes, dapd_outcomes,
                    oracle_stats_seq, screen, sequence_decisions, sequence_margin_failures,
                    threshold_outcome_check)


@pytest.mark.parametrize("name", ["tiny", "llada_step"])
def test_screened_workload_has_one_admissible_result_equal_to_the_oracle(name):
    cfg = synth.CONFIGS[name]
    log = []
    w, o = screen(cfg, 1000 + synth.ORDER.index(name), use_stored=False, log=log)
    blk = cfg.blk
    for b in range(cfg.batch):
        st = {k: v[b * blk:(b + 1) * blk] for k, v in o.items()}
        assert not sequence_margin_failures(w, b, st)
        dec = sequence_decisions(w, b, st)
        r, Dw, scope = dec["cap"]
        outs = cap_outcomes(cfg, st["conf"], w.masked[b], Dw, scope)
        assert outs == {frozenset(np.nonzero(r["selected"][0])[0].tolist())}
        rd = dec["dapd"]
        outs = dapd_outcomes(cfg, st["conf"], w.masked[b], rd["s"][0], rd["dtilde"][0])
        assert outs == {frozenset(np.nonzero(rd["selected"][0])[0].tolist())}
    if name == "tiny":
        assert log, "the tiny workload's first draw misses a margin and is redrawn"
        assert w.attempts[0] == len(log)


def test_redrawn_sequence_equals_a_fresh_draw_with_that_attempt():
    cfg = synth.CONFIGS["tiny"]
    w, o = screen(cfg, 1000, use_stored=False)
    fresh = synth.make(cfg, 1000, attempts=w.attempts)
    np.testing.assert_array_equal(fresh.cur, w.cur)
    st = oracle_stats_seq(fresh, 0)
    np.testing.assert_array_equal(st["conf"], o["conf"])


def _cap_case(c, D):
    cfg = synth.scaled(synth.CONFIGS["tiny"], tau_low=0.8, tau_high=0.95, gamma=-16.0, p_max=8, blk=len(c))
    return cfg, np.asarray(c, np.float64), np.ones(len(c), np.uint8), np.asarray(D, np.float64)


def test_cap_near_tie_admits_both_orders():
    # positions 0 and 1 conflict (D = -5 > gamma); 2 conflicts with neither
    D = np.full((3, 3), -40.0)
    D[0, 1] = D[1, 0] = -5.0
    cfg, c, m, D = _cap_case([0.97, 0.97 * (1 + 3e-6), 0.99], D)
    assert cap_outcomes(cfg, c, m, D, 3) == {frozenset({1, 2}), frozenset({0, 2})}
    cfg, c, m, D = _cap_case([0.97, 0.975, 0.99], D)                  # a clear gap: one result
    assert cap_outcomes(cfg, c, m, D, 3) == {frozenset({1, 2})}
    D2 = D.copy()
    D2[0, 1] = D2[1, 0] = -16.0 + 0.5 * MARGIN                         # conflict test inside the margin
    assert cap_outcomes(cfg, c, m, D2, 3) == {frozenset({1, 2}), frozenset({0, 1, 2})}
    # an empty pool falls back to the most confident masked position
    cfg, c, m, D = _cap_case([0.5, 0.6, 0.6 * (1 + 2e-6)], np.full((3, 3), np.nan))
    assert cap_outcomes(cfg, c, m, D, 3) == {frozenset({1}), frozenset({2})}


def test_dapd_near_tie_admits_both_orders():
    cfg = synth.scaled(synth.CONFIGS["tiny"], tau_edge=0.02, blk=3)
    s = np.full((3, 3), 0.001)
    s[0, 1] = s[1, 0] = 0.1                                           # one edge: 0 - 1
    dt = np.array([1.0, 1.0, 1.0])
    c = np.array([0.5, 0.5 * (1 + 1e-6), 0.2])
    assert dapd_outcomes(cfg, c, np.ones(3, np.uint8), s, dt) == {frozenset({0, 2}), frozenset({1, 2})}
    c = np.array([0.5, 0.6, 0.2])
    assert dapd_outcomes(cfg, c, np.ones(3, np.uint8), s, dt) == {frozenset({1, 2})}
    s2 = s.copy()
    s2[1, 2] = s2[2, 1] = 0.02 + 0.1 * MARGIN                        # edge test inside the margin
    outs = dapd_outcomes(cfg, c, np.ones(3, np.uint8), s2, dt)
    assert outs == {frozenset({1, 2}), frozenset({1})}


def test_greedy_over_orientations_and_cycles():
    nodes, edges = [0, 1, 2], [(0, 1), (1, 2)]
    assert _greedy_dag(nodes, edges, lambda u, v: u < v) == frozenset({0, 2})
    assert _greedy_dag(nodes, edges, lambda u, v: u > v) == frozenset({2, 0})
    # a path oriented 1 -> 0 and 1 -> 2: 1 first
    first = {1: 0, 0: 1, 2: 2}
    assert _greedy_dag(nodes, edges, lambda u, v: first[u] < first[v]) == frozenset({1})
    tri = [(0, 1), (1, 2), (0, 2)]
    cyc = {(0, 1): True, (1, 2): True, (0, 2): False}                  # 0 -> 1 -> 2 -> 0
    assert _greedy_dag(nodes, tri, lambda u, v: cyc[(u, v)] if (u, v) in cyc else not cyc[(v, u)]) is None


def test_threshold_and_boundary_validity_checks():
    c = np.array([0.95, 0.9 + 0.2 * MARGIN, 0.3, 0.2])
    m = np.ones(4, np.uint8)
    assert threshold_outcome_check(c, m, 0.9, np.array([1, 0, 0, 0])) == (True, False)
    assert threshold_outcome_check(c, m, 0.9, np.array([1, 1, 0, 0])) == (True, False)
    assert threshold_outcome_check(c, m, 0.9, np.array([0, 1, 0, 0]))[0] is False   # the clear one is missing
    assert threshold_outcome_check(c, m, 0.9, np.array([1, 0, 1, 0]))[0] is False
    c2 = np.array([0.5, 0.5 * (1 + FP32_ORDER_BAND / 4), 0.3, 0.2])  # fallback near tie
    assert threshold_outcome_check(c2, m, 0.9, np.array([0, 1, 0, 0])) == (True, False)
    assert threshold_outcome_check(c2, m, 0.9, np.array([1, 0, 0, 0])) == (True, False)
    assert threshold_outcome_check(c2, m, 0.9, np.array([0, 0, 1, 0]))[0] is False
    # boundary: S = [0.5, 0.4, 2e-4, -0.3]: k* is 2 or 3 (S_2 inside the margin)
    assert boundary_range(np.array([0.5, 0.4, 2e-4, -0.3, 0.1]), 1) == (2, 3)
    assert boundary_range(np.array([0.5, 0.4, 0.2, -0.3, 0.1]), 1) == (3, 3)
    assert boundary_range(np.array([0.5, 0.4, 0.2, 0.3]), 1) == (4, 4)
    assert boundary_range(np.array([-0.5, 0.4]), 2) == (2, 2)          # clipped to L_min


def test_oracle_cap_row_index_reads_the_named_rows():
    """CAP through a row index over rows stored in another order gives the
    result of the block-contiguous layout (DepCap, Methodology: the pool is
    the block's positions, wherever their rows are stored)."""
    rng = np.random.default_rng(4)
    B, blk, V = 3, 24, 512
    z = rng.standard_normal((B * blk, V)).astype(np.float32)
    tok = rng.integers(0, V, B * blk)
    z[np.arange(B * blk), tok] += 9.0
    for r in range(0, B * blk - 1, 3):
        z[r, tok[r + 1]] = z[r, tok[r]] - 3
        z[r + 1, tok[r]] = z[r + 1, tok[r + 1]] - 3
    o = oracle.row_stats(z)
    am, c, lse = o["argmax"].reshape(B, blk), o["conf"].reshape(B, blk), o["lse"].reshape(B, blk)
    m = np.ones((B, blk), np.uint8)
    ref = oracle.cap_select(z, am, c, lse, m, 0.8, 0.95, -16.0, blk)
    perm = rng.permutation(B * blk + 10)
    store = rng.standard_normal((B * blk + 10, V)).astype(np.float32)
    store[perm[:B * blk]] = z
    got = oracle.cap_select(store, am, c, lse, m, 0.8, 0.95, -16.0, blk, row_index=perm[:B * blk])
    np.testing.assert_array_equal(got["selected"], ref["selected"])
    np.testing.assert_array_equal(np.nan_to_num(got["D"], nan=1.0), np.nan_to_num(ref["D"], nan=1.0))
    assert ref["n_selected"].min() >= 1 and (ref["n_selected"] < blk).all()
