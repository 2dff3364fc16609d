"""Pins for the oracle's selection rules.

* Fast-dLLM threshold rule (Fast-dLLM review, Method; notes, Key ideas):
  brute-force definition, never empty while anything is masked.
* DepGA-Block boundary (DepCap, Methodology): a worked example, the
  clipping invariants, cold start, and the smoothing against numpy.
* CAP-Decoding (DepCap, Methodology): conflict-free, maximal within the pool,
  equal to the brute-force lexicographically first conflict-free set, the
  duplicate-token closed form for D_ij, pool clipping, the fallback.
* DAPD (关键设计 1-3): the page's 9-node MRF worked by hand, numpy's mean for
  a_ij, symmetry and row sums, brute force on small graphs, the 50% switch.
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from brute import greedy_consistent, is_independent, is_maximal, lex_first_mis

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- threshold
def test_threshold_matches_definition(oracle):
    rng = np.random.default_rng(1)
    for trial in range(50):
        B, blk = 3, int(rng.integers(1, 40))
        conf = rng.random((B, blk))
        masked = (rng.random((B, blk)) < 0.7).astype(np.uint8)
        tau = float(rng.choice([0.5, 0.9, 0.99]))
        sel, n = oracle.select_threshold(conf, masked, tau)
        for b in range(B):
            want = [i for i in range(blk) if masked[b, i] and np.float32(conf[b, i]) > np.float32(tau)]
            if not want and masked[b].any():
                cands = [i for i in range(blk) if masked[b, i]]
                want = [max(cands, key=lambda i: (np.float32(conf[b, i]), -i))]
            assert sorted(np.nonzero(sel[b])[0].tolist()) == want
            assert n[b] == len(want)
            if masked[b].any():
                assert n[b] >= 1


def test_threshold_fallback_tie_and_empty(oracle):
    conf = np.array([[0.3, 0.5, 0.5, 0.1], [0.95, 0.2, 0.99, 0.3]])
    masked = np.array([[1, 1, 1, 1], [0, 0, 0, 0]], np.uint8)
    sel, n = oracle.select_threshold(conf, masked, 0.9)
    assert sel[0].tolist() == [0, 1, 0, 0] and n[0] == 1   # tie -> lower index
    assert sel[1].tolist() == [0, 0, 0, 0] and n[1] == 0   # nothing masked


# ----------------------------------------------------------------- boundary
def test_boundary_worked_example(oracle):
    # I = 1 everywhere -> I~ = 1;  H / mean(H) with mean 0.875:
    # S = 1 - [0.5, 0.5, 2, 0.5] / 0.875 = [0.43, 0.43, -1.29, 0.43]
    # first negative at k = 2.
    I = np.array([[1.0, 1.0, 1.0, 1.0]] * 3)
    H = np.array([[0.5, 0.5, 2.0, 0.5]] * 3)
    blen, S = oracle.depcap_boundary(I, H, lam=1.0, L_min=1)
    np.testing.assert_allclose(S[0], 1 - np.array([0.5, 0.5, 2.0, 0.5]) / 0.875, rtol=1e-15)
    assert blen.tolist() == [2, 2, 2]
    blen, _ = oracle.depcap_boundary(I, H, lam=1.0, L_min=3)
    assert blen.tolist() == [3, 3, 3]
    blen, _ = oracle.depcap_boundary(I, H, lam=1.0, L_min=1, cold_start=np.array([0, 1, 0]))
    assert blen.tolist() == [2, 1, 2]
    blen, _ = oracle.depcap_boundary(I, H, lam=0.25, L_min=1)   # 1 - 0.25*2.29 > 0 everywhere
    assert blen.tolist() == [4, 4, 4]


def test_boundary_invariants(oracle):
    rng = np.random.default_rng(2)
    for _ in range(40):
        B, Lw = 4, int(rng.integers(1, 70))
        I = rng.gamma(1.0, 1.0, (B, Lw))
        H = rng.gamma(1.0, 1.0, (B, Lw))
        L_min = int(rng.integers(1, 12))
        w = int(rng.choice([1, 3, 5]))
        mode = int(rng.integers(0, 3))
        lam = float(rng.uniform(0.2, 2.0))
        blen, S = oracle.depcap_boundary(I, H, lam=lam, L_min=L_min, smooth_w=w, norm_mode=mode)
        for b in range(B):
            assert min(L_min, Lw) <= blen[b] <= Lw
            neg = np.nonzero(S[b].astype(np.float32) < 0)[0]
            kstar = int(neg[0]) if len(neg) else Lw
            assert blen[b] == min(max(kstar, L_min), Lw)


def test_boundary_smoothing_and_norms_against_numpy(oracle):
    rng = np.random.default_rng(3)
    Lw = 23
    I = rng.gamma(2.0, 1.0, (1, Lw))
    H = rng.gamma(2.0, 1.0, (1, Lw))
    for w in (1, 3, 7):
        k = np.ones(w)
        sm = lambda x: np.convolve(x, k, "same") / np.convolve(np.ones(Lw), k, "same")
        Is, Hs = sm(I[0]), sm(H[0])
        lam = float(np.float32(0.7))   # the rule takes lambda as fp32
        _, S0 = oracle.depcap_boundary(I, H, lam=0.7, L_min=1, smooth_w=w, norm_mode=0)
        np.testing.assert_allclose(S0[0], Is / Is.mean() - lam * Hs / Hs.mean(), rtol=1e-12)
        _, S1 = oracle.depcap_boundary(I, H, lam=0.7, L_min=1, smooth_w=w, norm_mode=1)
        mm = lambda x: (x - x.min()) / (x.max() - x.min())
        np.testing.assert_allclose(S1[0], mm(Is) - lam * mm(Hs), rtol=1e-12, atol=1e-15)
        _, S2 = oracle.depcap_boundary(I, H, lam=0.7, L_min=1, smooth_w=w, norm_mode=2)
        np.testing.assert_allclose(S2[0], Is - lam * Hs, rtol=1e-12)


def test_boundary_ragged_windows(oracle):
    # L_window = min(L_max, L_remain) per sequence: row stride 4, windows 4, 3, 2, 0.
    I = np.ones((4, 4))
    H = np.array([[0.5, 0.5, 2.0, 0.5]] * 4)
    blen, S = oracle.depcap_boundary(I, H, lam=1.0, L_min=1, window_len=np.array([4, 3, 2, 0]))
    # window 3: H/mean = [0.5, 0.5, 2] / 1 -> S = [0.5, 0.5, -1], first negative 2
    np.testing.assert_allclose(S[1, :3], [0.5, 0.5, -1.0], rtol=1e-15)
    # window 2: H/mean = [1, 1] -> S = [0, 0], none negative -> the whole window
    np.testing.assert_allclose(S[2, :2], [0.0, 0.0], atol=1e-15)
    assert blen.tolist() == [2, 2, 2, 0]
    assert np.isnan(S[1, 3]) and np.isnan(S[2, 2:]).all() and np.isnan(S[3]).all()
    blen, _ = oracle.depcap_boundary(I, H, lam=1.0, L_min=3, window_len=np.array([4, 3, 2, 0]),
                                     cold_start=np.array([0, 0, 1, 1]))
    assert blen.tolist() == [3, 3, 2, 0]      # clipped to the window; cold start min(L_min, window)


def test_boundary_ragged_against_numpy(oracle):
    rng = np.random.default_rng(4)
    B, Ls = 6, 19
    I = rng.gamma(2.0, 1.0, (B, Ls))
    H = rng.gamma(2.0, 1.0, (B, Ls))
    wl = np.array([19, 1, 7, 12, 2, 5])
    lam = float(np.float32(0.9))
    for w in (1, 3):
        _, S = oracle.depcap_boundary(I, H, lam=0.9, L_min=1, smooth_w=w, norm_mode=0, window_len=wl)
        for b in range(B):
            n = wl[b]
            k = np.ones(w)
            sm = lambda x: np.convolve(x, k, "same")[:n] / np.convolve(np.ones(n), k, "same")[:n]
            if n < w:   # np.convolve "same" needs len >= kernel: do it by hand
                sm = lambda x: np.array([x[max(0, j - w // 2):min(n, j + w // 2 + 1)].mean() for j in range(n)])
            Is, Hs = sm(I[b, :n]), sm(H[b, :n])
            np.testing.assert_allclose(S[b, :n], Is / Is.mean() - lam * Hs / Hs.mean(), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------- CAP
def _cap_case(rng, blk, V, n_conf_pairs, dup_pairs=0):
    z = rng.standard_normal((blk, V)).astype(np.float32)
    tok = rng.permutation(V)[:blk]
    for i in range(blk):
        z[i, tok[i]] = float(rng.uniform(5, 12))
    for _ in range(n_conf_pairs):
        i, j = rng.choice(blk, 2, replace=False)
        z[i, tok[j]] = z[i, tok[i]] - float(rng.uniform(2, 6))
        z[j, tok[i]] = z[j, tok[j]] - float(rng.uniform(2, 6))
    for _ in range(dup_pairs):
        i, j = rng.choice(blk, 2, replace=False)
        z[j, tok[i]] = z[j, tok[j]] + 1.0
    return z


def test_cap_brute_force_and_invariants(oracle):
    rng = np.random.default_rng(4)
    for trial in range(60):
        blk = int(rng.integers(2, 13))
        z = _cap_case(rng, blk, 64, int(rng.integers(0, blk)), int(rng.integers(0, 3)))
        st = oracle.row_stats(z)
        masked = (rng.random((1, blk)) < 0.85).astype(np.uint8)
        tau_low = float(rng.choice([0.0, 0.5, 0.9]))
        gamma = float(rng.choice([-16.0, -6.0, -3.0]))
        r = oracle.cap_select(z, st["argmax"], st["conf"], st["lse"], masked, tau_low, 0.95, gamma,
                              p_max=blk)
        pool = [int(p) for p in r["pool"][0][:r["pool_n"][0]]]
        c32 = st["conf"].astype(np.float32)
        want_pool = sorted([i for i in range(blk) if masked[0, i] and c32[i] >= np.float32(tau_low)],
                           key=lambda i: (-c32[i], i))
        assert pool == want_pool
        sel = set(np.nonzero(r["selected"][0])[0].tolist())
        if not pool:
            cands = [i for i in range(blk) if masked[0, i]]
            assert sel == ({max(cands, key=lambda i: (c32[i], -i))} if cands else set())
            continue
        D = r["D"][0]
        # D_ij from its definition with numpy logs
        logp = z.astype(np.float64) - st["lse"][:, None]
        for i in pool:
            for j in pool:
                if i != j:
                    assert D[i, j] == pytest.approx(logp[i, st["argmax"][j]] + logp[j, st["argmax"][i]], abs=1e-12)
                    assert D[i, j] == D[j, i]
        adj = np.zeros((blk, blk), bool)
        for i in pool:
            for j in pool:
                adj[i, j] = i != j and np.float32(D[i, j]) > np.float32(gamma)
        assert sel <= set(pool)
        assert is_independent(adj, sel)
        assert is_maximal(adj, sel, pool)
        sub = adj[np.ix_(pool, pool)]
        want = {pool[k] for k in lex_first_mis(sub, list(range(len(pool))))}
        assert sel == want
        assert r["n_selected"][0] == len(sel)


def test_cap_duplicate_token_closed_form(oracle):
    # two positions whose argmax is the same token: D = log c_i + log c_j
    z = np.full((3, 16), -20.0, np.float32)     # unrelated tokens: D far below gamma
    z[0, 4], z[1, 4], z[2, 9] = 6.0, 5.0, 7.0
    st = oracle.row_stats(z)
    masked = np.ones((1, 3), np.uint8)
    r = oracle.cap_select(z, st["argmax"], st["conf"], st["lse"], masked, 0.0, 0.95, -16.0, 3)
    assert r["D"][0][0, 1] == pytest.approx(math.log(st["conf"][0]) + math.log(st["conf"][1]), rel=1e-13)
    # 0 and 1 conflict (D ~ -0.1 > -16): the higher-confidence one (position 2, then 0) is kept
    assert r["selected"][0].tolist() == [1, 0, 1]


def test_cap_pool_clip_scope_and_high_tier(oracle):
    rng = np.random.default_rng(9)
    blk = 10
    z = _cap_case(rng, blk, 50, 0)
    st = oracle.row_stats(z)
    masked = np.ones((1, blk), np.uint8)
    r = oracle.cap_select(z, st["argmax"], st["conf"], st["lse"], masked, 0.0, 0.95, -16.0, p_max=4)
    c32 = st["conf"].astype(np.float32)
    top4 = sorted(range(blk), key=lambda i: (-c32[i], i))[:4]
    assert r["clipped"] and r["pool_n"][0] == 4 and r["pool"][0][:4].tolist() == top4
    assert set(np.nonzero(r["selected"][0])[0]) == set(top4)   # no conflicts planted
    r = oracle.cap_select(z, st["argmax"], st["conf"], st["lse"], masked, 0.0, 0.95, -16.0, p_max=10,
                          scope_len=np.array([3], np.int32))
    assert set(np.nonzero(r["selected"][0])[0]) == {0, 1, 2}
    # high tier unconditional: two tier members that conflict are both kept
    z2 = np.full((3, 8), -20.0, np.float32)
    z2[0, 1], z2[1, 1], z2[2, 5] = 9.0, 8.5, 1.0   # rows 0,1 share token 1 -> conflict
    st2 = oracle.row_stats(z2)
    m3 = np.ones((1, 3), np.uint8)
    a = oracle.cap_select(z2, st2["argmax"], st2["conf"], st2["lse"], m3, 0.0, 0.9, -16.0, 3)
    b = oracle.cap_select(z2, st2["argmax"], st2["conf"], st2["lse"], m3, 0.0, 0.9, -16.0, 3,
                          high_tier_unconditional=True)
    assert a["selected"][0].tolist() == [1, 0, 1]
    assert b["selected"][0].tolist() == [1, 1, 1]


def test_cap_fallback_when_pool_empty(oracle):
    z = np.zeros((4, 32), np.float32)
    z[:, 3] = [0.1, 0.4, 0.4, 0.2]
    st = oracle.row_stats(z)
    masked = np.array([[1, 0, 1, 1]], np.uint8)
    r = oracle.cap_select(z, st["argmax"], st["conf"], st["lse"], masked, 0.8, 0.95, -16.0, 4)
    assert r["pool_n"][0] == 0 and r["selected"][0].tolist() == [0, 0, 1, 0]


# --------------------------------------------------------------------- DAPD
def test_dapd_mrf9_worked_example(oracle):
    g = json.load(open(os.path.join(GOLDEN, "dapd_mrf9.json")))
    n = len(g["nodes"])
    A = np.full((n, n), 0.001, np.float32)
    for a, b in g["edges"]:
        A[a, b] = A[b, a] = 0.1
    attn = A[None, None, None]                # B=1, L=1, H=1
    conf = np.array([[0.9, 0.8, 0.95, 0.7, 0.6, 0.99, 0.5, 0.85, 0.75]])
    masked = np.ones((1, n), np.uint8)
    r = oracle.dapd(attn, masked, conf, tau_edge=0.05)
    # d~ = 0.1*deg + 0.001*(8-deg); keys d~*conf order X3,X2,X4,Y1,X1,Y3,Y4,X5,Y2;
    # greedy keeps X3, then Y1 (X1,X2 free of X3), then Y4 (X4 is out, X5 free).
    assert r["deg"][0].tolist() == g["true_degree"]
    deg = np.array(g["true_degree"])
    np.testing.assert_allclose(r["dtilde"][0], np.float32(0.1) * deg + np.float32(0.001) * (8 - deg), rtol=1e-6)
    assert np.nonzero(r["selected"][0])[0].tolist() == [2, 5, 8]
    assert r["path"][0] == 0


def test_dapd_graph_properties_and_brute_force(oracle):
    rng = np.random.default_rng(6)
    for trial in range(40):
        blk = int(rng.integers(2, 13))
        L, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        A = rng.random((1, L, H, blk, blk)).astype(np.float32) * 0.2
        conf = rng.random((1, blk))
        masked = np.ones((1, blk), np.uint8)
        masked[0, rng.random(blk) < 0.3] = 0
        if 2 * masked.sum() < blk:
            continue
        tau = 0.1
        r = oracle.dapd(A, masked, conf, tau_edge=tau)
        nodes = np.nonzero(masked[0])[0]
        a = A[0].astype(np.float64).mean(axis=(0, 1))
        s = 0.5 * (a + a.T)
        S = r["s"][0]
        np.testing.assert_allclose(S[np.ix_(nodes, nodes)], s[np.ix_(nodes, nodes)], rtol=1e-13)
        assert np.allclose(S[np.ix_(nodes, nodes)], S[np.ix_(nodes, nodes)].T)
        sub = s[np.ix_(nodes, nodes)]
        adj = (sub > tau) & ~np.eye(len(nodes), dtype=bool)
        dt = sub.sum(axis=1) - np.diag(sub)
        np.testing.assert_allclose(r["dtilde"][0][nodes], dt, rtol=1e-12)
        assert r["deg"][0][nodes].tolist() == adj.sum(axis=1).tolist()
        key = dt * conf[0][nodes]
        order = sorted(range(len(nodes)), key=lambda x: (-key[x], x))
        want = {int(nodes[k]) for k in lex_first_mis(adj, order)}
        got = set(np.nonzero(r["selected"][0])[0].tolist())
        assert got == want
        loc = {int(v): k for k, v in enumerate(nodes)}
        assert is_independent(adj, [loc[v] for v in got])
        assert is_maximal(adj, [loc[v] for v in got], range(len(nodes)))
        assert greedy_consistent(adj, [loc[v] for v in got], key, range(len(nodes)), 0.0)
        # order_mode 1: key = d~ only
        r1 = oracle.dapd(A, masked, conf, tau_edge=tau, order_mode=1)
        order1 = sorted(range(len(nodes)), key=lambda x: (-dt[x], x))
        assert set(np.nonzero(r1["selected"][0])[0].tolist()) == {int(nodes[k]) for k in lex_first_mis(adj, order1)}


def test_dapd_late_phase_switch(oracle):
    blk = 16
    rng = np.random.default_rng(8)
    A = rng.random((1, 1, 1, blk, blk)).astype(np.float32)
    conf = np.array([np.linspace(0.5, 0.99, blk)])
    for n_masked, path in [(8, 0), (7, 1)]:       # r = 0.5 -> graph, r = 0.4375 -> late phase
        masked = np.zeros((1, blk), np.uint8)
        masked[0, :n_masked] = 1
        r = oracle.dapd(A, masked, conf, tau_edge=0.5)
        assert r["path"][0] == path
        if path == 1:
            want = [i for i in range(n_masked) if np.float32(conf[0, i]) > np.float32(0.9)]
            want = want or [n_masked - 1]
            assert np.nonzero(r["selected"][0])[0].tolist() == want
    # late phase, nothing above 0.9 -> top-confidence masked position
    masked = np.zeros((1, blk), np.uint8)
    masked[0, [1, 4, 6]] = 1
    r = oracle.dapd(A, masked, np.full((1, blk), 0.3), tau_edge=0.5)
    assert np.nonzero(r["selected"][0])[0].tolist() == [1]


def test_dapd_on_generated_workload(oracle):
    cfg = synth.scaled(synth.CONFIGS["stress_graph"], batch=2, blk=48, vocab=512, seq_len=192,
                       block_start=144)
    w = synth.make(cfg, seed=5)
    st = oracle.row_stats(w.cur, dtype=synth.BF16)
    r = oracle.dapd(w.attn, w.masked, st["conf"].reshape(2, -1), tau_edge=cfg.tau_edge, dtype=synth.F16)
    for b in range(2):
        nodes = np.arange(cfg.blk)
        s = r["s"][b]
        adj = (s > cfg.tau_edge) & ~np.eye(cfg.blk, dtype=bool)
        # planted links are exactly the edges (the generator's separation)
        assert (adj == w.links[b]).all()
        sel = np.nonzero(r["selected"][b])[0]
        assert is_independent(adj, sel) and is_maximal(adj, sel, nodes)


def test_dapd_preunmask_certain(oracle):
    """Positions of confidence exactly 1.0 join the selection on both paths."""
    g = __import__("json").load(open(os.path.join(GOLDEN, "dapd_mrf9.json")))
    n = len(g["nodes"])
    A = np.full((n, n), 0.001, np.float32)
    for a, b in g["edges"]:
        A[a, b] = A[b, a] = 0.1
    conf = np.array([[0.9, 0.8, 0.95, 0.7, 0.6, 0.99, 0.5, 0.85, 0.75]])
    conf[0, 6] = 1.0  # Y2: key 0.206, shut out by the kept X3 (order X3, X2, X4, Y2, Y1, ...)
    masked = np.ones((1, n), np.uint8)
    plain = oracle.dapd(A[None, None, None], masked, conf, tau_edge=0.05)
    pre = oracle.dapd(A[None, None, None], masked, conf, tau_edge=0.05, preunmask_certain=True)
    assert np.nonzero(plain["selected"][0])[0].tolist() == [2, 5, 8]
    assert np.nonzero(pre["selected"][0])[0].tolist() == [2, 5, 6, 8]
    assert pre["n_selected"][0] == 4
    # late phase: certain positions join the confidence rule's selection
    masked2 = np.zeros((1, n), np.uint8)
    masked2[0, [0, 1, 3]] = 1
    conf2 = np.array([[0.95, 1.0, 0.2, 0.3, 0, 0, 0, 0, 0]])
    r = oracle.dapd(A[None, None, None], masked2, conf2, tau_edge=0.05, preunmask_certain=True)
    assert r["path"][0] == 1 and np.nonzero(r["selected"][0])[0].tolist() == [0, 1]
