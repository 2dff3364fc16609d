"""Pins for the oracle's row statistics (argmax, confidence, LSE, entropy, KL).

The definitions come from "DepCap" (Methodology: I_k = KL(p_curr || p_prev),
H_k = H(p_curr), c_i = max_v p_i(v)) and the Fast-dLLM review (Method:
max-softmax confidence).  Each pin below is independent of the oracle's own
code: closed forms, scipy's library routines, and the chain rules of
log-sum-exp, entropy and KL over a split vocabulary.
"""
import math

import numpy as np
import pytest
from scipy import special, stats

import synth


def _bits(x, code):
    return synth.to_bf16_bits(x) if code == synth.BF16 else synth.to_f16_bits(x)


def _decoded(x, code):
    if code == synth.F32:
        return np.asarray(x, np.float64)
    if code == synth.BF16:
        return synth.from_bf16_bits(x).astype(np.float64)
    return x.view(np.float16).astype(np.float64)


def test_uniform_row_closed_form(oracle):
    V = 1000
    cur = np.full((3, V), 1.75, np.float32)
    out = oracle.row_stats(cur, cur.copy())
    assert np.all(out["argmax"] == 0)
    np.testing.assert_allclose(out["conf"], 1.0 / V, rtol=1e-12)
    np.testing.assert_allclose(out["entropy"], math.log(V), rtol=1e-12)
    np.testing.assert_allclose(out["lse"], 1.75 + math.log(V), rtol=1e-14)
    assert np.all(out["kl"] == 0.0)  # identical rows: every term is exactly zero


@pytest.mark.parametrize("a,b", [(3.0, 1.0), (0.5, 7.0), (-2.0, 2.0)])
def test_two_level_rows_closed_form(oracle, a, b):
    # one token at a (resp. b), V-1 tokens at 0
    V = 257
    cur = np.zeros((1, V), np.float32)
    prev = np.zeros((1, V), np.float32)
    cur[0, 5] = a
    prev[0, 5] = b
    out = oracle.row_stats(cur, prev)
    S = math.exp(a) + (V - 1)
    p_top, p_rest = math.exp(a) / S, 1.0 / S
    Sq = math.exp(b) + (V - 1)
    q_top, q_rest = math.exp(b) / Sq, 1.0 / Sq
    H = -(p_top * math.log(p_top) + (V - 1) * p_rest * math.log(p_rest))
    KL = p_top * math.log(p_top / q_top) + (V - 1) * p_rest * math.log(p_rest / q_rest)
    assert out["argmax"][0] == (5 if a > 0 else 0)
    assert out["conf"][0] == pytest.approx(max(p_top, p_rest), rel=1e-13)
    assert out["entropy"][0] == pytest.approx(H, rel=1e-12)
    assert out["kl"][0] == pytest.approx(KL, rel=1e-11, abs=1e-15)
    assert out["lse"][0] == pytest.approx(math.log(S), rel=1e-14)
    assert out["lse_prev"][0] == pytest.approx(math.log(Sq), rel=1e-14)


@pytest.mark.parametrize("code", [synth.F32, synth.BF16, synth.F16])
def test_against_scipy(oracle, code):
    rng = np.random.default_rng(7)
    R, V = 6, 3001
    x = (rng.standard_normal((R, V)) * 2).astype(np.float32)
    y = x + (rng.standard_normal((R, V)) * 0.3).astype(np.float32)
    x[1, 17] += 15.0
    if code != synth.F32:
        x, y = _bits(x, code), _bits(y, code)
    out = oracle.row_stats(x, y, dtype=None if code == synth.F32 else code)
    zx, zy = _decoded(x, code), _decoded(y, code)
    for r in range(R):
        p = special.softmax(zx[r])
        q = special.softmax(zy[r])
        assert out["argmax"][r] == int(np.argmax(zx[r]))
        assert out["lse"][r] == pytest.approx(special.logsumexp(zx[r]), rel=1e-13)
        assert out["lse_prev"][r] == pytest.approx(special.logsumexp(zy[r]), rel=1e-13)
        assert out["conf"][r] == pytest.approx(p.max(), rel=1e-12)
        assert out["entropy"][r] == pytest.approx(stats.entropy(p), rel=1e-11)
        assert out["kl"][r] == pytest.approx(np.sum(special.rel_entr(p, q)), rel=1e-9, abs=1e-14)


def test_argmax_ties_lowest_index(oracle):
    cur = np.zeros((2, 64), np.float32)
    cur[0, [9, 3, 40]] = 2.0
    cur[1, [63, 62]] = 5.0
    out = oracle.row_stats(cur)
    assert list(out["argmax"]) == [3, 62]


def test_vocab_split_chain_rules(oracle):
    """Stats over V equal the merge of the stats over two halves: LSE by
    log-add-exp, conf by rescaling, entropy and KL by their chain rules."""
    rng = np.random.default_rng(11)
    V = 4096
    x = (rng.standard_normal((4, V)) * 2).astype(np.float32)
    y = x + (rng.standard_normal((4, V)) * 0.5).astype(np.float32)
    full = oracle.row_stats(x, y)
    h = V // 2 + 37
    parts = [oracle.row_stats(np.ascontiguousarray(x[:, s]), np.ascontiguousarray(y[:, s]))
             for s in (slice(0, h), slice(h, V))]
    L = np.logaddexp(parts[0]["lse"], parts[1]["lse"])
    Lq = np.logaddexp(parts[0]["lse_prev"], parts[1]["lse_prev"])
    w = [np.exp(p["lse"] - L) for p in parts]
    wq = [np.exp(p["lse_prev"] - Lq) for p in parts]
    np.testing.assert_allclose(full["lse"], L, rtol=1e-13)
    np.testing.assert_allclose(full["lse_prev"], Lq, rtol=1e-13)
    np.testing.assert_allclose(full["conf"], np.maximum(w[0] * parts[0]["conf"], w[1] * parts[1]["conf"]),
                               rtol=1e-12)
    H = sum(wk * (p["entropy"] - np.log(wk)) for wk, p in zip(w, parts))
    np.testing.assert_allclose(full["entropy"], H, rtol=1e-12)
    KL = sum(wk * (p["kl"] + np.log(wk / wqk)) for wk, wqk, p in zip(w, wq, parts))
    np.testing.assert_allclose(full["kl"], KL, rtol=1e-10, atol=1e-14)
    am = np.where(parts[0]["lse"] + np.log(parts[0]["conf"]) >= parts[1]["lse"] + np.log(parts[1]["conf"]),
                  parts[0]["argmax"], parts[1]["argmax"] + h)
    np.testing.assert_array_equal(full["argmax"], am)


def test_invariants_on_workload_rows(oracle):
    w = synth.make(synth.scaled(synth.CONFIGS["llada_step"], vocab=8192, blk=16), seed=3)
    out = oracle.row_stats(w.cur, w.prev, dtype=synth.BF16)
    V = 8192
    assert np.all(out["kl"] >= -1e-12)
    assert np.all(out["entropy"] >= -1e-12) and np.all(out["entropy"] <= math.log(V) + 1e-12)
    assert np.all(out["conf"] >= 1.0 / V - 1e-15) and np.all(out["conf"] <= 1.0)
    np.testing.assert_allclose(out["lse"] + np.log(out["conf"]),
                               synth.from_bf16_bits(w.cur[np.arange(16), out["argmax"]]), rtol=1e-12)


def test_negative_infinity_logits(oracle):
    """Logits of -inf have probability 0 and drop out of every sum."""
    x = np.array([[0.5, -np.inf, 2.0, 1.0, -np.inf]], np.float32)
    y = np.array([[0.0, -np.inf, 1.0, 1.5, 3.0]], np.float32)
    out = oracle.row_stats(x, y)
    fin = np.isfinite(x[0])
    p = special.softmax(x[0][fin].astype(np.float64))
    q = special.softmax(y[0].astype(np.float64))[fin]
    assert out["argmax"][0] == 2
    assert out["entropy"][0] == pytest.approx(stats.entropy(p), rel=1e-13)
    assert out["kl"][0] == pytest.approx(np.sum(p * np.log(p / q)), rel=1e-12)


def test_row_index_scatter(oracle):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 100)).astype(np.float32)
    ri = np.array([6, 1, 3], np.int32)
    out = oracle.row_stats(x, row_index=ri)
    full = oracle.row_stats(x)
    for q in range(8):
        if q in ri:
            assert out["lse"][q] == full["lse"][q]
            assert out["argmax"][q] == full["argmax"][q]
        else:
            assert np.isnan(out["lse"][q]) and out["argmax"][q] == -1
