"""Pins of the oracle's revocable-decoding step (COVER page: Revocable
Parallel Diffusion Decoding; Method): a hand-worked three-step trace,
reductions to the threshold and top-K rules, the seed count and score
against numpy, and the state-update invariants."""
import math

import numpy as np

import oracle


def test_worked_three_steps():
    st = oracle.revocable_init(1, 6)
    kw = dict(tau_replace=0.9, tau_draft=0.9, draft_budget=2, w_unc=1.0, w_infl=0.0, w_drift=0.0, pi=0.5,
              cooldown=1, remask_budget=2)
    # step 0: 0.95, 0.99, 0.91 clear 0.9; the budget keeps the two most confident (2, 0)
    r = oracle.revocable_step(np.array([[5, 6, 7, 8, 9, 10]]), np.array([[0.95, 0.5, 0.99, 0.2, 0.91, 0.3]]),
                              st, 0, **kw)
    assert r["outcome"].tolist() == [[1, 0, 1, 0, 0, 0]]
    assert st["tok"].tolist() == [[5, -1, 7, -1, -1, -1]]
    # seeds: eligible {0, 2}, k = ceil(sqrt(2) * 0.5) = 1, score 1 - c: 0.05 vs 0.01 -> position 0
    assert st["seed"].tolist() == [[1, 0, 0, 0, 0, 0]] and st["last_seed"][0, 0] == 0
    # step 1: the seed re-predicts 3 != 5 with c 0.6 < 0.9 -> REMASK; drafting over {1, 3, 4, 5}
    r = oracle.revocable_step(np.array([[3, 6, 7, 8, 9, 10]]), np.array([[0.6, 0.92, 0.99, 0.3, 0.95, 0.1]]),
                              st, 1, **kw)
    assert r["outcome"].tolist() == [[4, 1, 0, 0, 1, 0]]
    assert r["n_drafted"].tolist() == [2] and r["n_revoked"].tolist() == [1]
    assert st["masked"].tolist() == [[1, 0, 0, 1, 0, 1]] and st["tok"].tolist() == [[-1, 6, 7, -1, 9, -1]]
    assert st["last_tok"][0, 0] == 5 and st["remasks"][0, 0] == 1
    # seeds: eligible {1, 2, 4} (0 masked), k = ceil(sqrt(3) * 0.5) = 1; scores 0.08, 0.01, 0.05 -> 1
    assert st["seed"].tolist() == [[0, 1, 0, 0, 0, 0]]
    # step 2: seed 1 re-predicts 4 != 6 with c 0.97 -> REPLACE; nothing masked clears 0.9 -> top-1
    # fallback picks position 0 (0.8), drafting 5 again = the token it lost: a flip-flop
    r = oracle.revocable_step(np.array([[5, 4, 7, 8, 9, 10]]), np.array([[0.8, 0.97, 0.99, 0.7, 0.95, 0.1]]),
                              st, 2, **kw)
    assert r["outcome"].tolist() == [[1, 3, 0, 0, 0, 0]]
    assert st["tok"].tolist() == [[5, 4, 7, -1, 9, -1]] and st["flipflops"].tolist() == [1]
    # seeds: eligible {0, 2, 4} (1 was a seed at step 1: 2 - 1 = 1, not > cooldown)
    # k = 1; scores 0.2, 0.01, 0.05 -> position 0
    assert st["seed"].tolist() == [[1, 0, 0, 0, 0, 0]]


def test_finished_sequence_is_unchanged():
    st = oracle.revocable_init(2, 4)
    st["masked"][0] = 0
    st["tok"][0] = [1, 2, 3, 4]
    st["seed"][0] = [1, 0, 1, 0]
    before = {k: v.copy() for k, v in st.items()}
    r = oracle.revocable_step(np.zeros((2, 4), np.int32), np.full((2, 4), 0.5), st, 3)
    for k in ("tok", "masked", "seed", "last_seed", "remasks", "last_tok"):
        np.testing.assert_array_equal(st[k][0], before[k][0])
    assert r["outcome"][0].tolist() == [0, 0, 0, 0] and r["n_drafted"][0] == 0


def test_drafting_reduces_to_threshold_and_topk():
    rng = np.random.default_rng(7)
    B, blk = 16, 40
    for trial in range(5):
        conf = rng.random((B, blk)) ** 0.3
        masked = (rng.random((B, blk)) < 0.6).astype(np.uint8)
        masked[0] = 1
        am = rng.integers(0, 100, (B, blk)).astype(np.int32)
        # no seeds, no budget: the Fast-dLLM threshold rule with its fallback
        st = oracle.revocable_init(B, blk)
        st["masked"][:] = masked
        st["tok"][:] = np.where(masked > 0, -1, 7)
        r = oracle.revocable_step(am, conf, st, 0, tau_draft=0.9, pi=0.0)
        sel, n = oracle.select_threshold(conf, masked, 0.9)
        np.testing.assert_array_equal((r["outcome"] == 1).astype(np.uint8), sel)
        np.testing.assert_array_equal(r["n_drafted"], n)
        # every masked position qualifies, budget K: the fixed top-K rule
        st = oracle.revocable_init(B, blk)
        st["masked"][:] = masked
        K = 1 + trial
        r = oracle.revocable_step(am, conf, st, 0, tau_draft=-1.0, draft_budget=K, pi=0.0)
        sel, n = oracle.select_topk(conf, masked, K)
        np.testing.assert_array_equal((r["outcome"] == 1).astype(np.uint8), sel)


def test_seed_count_and_score_against_numpy():
    rng = np.random.default_rng(8)
    B, blk = 12, 64
    conf = rng.random((B, blk))
    infl = rng.random((B, blk)) * 3
    drift = rng.random((B, blk)) * 0.5
    am = np.zeros((B, blk), np.int32)
    checked = 0
    for pi in (0.3, 1.0, 2.5):
        st = oracle.revocable_init(B, blk)
        st["masked"][:] = (rng.random((B, blk)) < 0.5).astype(np.uint8)
        st["masked"][:, 0] = 1
        st["tok"][:] = np.where(st["masked"] > 0, -1, 0)
        st["last_seed"][:] = np.where(rng.random((B, blk)) < 0.2, 4, -(2 ** 30))
        st["remasks"][:] = np.where(rng.random((B, blk)) < 0.2, 2, 0)
        oracle.revocable_step(am, conf, st, 5, tau_draft=2.0, pi=pi, w_unc=1.5, w_infl=0.7, w_drift=2.0,
                              cooldown=1, remask_budget=2, influence=infl, drift=drift)
        f = np.float32
        score = ((f(1.5) * (f(1) - conf.astype(f))) + f(0.7) * infl.astype(f)) - f(2.0) * drift.astype(f)
        for b in range(B):
            decoded = st["masked"][b] == 0
            # eligibility from the state before selection: not a seed at step 4 (5 - 4 = 1 is not > 1)
            # and fewer than 2 remasks
            lastseed_before = np.where(st["seed"][b] > 0, -(2 ** 30), st["last_seed"][b])
            elig = decoded & (5 - lastseed_before > 1) & (st["remasks"][b] < 2)
            n = int(elig.sum())
            k = min(n, math.ceil(float(np.float32(np.sqrt(np.float32(n))) * np.float32(pi))))
            idx = np.nonzero(elig)[0]
            order = idx[np.lexsort((idx, -score[b, idx]))]
            assert sorted(np.nonzero(st["seed"][b])[0].tolist()) == sorted(order[:k].tolist())
            # the same seeds as the exact (fp64) score wherever the k-th and
            # (k+1)-th exact scores are further apart than fp32 rounding
            exact = 1.5 * (1.0 - conf[b]) + 0.7 * infl[b] - 2.0 * drift[b]
            o64 = idx[np.lexsort((idx, -exact[idx]))]
            if 0 < k < n and exact[o64[k - 1]] - exact[o64[k]] > 1e-5:
                checked += 1
                assert sorted(np.nonzero(st["seed"][b])[0].tolist()) == sorted(o64[:k].tolist())
    assert checked >= 20


def test_invariants_random_runs():
    rng = np.random.default_rng(9)
    B, blk, V = 6, 24, 5
    st = oracle.revocable_init(B, blk)
    for step in range(60):
        if st["masked"].sum() == 0:
            break
        am = rng.integers(0, V, (B, blk)).astype(np.int32)
        conf = rng.random((B, blk)) ** 0.2
        before = {k: v.copy() for k, v in st.items()}
        r = oracle.revocable_step(am, conf, st, step, tau_replace=0.95, tau_draft=0.85, draft_budget=6, pi=0.8,
                                  remask_budget=2)
        out = r["outcome"]
        for b in range(B):
            if before["masked"][b].sum() == 0:
                assert (out[b] == 0).all()
                continue
            dec_before = int((before["masked"][b] == 0).sum())
            dec_after = int((st["masked"][b] == 0).sum())
            assert dec_after - dec_before == r["n_drafted"][b] - r["n_revoked"][b]     # net growth
            assert r["n_drafted"][b] >= 1                                               # progress
            assert ((out[b] == 1) <= (before["masked"][b] == 1)).all()                 # drafts were masked
            verified = (before["seed"][b] == 1) & (before["masked"][b] == 0)
            assert ((out[b] >= 2) == verified).all()                                    # every seed verified
            assert (st["tok"][b][st["masked"][b] == 1] == -1).all()
            assert (st["tok"][b][st["masked"][b] == 0] >= 0).all()
            assert (st["remasks"][b] <= 2).all()
            assert ((st["seed"][b] == 1) <= (st["masked"][b] == 0)).all()              # seeds are decoded
    assert st["masked"].sum() == 0


# ------------------------------------------------------------ influence
def test_influence_closed_form_permutation_attention():
    """One layer and head whose query q attends only to column pi(q): the
    influence of i is 1 when the query pointing at i is masked, else 0."""
    import oracle
    rng = np.random.default_rng(3)
    B, blk = 3, 17
    A = np.zeros((B, 1, 1, blk, blk), np.float32)
    perms = [rng.permutation(blk) for _ in range(B)]
    for b in range(B):
        A[b, 0, 0, np.arange(blk), perms[b]] = 1.0
    masked = (rng.random((B, blk)) < 0.5).astype(np.uint8)
    infl = oracle.attention_influence(A, masked)
    for b in range(B):
        want = np.zeros(blk)
        want[perms[b][masked[b] > 0]] = 1.0
        np.testing.assert_array_equal(infl[b], want)


def test_influence_of_row_stochastic_attention_sums_to_the_masked_count():
    """Rows softmaxed over the block (N = blk): every masked query spreads a
    unit of attention over the block, so the influences sum to the number of
    masked positions; with layers/heads averaged the same holds, and a
    block inside a larger map reads only the block."""
    import oracle
    rng = np.random.default_rng(4)
    B, L, H, blk = 4, 3, 5, 24
    x = np.exp(rng.standard_normal((B, L, H, blk, blk)))
    A = x / x.sum(-1, keepdims=True)
    masked = (rng.random((B, blk)) < 0.6).astype(np.uint8)
    infl = oracle.attention_influence(A.astype(np.float32), masked)
    np.testing.assert_allclose(infl.sum(-1), masked.sum(-1), rtol=1e-6)
    big = np.zeros((B, L, H, blk + 9, blk + 9), np.float32)
    big[:, :, :, 5:5 + blk, 5:5 + blk] = A
    np.testing.assert_array_equal(oracle.attention_influence(big, masked, block_start=5), infl)


def test_influence_identity_with_dapd_degree():
    """For a masked i, DAPD's d~_i = sum_{j in V_t, j != i} (a_ij + a_ji) / 2,
    so 2 d~_i = (row sum of a over masked columns) + infl_i - 2 a_ii: the
    influence pinned against the DAPD oracle's proxy degree."""
    import oracle
    import synth
    rng = np.random.default_rng(5)
    B, L, H, blk = 3, 2, 4, 32
    A = (rng.random((B, L, H, blk, blk)) ** 4 * 0.1).astype(np.float32)
    A16 = synth.to_f16_bits(A)
    masked = np.ones((B, blk), np.uint8)
    masked[:, ::5] = 0
    r = oracle.dapd(A16, masked, np.full((B, blk), 0.5), 0.05, dtype=synth.F16)
    infl = oracle.attention_influence(A16, masked, dtype=synth.F16)
    a = A16.view(np.float16).astype(np.float64).mean(axis=(1, 2))
    for b in range(B):
        assert r["path"][b] == 0
        for i in np.nonzero(masked[b])[0]:
            row = a[b, i, masked[b] > 0].sum()
            np.testing.assert_allclose(2 * r["dtilde"][b][i], row + infl[b][i] - 2 * a[b, i, i], rtol=1e-12)
