"""Pins for the oracle's Fast-dLLM factor decoding, Theorem-1 certificate and
fixed top-K baseline (Fast-dLLM review: Method appendix variant, Key idea,
Prior limitations)."""
import numpy as np


def test_factor_worked_example(oracle):
    # sorted c: 0.99, 0.97, 0.9, 0.5 (positions 2, 0, 3, 1)
    # (n+1)(1-c^(n)): n=1: 0.02, n=2: 0.09, n=3: 0.4, n=4: 2.5
    conf = np.array([[0.97, 0.5, 0.99, 0.9]])
    m = np.ones((1, 4), np.uint8)
    for f, n in [(0.5, 3), (0.1, 2), (0.05, 1), (0.01, 1), (3.0, 4)]:
        sel, cnt = oracle.select_factor(conf, m, f)
        order = [2, 0, 3, 1]
        assert cnt[0] == n
        assert sorted(np.nonzero(sel[0])[0].tolist()) == sorted(order[:n])


def test_factor_brute_force_and_prefix(oracle):
    rng = np.random.default_rng(0)
    for _ in range(200):
        blk = int(rng.integers(1, 40))
        conf = 1 - rng.random((2, blk)) ** 3 * 0.5
        m = (rng.random((2, blk)) < 0.8).astype(np.uint8)
        f = float(rng.choice([0.05, 0.3, 1.0, 2.0]))
        sel, cnt = oracle.select_factor(conf, m, f)
        for b in range(2):
            idx = [i for i in range(blk) if m[b, i]]
            c32 = conf[b].astype(np.float32)
            order = sorted(idx, key=lambda i: (-c32[i], i))
            ok = [np.float32(n + 1) * (np.float32(1) - c32[order[n - 1]]) < np.float32(f) for n in range(1, len(order) + 1)]
            # the qualifying n form a prefix
            assert ok == sorted(ok, reverse=True)
            n = sum(ok) if any(ok) else (1 if order else 0)
            assert cnt[b] == n
            assert sorted(np.nonzero(sel[b])[0].tolist()) == sorted(order[:n])


def test_topk_brute_force(oracle):
    rng = np.random.default_rng(1)
    for _ in range(100):
        blk = int(rng.integers(1, 50))
        conf = rng.random((3, blk))
        conf[:, ::5] = 0.5  # ties
        m = (rng.random((3, blk)) < 0.7).astype(np.uint8)
        k = int(rng.integers(0, blk + 3))
        sel, cnt = oracle.select_topk(conf, m, k)
        for b in range(3):
            idx = [i for i in range(blk) if m[b, i]]
            c32 = conf[b].astype(np.float32)
            want = sorted(idx, key=lambda i: (-c32[i], i))[:k]
            assert sorted(np.nonzero(sel[b])[0].tolist()) == sorted(want)
            assert cnt[b] == len(want)


def test_certificate_inequality(oracle):
    conf = np.array([[0.7, 0.8, 0.1], [0.6, 0.9, 0.1], [0.1, 0.2, 0.3], [0.51, 0.2, 0.3]])
    sel = np.array([[1, 1, 0], [1, 1, 0], [0, 0, 0], [1, 0, 0]], np.uint8)
    # n=2: bound 1 - 1/3 = 0.667 -> [0.7, 0.8] certified, [0.6, 0.9] not;
    # empty selection certified; n=1: bound 0.5 -> 0.51 certified
    assert oracle.parallel_certificate(conf, sel).tolist() == [1, 0, 1, 1]
    rng = np.random.default_rng(2)
    for _ in range(100):
        c = rng.random((1, 20))
        s = (rng.random((1, 20)) < 0.3).astype(np.uint8)
        n = int(s.sum())
        cert = oracle.parallel_certificate(c, s)[0]
        cmin = np.float32(c[0][s[0] > 0].min()) if n else np.float32(1.0)
        # equivalent form of the theorem's condition: (n+1)(1 - c_min) < 1
        assert cert == (n == 0 or cmin > np.float32(1) - np.float32(1) / np.float32(n + 1))


def test_factor_with_f_one_is_certified(oracle):
    """Factor decoding at f = 1 commits exactly a set the Theorem-1 bound
    certifies, unless it had to fall back to the single top position."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        conf = 1 - rng.random((1, 32)) ** 2 * 0.6
        m = np.ones((1, 32), np.uint8)
        sel, cnt = oracle.select_factor(conf, m, 1.0)
        c32 = np.sort(conf[0].astype(np.float32))[::-1]
        fell_back = not (np.float32(2) * (np.float32(1) - c32[0]) < np.float32(1))
        if not fell_back:
            assert oracle.parallel_certificate(conf, sel)[0] == 1
