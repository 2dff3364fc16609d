"""GPU parity of dlm_row_stats against the fp64 oracle (through the C ABI).

Bar: argmax bit-exact; conf, lse, entropy, KL and lse_prev within
1e-4 absolute + 1e-4 relative.  Covers every workload at full size, the
split (cluster) and unsplit launch shapes, ragged vocabularies, exact ties,
-inf logits, a NaN row and the empty call.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import DeviceWorkload, close, gpu_stats, oracle_stats, to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dlm():
    import diffusion_decoding_token_gb300 as d
    d.lib()
    return d


def _compare(g, o, rows, with_prev=True):
    am = g.argmax.cpu().numpy()[rows]
    np.testing.assert_array_equal(am, o["argmax"][rows])
    for k in ("conf", "lse", "entropy") + (("kl", "lse_prev") if with_prev else ()):
        gv = getattr(g, k).cpu().numpy()[rows]
        ov = o[k][rows]
        ok = close(gv, ov)
        assert ok.all(), f"{k}: worst |g-o| {np.max(np.abs(gv - ov)):.3e} at row {rows[np.argmin(ok)]}"


@pytest.mark.parametrize("name", synth.ORDER)
def test_row_stats_workloads(dlm, name):
    w = synth.make(name, seed=1000 + synth.ORDER.index(name))
    dw = DeviceWorkload(w, compact_attn=True)
    st = dlm.new_status()
    g = gpu_stats(dw, status=st)
    o = oracle_stats(w)
    rows = np.nonzero(w.masked.reshape(-1))[0]
    _compare(g, o, rows)
    assert int(st.item()) == 0


@pytest.mark.parametrize("code", [synth.F32, synth.BF16, synth.F16])
@pytest.mark.parametrize("rows,V,stride", [(3, 1, 8), (5, 7, 8), (4, 1000, 1008), (2, 8193, 8200),
                                            (40, 126464, 126464), (1, 262147, 262152)])
def test_row_stats_shapes(dlm, code, rows, V, stride):
    """Ragged vocab tails, a single element, sub-vector rows, split rows."""
    rng = np.random.default_rng(rows * 7 + V)
    x = (rng.standard_normal((rows, stride)) * 2).astype(np.float32)
    y = x + (rng.standard_normal((rows, stride)) * 0.4).astype(np.float32)
    x[0, V - 1] += 9.0  # a peak in the tail
    if code == synth.F16:
        x, y = np.clip(x, -60000, 60000), np.clip(y, -60000, 60000)
    st = {synth.F32: lambda a: a, synth.BF16: synth.to_bf16_bits, synth.F16: synth.to_f16_bits}[code]
    xs, ys = st(x), st(y)
    o = oracle.row_stats(np.ascontiguousarray(xs[:, :V]), np.ascontiguousarray(ys[:, :V]),
                         dtype=None if code == synth.F32 else code)
    cur = to_torch(xs, code, "cuda")[:, :V]
    prev = to_torch(ys, code, "cuda")[:, :V]
    g = dlm.row_stats(cur, prev)
    _compare(g, o, np.arange(rows))


def test_ties_neg_inf_and_no_prev(dlm):
    V = 4096
    x = np.zeros((4, V), np.float32)
    x[0, [100, 37, 4000]] = 3.0          # tie -> 37
    x[1, :] = -np.inf
    x[1, [5, 9]] = [1.0, 2.0]           # mostly -inf row
    x[2, 2048:] = -np.inf
    x[3] = np.linspace(-5, 5, V, dtype=np.float32)
    xs = synth.to_bf16_bits(x)
    o = oracle.row_stats(xs, dtype=synth.BF16)
    g = dlm.row_stats(to_torch(xs, synth.BF16, "cuda"))
    _compare(g, o, np.arange(4), with_prev=False)
    assert g.kl is None and int(g.argmax[0]) == 37 and int(g.argmax[1]) == 9


def test_nan_row_sets_status(dlm):
    x = np.zeros((3, 512), np.float32)
    x[1, 77] = np.nan
    st = dlm.new_status()
    g = dlm.row_stats(to_torch(x, synth.F32, "cuda"), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & dlm.DEV_NONFINITE
    o = oracle.row_stats(x[[0, 2]])
    np.testing.assert_allclose(g.conf.cpu().numpy()[[0, 2]], o["conf"], rtol=1e-5)


def test_row_index_and_empty(dlm):
    rng = np.random.default_rng(3)
    x = synth.to_bf16_bits(rng.standard_normal((10, 2048)).astype(np.float32))
    ri = np.array([7, 2, 5], np.int32)
    cur = to_torch(x, synth.BF16, "cuda")
    out = dlm.RowStats(*[torch.full((10,), -5, dtype=dt, device="cuda") for dt in
                         (torch.int32, torch.float32, torch.float32, torch.float32, torch.float32, torch.float32)])
    g = dlm.row_stats(cur, row_index=torch.from_numpy(ri).cuda(), out=out)
    o = oracle.row_stats(x, dtype=synth.BF16)
    _compare(g, o, ri, with_prev=False)
    untouched = [q for q in range(10) if q not in ri]
    assert (g.lse.cpu().numpy()[untouched] == -5).all()
    # n_rows = 0 launches nothing and returns OK
    dlm.row_stats(cur[:0])


def test_split_and_unsplit_agree(dlm):
    """The same rows through a cluster-split launch (few rows) and an
    unsplit one (many rows) match the oracle and each other exactly."""
    w = synth.make(synth.scaled(synth.CONFIGS["llada_step"], blk=8), seed=11)
    dw = DeviceWorkload(w, compact_attn=True)
    few = dlm.row_stats(dw.cur, dw.prev)
    many_cur = dw.cur.repeat(64, 1)
    many_prev = dw.prev.repeat(64, 1)
    many = dlm.row_stats(many_cur, many_prev)
    o = oracle_stats(w)
    _compare(few, o, np.arange(8))
    for k in ("argmax", "conf", "lse", "entropy", "kl"):
        a = getattr(few, k).cpu().numpy()
        b = getattr(many, k).cpu().numpy()[:8]
        assert close(a, b, atol=2e-5, rtol=2e-5).all()


def test_all_nan_row_argmax_in_range(dlm):
    # a row holding only NaN has no maximum: its argmax is position 0 and the
    # status word flags it, so downstream gathers stay inside the row
    x = np.zeros((2, 4096), np.float32)
    x[0] = np.nan
    x[1, 1234] = 3.0
    st = dlm.new_status()
    g = dlm.row_stats(to_torch(x, synth.F32, "cuda"), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & dlm.DEV_NONFINITE
    assert int(g.argmax[0]) == 0 and int(g.argmax[1]) == 1234


@pytest.mark.parametrize("name,cuts", [("llada_step", (0, 40000, 90000)), ("tiny", (0, 512)),
                                       ("stress_bulk", (0, 8, 63232, 100000))])
def test_vocab_split_partials_merge_to_whole_rows(dlm, name, cuts):
    """Each vocabulary slice's partial states, merged in slice order, give the
    whole rows' statistics (against the oracle on whole rows); argmax is a
    global position."""
    cfg = synth.CONFIGS[name]
    w = synth.make(cfg, seed=77)
    code = cfg.logit_dtype
    cur = to_torch(w.cur, code, "cuda")
    prev = to_torch(w.prev, code, "cuda")
    V = cfg.vocab
    bounds = list(cuts) + [V]
    parts = torch.stack([dlm.row_stats_partial(cur[:, a:b], prev[:, a:b], vocab_offset=a)
                         for a, b in zip(bounds[:-1], bounds[1:])]).contiguous()
    st = dlm.new_status()
    g = dlm.row_stats_merge(parts, True, status=st)
    o = oracle.row_stats(w.cur, w.prev, dtype=None if code == synth.F32 else code)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare(g, o, np.arange(w.cur.shape[0]), with_prev=True)
    # without prev rows, and with a row index
    ri = torch.tensor([3, 0, 7], dtype=torch.int32, device="cuda")
    parts = torch.stack([dlm.row_stats_partial(cur[:, a:b], vocab_offset=a, row_index=ri,
                                               out=torch.zeros((cur.shape[0], 8), device="cuda"))
                         for a, b in zip(bounds[:-1], bounds[1:])]).contiguous()
    g2 = dlm.row_stats_merge(parts, False, row_index=ri)
    torch.cuda.synchronize()
    o2 = oracle.row_stats(w.cur[[3, 0, 7]], dtype=None if code == synth.F32 else code)
    for k in ("argmax", "conf", "lse", "entropy"):
        gv = getattr(g2, k).cpu().numpy()[[3, 0, 7]]
        if k == "argmax":
            np.testing.assert_array_equal(gv, o2[k])
        else:
            assert np.all(np.abs(gv - o2[k]) <= 1e-4 + 1e-4 * np.abs(o2[k])), k


def test_vocab_split_with_empty_and_nan_slices(dlm):
    # a slice of -inf only contributes nothing; a NaN slice flags the row
    x = np.random.default_rng(5).standard_normal((3, 96)).astype(np.float32)
    x[0, 32:64] = -np.inf
    x[1, 64:] = np.nan
    t = to_torch(x, synth.F32, "cuda")
    parts = torch.stack([dlm.row_stats_partial(t[:, a:a + 32], vocab_offset=a) for a in (0, 32, 64)]).contiguous()
    st = dlm.new_status()
    g = dlm.row_stats_merge(parts, False, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & dlm.DEV_NONFINITE
    o = oracle.row_stats(x[[0, 2]])
    np.testing.assert_array_equal(g.argmax.cpu().numpy()[[0, 2]], o["argmax"])
    assert np.all(np.abs(g.lse.cpu().numpy()[[0, 2]] - o["lse"]) <= 1e-4 + 1e-4 * np.abs(o["lse"]))


def test_tail_grid_of_half_rows(dlm):
    """Rows beyond whole waves of the GPU run as half rows in a second grid:
    the count query says so, and rows on both sides of the cut match the
    oracle (the batched workload's 2048 rows are checked in full above)."""
    L = dlm.lib()
    slots_rows = torch.cuda.get_device_properties(0).multi_processor_count * 4
    assert L.dlm_row_stats_launches(1, 1, slots_rows, 152064, 0) == 1
    assert L.dlm_row_stats_launches(1, 1, slots_rows + 37, 152064, 0) == 2
    assert L.dlm_row_stats_launches(1, 1, slots_rows + 37, 152064, 1) == 1
    rng = np.random.default_rng(9)
    R, V = slots_rows + 37, 8192
    x = synth.to_bf16_bits((rng.standard_normal((R, V)) * 2).astype(np.float32))
    xp = synth.to_bf16_bits((rng.standard_normal((R, V)) * 2).astype(np.float32))
    g = dlm.row_stats(to_torch(x, synth.BF16, "cuda"), to_torch(xp, synth.BF16, "cuda"))
    torch.cuda.synchronize()
    rows = np.array([0, slots_rows - 1, slots_rows, R - 1])
    o = oracle.row_stats(x[rows], xp[rows], dtype=synth.BF16)
    for k in ("argmax", "conf", "lse", "entropy", "kl", "lse_prev"):
        gv = getattr(g, k).cpu().numpy()[rows]
        if k == "argmax":
            np.testing.assert_array_equal(gv, o[k])
        else:
            assert close(gv, o[k]).all(), k


def test_single_grid_flag_same_statistics(dlm):
    """DLM_ROWS_SINGLE_GRID only changes how the rows are launched: the
    statistics agree with the two-grid pass (summation order aside)."""
    rows = torch.cuda.get_device_properties(0).multi_processor_count * 4 + 100
    rng = np.random.default_rng(11)
    x = synth.to_bf16_bits((rng.standard_normal((rows, 4096)) * 2).astype(np.float32))
    xp = synth.to_bf16_bits((rng.standard_normal((rows, 4096)) * 2).astype(np.float32))
    cur, prev = to_torch(x, synth.BF16, "cuda"), to_torch(xp, synth.BF16, "cuda")
    a = dlm.row_stats(cur, prev)
    b = dlm.row_stats(cur, prev, single_grid=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a.argmax.cpu().numpy(), b.argmax.cpu().numpy())
    for k in ("conf", "lse", "entropy", "kl", "lse_prev"):
        assert close(getattr(a, k).cpu().numpy(), getattr(b, k).cpu().numpy(), atol=2e-5, rtol=2e-5).all(), k


@pytest.mark.parametrize("trial", range(16))
def test_row_stats_random_shapes(dlm, trial):
    """Random row counts (one grid, tail grid, split rows), vocab sizes with
    ragged tails, padded strides, storage types, with and without the
    previous rows and a row index: every output within tolerance of the
    oracle, argmax exact."""
    rng = np.random.default_rng(900 + trial)
    rows = int(rng.choice([1, 3, 17, 150, 700, 1300]))
    V = int(rng.integers(1, 6000)) if rng.random() < 0.7 else int(rng.integers(6000, 40000))
    stride = (V + 7) // 8 * 8 + 8 * int(rng.integers(0, 3))
    code = int(rng.choice([synth.F32, synth.BF16, synth.F16]))
    with_prev = bool(rng.random() < 0.75)
    x = (rng.standard_normal((rows, stride)) * rng.uniform(0.5, 3.0)).astype(np.float32)
    hot = rng.integers(0, V, rows)
    x[np.arange(rows), hot] += rng.uniform(0, 12, rows).astype(np.float32)
    y = x + (rng.standard_normal((rows, stride)) * 0.3).astype(np.float32)
    st = {synth.F32: lambda a: a, synth.BF16: synth.to_bf16_bits, synth.F16: synth.to_f16_bits}[code]
    xs, ys = st(x), st(y)
    dcode = None if code == synth.F32 else code
    cur = to_torch(xs, code, "cuda")[:, :V]
    prev = to_torch(ys, code, "cuda")[:, :V] if with_prev else None
    if rng.random() < 0.4:   # a gathered subset of the rows, outputs at the row positions
        sel = np.sort(rng.choice(rows, max(1, rows // 2), replace=False)).astype(np.int32)
        out = dlm.alloc_row_stats(rows, "cuda", with_prev)
        g = dlm.row_stats(cur, prev, row_index=torch.from_numpy(sel).cuda(), out=out)
    else:
        sel = np.arange(rows)
        g = dlm.row_stats(cur, prev)
    o = oracle.row_stats(np.ascontiguousarray(xs[:, :V]), np.ascontiguousarray(ys[:, :V]) if with_prev else None,
                         dtype=dcode)
    _compare(g, o, sel, with_prev)


@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("rows,V", [(6, 126464), (700, 8192)])
def test_row_index_bounds_and_gather(dlm, rows, V, gather):
    """Row indices outside [0, n_src) -- negative, or past the rows the
    arrays hold -- are skipped: nothing is read or written for them and
    DLM_DEV_BAD_INDEX is set, on a cluster-split launch (6 rows) and on the
    tail grid of half rows (700 rows, bad entries among the last ones).  The
    other rows match the oracle, stored at q (default) or at r (gather)."""
    rng = np.random.default_rng(rows + int(gather))
    n_src = rows + 9
    x = (rng.standard_normal((n_src, V)) * 2).astype(np.float32)
    y = x + (rng.standard_normal((n_src, V)) * 0.3).astype(np.float32)
    xs, ys = synth.to_bf16_bits(x), synth.to_bf16_bits(y)
    ri = rng.permutation(n_src)[:rows].astype(np.int32)
    bad = [1, rows - 1, rows - 3]
    ri[bad] = [-3, n_src + 7, n_src]
    good = np.setdiff1d(np.arange(rows), bad)
    n_out = rows if gather else n_src
    out = dlm.RowStats(*[torch.full((n_out,), -5, dtype=dt, device="cuda") for dt in
                         (torch.int32, torch.float32, torch.float32, torch.float32, torch.float32, torch.float32)])
    st = dlm.new_status()
    g = dlm.row_stats(to_torch(xs, synth.BF16, "cuda"), to_torch(ys, synth.BF16, "cuda"),
                      row_index=torch.from_numpy(ri).cuda(), out=out, status=st, gather=gather)
    torch.cuda.synchronize()
    assert int(st.item()) == dlm.DEV_BAD_INDEX
    o = oracle.row_stats(xs, ys, dtype=synth.BF16, row_index=ri[good], n_out=n_src)
    if gather:   # outputs in gathered order: slot r holds row ri[r]
        o = {k: v[np.where(np.isin(np.arange(rows), good), ri, 0)] for k, v in o.items()}
        _compare(g, o, good)
        untouched = np.array(bad)
    else:
        _compare(g, o, ri[good])
        untouched = np.setdiff1d(np.arange(n_src), ri[good])
    assert (g.lse.cpu().numpy()[untouched] == -5).all() and (g.argmax.cpu().numpy()[untouched] == -5).all()


def test_merge_skips_row_indices_outside_the_partials(dlm):
    x = np.random.default_rng(8).standard_normal((5, 64)).astype(np.float32)
    t = to_torch(x, synth.F32, "cuda")
    parts = torch.stack([dlm.row_stats_partial(t[:, a:a + 32], vocab_offset=a) for a in (0, 32)]).contiguous()
    ri = torch.tensor([4, -1, 5, 0], dtype=torch.int32, device="cuda")      # 5 rows of partials: 5 is past them
    out = dlm.RowStats(*[torch.full((8,), -5, dtype=dt, device="cuda") for dt in
                         (torch.int32, torch.float32, torch.float32, torch.float32, torch.float32, torch.float32)])
    st = dlm.new_status()
    g = dlm.row_stats_merge(parts, False, row_index=ri, out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == dlm.DEV_BAD_INDEX
    o = oracle.row_stats(x[[4, 0]])
    np.testing.assert_array_equal(g.argmax.cpu().numpy()[[4, 0]], o["argmax"])
    assert close(g.lse.cpu().numpy()[[4, 0]], o["lse"]).all()
    assert (g.lse.cpu().numpy()[[1, 2, 3, 5, 6, 7]] == -5).all()
