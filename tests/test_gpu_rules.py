"""GPU parity of the four selection rules against the oracle (through the C ABI).

Two levels, both on the pages' five workloads (six with the late phase of the
stress case) at full size, screened so that every oracle decision clears the
decision margins of ``parity.py`` (sequences that miss one are redrawn):
* unit parity -- each rule gets the SAME fp32 inputs on both sides (the
  oracle's statistics rounded to fp32), so the decisions must agree bit for
  bit: selections, counts, boundary lengths, pool order, degrees.  Float side
  outputs (S_k, D_ij, s_ij, d~_i) agree within 1e-4 abs + 1e-4 rel.
* pipeline parity -- GPU statistics feed GPU rules, oracle statistics feed
  oracle rules; every decision of every sequence must match exactly.
An unscreened draw of each workload is checked too: there the GPU's result
must be one that some resolution of the near-tied decisions gives.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import (DeviceWorkload, boundary_margin_failures, boundary_range, cap_outcomes, close,
                    dapd_late, dapd_margin_failures, dapd_outcomes, gpu_stats, oracle_stats, order_margin, screen,
                    sequence_decisions, threshold_outcome_check, to_torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dlm():
    import diffusion_decoding_token_gb300 as d
    d.lib()
    return d


_CACHE = {}


LITERAL = ["tiny:absolute", "llada_step:absolute"]


def workload(name, screened=True):
    """A workload by name; "<name>:absolute" is the literal reading of the
    logit boost (u added to the token's own value, so confidences stay below
    every threshold and the rules run on their fallbacks).  ``screened``:
    every sequence clears the decision margins (else the first draw)."""
    key = (name, screened)
    if key not in _CACHE:
        base, _, mode = name.partition(":")
        cfg = synth.CONFIGS[base] if not mode else synth.scaled(synth.CONFIGS[base], boost_mode=mode)
        seed = 1000 + synth.ORDER.index(base)
        if screened:
            w, o = screen(cfg, seed)
        else:
            w = synth.make(cfg, seed)
            o = oracle_stats(w)
        _CACHE.clear()
        _CACHE[key] = (w, DeviceWorkload(w), o)
    return _CACHE[key]


def f32(x):
    return np.nan_to_num(np.asarray(x, np.float64), nan=0.0).astype(np.float32)


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------ unit
def run_unit_threshold(dlm, cfg, w, o):
    B, blk = cfg.batch, cfg.blk
    c32 = f32(o["conf"]).reshape(B, blk)
    gs, gn = dlm.select_threshold(cuda(c32), cuda(w.masked), cfg.tau)
    os_, on = oracle.select_threshold(c32.astype(np.float64), w.masked, cfg.tau)
    np.testing.assert_array_equal(gs.cpu().numpy(), os_)
    np.testing.assert_array_equal(gn.cpu().numpy(), on)


def run_unit_boundary(dlm, cfg, w, o):
    B, blk = cfg.batch, cfg.blk
    kl32, en32 = f32(o["kl"]).reshape(B, blk), f32(o["entropy"]).reshape(B, blk)
    gl, gsc = dlm.depcap_boundary(cuda(kl32), cuda(en32), cfg.lam, cfg.L_min)
    ol, osc = oracle.depcap_boundary(kl32.astype(np.float64), en32.astype(np.float64), cfg.lam, cfg.L_min)
    assert close(gsc.cpu().numpy(), osc).all()
    gl = gl.cpu().numpy()
    for b in range(B):
        assert not boundary_margin_failures(osc[b]), b
        assert gl[b] == ol[b], b


def run_unit_cap(dlm, cfg, w, dw, o, scope=None):
    B, blk = cfg.batch, cfg.blk
    am = np.nan_to_num(o["argmax"]).astype(np.int32).reshape(B, blk)
    am[am < 0] = 0
    c32, l32 = f32(o["conf"]).reshape(B, blk), f32(o["lse"]).reshape(B, blk)
    D = torch.full((B, blk, blk), float("nan"), device="cuda")
    st = dlm.new_status()
    gs, gn = dlm.cap_select(dw.cur, cuda(am), cuda(c32), cuda(l32), dw.masked, cfg.tau_low, cfg.tau_high,
                            cfg.gamma, cfg.p_max, scope_len=None if scope is None else cuda(scope), D_out=D,
                            status=st)
    r = oracle.cap_select(w.cur, am, c32.astype(np.float64), l32.astype(np.float64), w.masked, cfg.tau_low,
                          cfg.tau_high, cfg.gamma, cfg.p_max, scope_len=scope, dtype=_code(cfg))
    gs, gn, D = gs.cpu().numpy(), gn.cpu().numpy(), D.cpu().numpy()
    for b in range(B):
        pn = r["pool_n"][b]
        pool = r["pool"][b][:pn]
        if pn:
            Dg = D[b][np.ix_(pool, pool)]
            Do = r["D"][b][np.ix_(pool, pool)]
            off = ~np.eye(pn, dtype=bool)
            assert close(Dg[off], Do[off]).all()
        np.testing.assert_array_equal(gs[b], r["selected"][b], err_msg=f"sequence {b}")
        assert gn[b] == r["n_selected"][b]
    assert bool(int(st.item()) & dlm.DEV_POOL_CLIPPED) == r["clipped"]


def _code(cfg):
    return None if cfg.logit_dtype == synth.F32 else cfg.logit_dtype


def run_unit_dapd(dlm, cfg, w, dw, o, order_mode=0, order_tol=None):
    """Graph outputs everywhere; selections compared on every sequence whose
    decisions clear the margins (all of them on a screened workload).
    Returns the number compared."""
    B, blk = cfg.batch, cfg.blk
    c32 = f32(o["conf"]).reshape(B, blk)
    s = torch.full((B, blk, blk), float("nan"), device="cuda")
    dt = torch.full((B, blk), float("nan"), device="cuda")
    deg = torch.full((B, blk), -1, dtype=torch.int32, device="cuda")
    gs, gn = dlm.dapd_graph_mis(dw.attn, dw.masked, cuda(c32), cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac,
                                order_mode, dw.block_start, s_out=s, dtilde_out=dt, deg_out=deg)
    code = None if cfg.attn_dtype == synth.F32 else cfg.attn_dtype
    r = oracle.dapd(w.attn, w.masked, c32.astype(np.float64), cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac,
                    order_mode, dtype=code)
    gs, gn, s, dt, deg = (t.cpu().numpy() for t in (gs, gn, s, dt, deg))
    compared = 0
    for b in range(B):
        m = w.masked[b].astype(bool)
        if r["path"][b] == 0:
            nodes = np.nonzero(m)[0]
            assert close(s[b][np.ix_(nodes, nodes)], r["s"][b][np.ix_(nodes, nodes)]).all()
            assert close(dt[b][nodes], r["dtilde"][b][nodes]).all()
            np.testing.assert_array_equal(deg[b][nodes], r["deg"][b][nodes])
        tol = order_margin(cfg, "dapd") if order_tol is None else order_tol
        cb = c32[b].astype(np.float64)
        if not dapd_margin_failures(cfg, cb, w.masked[b], r["s"][b], r["dtilde"][b], order_mode, order_tol=tol):
            np.testing.assert_array_equal(gs[b], r["selected"][b], err_msg=f"sequence {b}")
            assert gn[b] == r["n_selected"][b]
            compared += 1
        elif dapd_late(cfg, w.masked[b]):
            assert threshold_outcome_check(cb, w.masked[b], cfg.bulk_conf, gs[b])[0], b
        else:        # one of the results the near-tied decisions admit
            outs = dapd_outcomes(cfg, cb, w.masked[b], r["s"][b], r["dtilde"][b], order_mode)
            assert frozenset(np.nonzero(gs[b])[0].tolist()) in outs, b
    return compared


@pytest.mark.parametrize("name", synth.ORDER)
def test_unit_rules(dlm, name):
    w, dw, o = workload(name)
    cfg = w.cfg
    if "threshold" in cfg.rules:
        run_unit_threshold(dlm, cfg, w, o)
    scope = None
    if "boundary" in cfg.rules:
        run_unit_boundary(dlm, cfg, w, o)
        if name == "depcap_window":
            kl32, en32 = f32(o["kl"]).reshape(1, -1), f32(o["entropy"]).reshape(1, -1)
            scope, _ = oracle.depcap_boundary(kl32.astype(np.float64), en32.astype(np.float64), cfg.lam,
                                              cfg.L_min)
    if "cap" in cfg.rules:
        run_unit_cap(dlm, cfg, w, dw, o, scope)
    if "dapd" in cfg.rules:
        # on a screened workload every sequence is compared; the degree-only
        # order is exact on both sides for f16 attention (fixed-point sums in
        # the kernel, fp64 in the oracle), so it needs no margin there
        assert run_unit_dapd(dlm, cfg, w, dw, o) == cfg.batch
        if cfg.attn_dtype == synth.F16:
            assert run_unit_dapd(dlm, cfg, w, dw, o, order_mode=1, order_tol=0.0) == cfg.batch
        else:
            run_unit_dapd(dlm, cfg, w, dw, o, order_mode=1)


# -------------------------------------------------------------- pipeline
def check_rules_exact(name, w, o, sel, block_len):
    """Every decision of every sequence equal to the oracle's (GPU selections
    ``sel``: rule -> [B][blk] uint8; ``block_len``: [B] or None).  Returns
    the number of (rule, sequence) decisions compared."""
    cfg = w.cfg
    B, blk = cfg.batch, cfg.blk
    oconf = o["conf"].reshape(B, blk)
    exact = 0
    if "threshold" in cfg.rules:
        os_, _ = oracle.select_threshold(oconf, w.masked, cfg.tau)
        np.testing.assert_array_equal(sel["threshold"], os_)
        exact += B
    scope_o = None
    if "boundary" in cfg.rules:
        ol, _ = oracle.depcap_boundary(o["kl"].reshape(B, blk), o["entropy"].reshape(B, blk), cfg.lam, cfg.L_min)
        np.testing.assert_array_equal(block_len, ol)
        exact += B
        if name.startswith("depcap_window"):
            scope_o = ol
    if "cap" in cfg.rules:
        am = np.where(o["argmax"] < 0, 0, o["argmax"]).reshape(B, blk)
        r = oracle.cap_select(w.cur, am, oconf, o["lse"].reshape(B, blk), w.masked, cfg.tau_low, cfg.tau_high,
                              cfg.gamma, cfg.p_max, scope_len=scope_o, dtype=_code(cfg))
        for b in range(B):
            np.testing.assert_array_equal(sel["cap"][b], r["selected"][b], err_msg=f"CAP sequence {b}")
        exact += B
    if "dapd" in cfg.rules:
        code = None if cfg.attn_dtype == synth.F32 else cfg.attn_dtype
        r = oracle.dapd(w.attn, w.masked, oconf, cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0, dtype=code)
        for b in range(B):
            np.testing.assert_array_equal(sel["dapd"][b], r["selected"][b], err_msg=f"DAPD sequence {b}")
        exact += B
    return exact


def check_rules_valid(name, w, o, sel, block_len):
    """Unscreened draws: the GPU's result of each (rule, sequence) must be
    one that some resolution of the decisions inside the bands gives.
    Returns (unique, ambiguous): decisions with one admissible result
    (compared exactly) and with several."""
    cfg = w.cfg
    B, blk = cfg.batch, cfg.blk
    unique = ambiguous = 0
    for b in range(B):
        st = {k: v[b * blk:(b + 1) * blk] for k, v in o.items()}
        dec = sequence_decisions(w, b, st)
        c, m = st["conf"], w.masked[b]
        if "threshold" in cfg.rules:
            ok, u = threshold_outcome_check(c, m, cfg.tau, sel["threshold"][b])
            assert ok, f"threshold sequence {b}"
            unique, ambiguous = unique + u, ambiguous + (not u)
        scopes = [blk]
        if "boundary" in cfg.rules:
            lo, hi = boundary_range(dec["boundary"][1], cfg.L_min)
            assert lo <= block_len[b] <= hi, f"boundary sequence {b}: {block_len[b]} not in [{lo}, {hi}]"
            unique, ambiguous = unique + (lo == hi), ambiguous + (lo != hi)
            if name.startswith("depcap_window"):
                scopes = list(range(lo, hi + 1))
        if "cap" in cfg.rules:
            _, Dw, _ = dec["cap"]
            outs = set()
            for sc in scopes:
                outs |= cap_outcomes(cfg, c, m, Dw, sc)
            got = frozenset(np.nonzero(sel["cap"][b])[0].tolist())
            assert got in outs, f"CAP sequence {b}: {sorted(got)} is none of {len(outs)} admissible results"
            unique, ambiguous = unique + (len(outs) == 1), ambiguous + (len(outs) > 1)
        if "dapd" in cfg.rules:
            r = dec["dapd"]
            if dapd_late(cfg, m):
                ok, u = threshold_outcome_check(c, m, cfg.bulk_conf, sel["dapd"][b])
                assert ok, f"DAPD late phase sequence {b}"
            else:
                outs = dapd_outcomes(cfg, c, m, r["s"][0], r["dtilde"][0])
                got = frozenset(np.nonzero(sel["dapd"][b])[0].tolist())
                assert got in outs, f"DAPD sequence {b}: {sorted(got)} is none of {len(outs)} admissible results"
                u = len(outs) == 1
            unique, ambiguous = unique + u, ambiguous + (not u)
    return unique, ambiguous


def run_pipeline(dlm, name, dw, cfg, st):
    B, blk = cfg.batch, cfg.blk
    g = gpu_stats(dw, status=st)
    gconf, glse = g.conf.view(B, blk), g.lse.view(B, blk)
    sel, block_len, scope_g = {}, None, None
    if "threshold" in cfg.rules:
        sel["threshold"] = dlm.select_threshold(gconf, dw.masked, cfg.tau)[0].cpu().numpy()
    if "boundary" in cfg.rules:
        gl, _ = dlm.depcap_boundary(g.kl.view(B, blk), g.entropy.view(B, blk), cfg.lam, cfg.L_min)
        block_len = gl.cpu().numpy()
        if name.startswith("depcap_window"):
            scope_g = gl
    if "cap" in cfg.rules:
        sel["cap"] = dlm.cap_select(dw.cur, g.argmax.view(B, blk), gconf, glse, dw.masked, cfg.tau_low,
                                    cfg.tau_high, cfg.gamma, cfg.p_max, scope_len=scope_g)[0].cpu().numpy()
    if "dapd" in cfg.rules:
        sel["dapd"] = dlm.dapd_graph_mis(dw.attn, dw.masked, gconf, cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0,
                                         dw.block_start)[0].cpu().numpy()
    return g, sel, block_len


@pytest.mark.parametrize("name", synth.ORDER + LITERAL)
def test_pipeline(dlm, name):
    w, dw, o = workload(name)
    cfg = w.cfg
    st = dlm.new_status()
    g, sel, block_len = run_pipeline(dlm, name, dw, cfg, st)
    exact = check_rules_exact(name, w, o, sel, block_len)
    assert int(st.item()) == 0
    # no screened order gap is below 1e-5 relative (CAP on the stress graph
    # workload; DAPD keys there 1e-4, 1e-3 elsewhere): with every GPU
    # confidence within 5e-6 of the oracle's, no such pair can swap
    m = ~np.isnan(o["conf"])
    err = np.abs(g.conf.cpu().numpy()[m] - o["conf"][m]) / o["conf"][m]
    hi = o["conf"][m] >= 0.5
    assert err.max() < 5e-6, err.max()
    assert exact == cfg.batch * len(cfg.rules)
    print(f"{name}: {exact} exact, 0 validity-checked decisions (relative conf error: max {err.max():.2e}, "
          f"max over c >= 0.5 {err[hi].max() if hi.any() else 0.0:.2e})")


@pytest.mark.parametrize("name", synth.ORDER)
def test_pipeline_unscreened(dlm, name):
    """The first draw of each workload, not screened: each decision must be
    a result that some resolution of the near-tied decisions gives, and is
    compared exactly where only one result is admissible."""
    w, dw, o = workload(name, screened=False)
    cfg = w.cfg
    st = dlm.new_status()
    _, sel, block_len = run_pipeline(dlm, name, dw, cfg, st)
    assert int(st.item()) == 0
    unique, ambiguous = check_rules_valid(name, w, o, sel, block_len)
    print(f"{name} (unscreened): {unique} exact, {ambiguous} with several admissible results")
    assert unique + ambiguous == cfg.batch * len(cfg.rules)


@pytest.mark.parametrize("mode", ["rules", "whole"])
@pytest.mark.parametrize("name", ["batched", "stress_graph", "depcap_window", "llada_step", "tiny"])
def test_bench_launch_configuration_matches_oracle(dlm, name, mode):
    """The step as the benchmark times it -- one StepPlan with the DAPD
    attention pass on a side stream from the step's start, the other rules as
    parallel graph branches, the row pass's tail grid where it applies; two
    steps back to back, either as the benchmark's default runs them (row pass
    and DAPD chain launched, the rules replayed as a captured graph, timing
    events around the row pass) or captured whole in one CUDA graph with
    external timing events -- at full size, against the oracle."""
    w, dw, o = workload(name)
    cfg = w.cfg
    kw = dict(tau=cfg.tau, lam=cfg.lam, L_min=cfg.L_min, tau_low=cfg.tau_low, tau_high=cfg.tau_high,
              gamma=cfg.gamma, p_max=cfg.p_max, tau_edge=cfg.tau_edge, bulk_conf=cfg.bulk_conf,
              bulk_frac=cfg.bulk_frac, rules=tuple(cfg.rules), cap_scope_from_boundary=(cfg.name == "depcap_window"),
              concurrent_dapd=True, dapd_early=True, parallel_rules=True)
    if "dapd" in cfg.rules:
        kw.update(attn=dw.attn, block_start=dw.block_start)
    plan = dlm.StepPlan(dw.cur, dw.prev, dw.masked, row_index=dw.row_index, **kw)
    # the one-sequence step folds its DAPD attention sums into the row pass
    assert plan.folded == (name == "llada_step")
    _, hi = torch.cuda.Stream.priority_range()
    main = torch.cuda.Stream(priority=hi)
    external = mode == "whole"
    evs = [(torch.cuda.Event(enable_timing=True, external=external),
            torch.cuda.Event(enable_timing=True, external=external)) for _ in range(2)]
    with torch.cuda.stream(main):
        plan.run(main)
        torch.cuda.synchronize()
        g = None
        if external or plan.has_rules_after_rows:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=main):
                if external:
                    for e in evs:
                        plan.run(main, events=e)
                else:
                    plan.run(rules_only=True)
        for v in plan.out.values():
            v[0].fill_(7)
        if external:
            g.replay()
        else:
            for e in evs:
                plan.run_rows(main, events=e)
                if g is not None:
                    g.replay()
                plan.join(main)
    torch.cuda.synchronize()
    sel = {k: v[0].cpu().numpy() for k, v in plan.out.items()}
    block_len = None if plan.block_len is None else plan.block_len.cpu().numpy()
    exact = check_rules_exact(name, w, o, sel, block_len)
    assert int(plan.status.item()) == 0
    assert all(a.elapsed_time(b) > 0 for a, b in evs)
    assert exact == cfg.batch * len(cfg.rules)


def test_dapd_selection_waits_for_the_row_pass(dlm):
    """The DAPD selection follows the attention pass on the side stream, behind
    an event on the row pass.  With a one-head attention pass (done long
    before the 2048-row pass) and the statistics zeroed before the step, it
    must still read the row pass's confidences: its selection equals the one
    run again after a full synchronisation, and differs from what zeroed
    confidences give."""
    w, dw, o = workload("batched")
    cfg = w.cfg
    plan = dlm.StepPlan(dw.cur, dw.prev, dw.masked, tau_edge=cfg.tau_edge, bulk_conf=cfg.bulk_conf,
                        bulk_frac=cfg.bulk_frac, rules=("dapd",), attn=dw.attn[:, :1, :1],
                        block_start=dw.block_start, concurrent_dapd=True, dapd_early=True)
    _, hi = torch.cuda.Stream.priority_range()
    main = torch.cuda.Stream(priority=hi)
    sel, n = plan.out["dapd"]
    kw = dict(tau_edge=cfg.tau_edge, bulk_conf=cfg.bulk_conf, bulk_frac=cfg.bulk_frac)
    with torch.cuda.stream(main):
        plan.run(main)
        torch.cuda.synchronize()
        for t in plan.stats:
            if t is not None:
                t.zero_()
        sel.fill_(7)
        torch.cuda.synchronize()
        plan.run_rows(main)
        plan.join(main)
        torch.cuda.synchronize()
        got = sel.clone()
        ref, _ = dlm.dapd_select(plan.dapd_ws, dw.masked, plan.stats.conf, **kw)
        zero, _ = dlm.dapd_select(plan.dapd_ws, dw.masked, torch.zeros_like(plan.stats.conf), **kw)
    torch.cuda.synchronize()
    assert int(plan.status.item()) == 0
    assert torch.equal(got, ref)
    assert not torch.equal(zero, ref)


# ------------------------------------------------------------- edge cases
def test_threshold_edges(dlm):
    conf = np.array([[0.3, 0.5, 0.5, 0.1], [0.95, 0.2, 0.99, 0.3], [0.91, 0.2, 0.1, 0.95]], np.float32)
    masked = np.array([[1, 1, 1, 1], [0, 0, 0, 0], [1, 0, 0, 0]], np.uint8)
    gs, gn = dlm.select_threshold(cuda(conf), cuda(masked), 0.9)
    os_, on = oracle.select_threshold(conf.astype(np.float64), masked, 0.9)
    np.testing.assert_array_equal(gs.cpu().numpy(), os_)
    np.testing.assert_array_equal(gn.cpu().numpy(), on)
    assert gn.cpu().tolist() == [1, 0, 1]


@pytest.mark.parametrize("blk", [1, 5, 256])
def test_threshold_random_sizes(dlm, blk):
    rng = np.random.default_rng(blk)
    conf = rng.random((33, blk)).astype(np.float32)
    masked = (rng.random((33, blk)) < 0.6).astype(np.uint8)
    gs, gn = dlm.select_threshold(cuda(conf), cuda(masked), 0.9)
    os_, on = oracle.select_threshold(conf.astype(np.float64), masked, 0.9)
    np.testing.assert_array_equal(gs.cpu().numpy(), os_)
    np.testing.assert_array_equal(gn.cpu().numpy(), on)


@pytest.mark.parametrize("w_,mode", [(1, 0), (3, 0), (5, 1), (1, 2), (7, 2)])
def test_boundary_modes(dlm, w_, mode):
    rng = np.random.default_rng(w_ * 10 + mode)
    B, L = 17, 77
    I = rng.gamma(1.0, 1.0, (B, L)).astype(np.float32)
    H = rng.gamma(1.0, 1.0, (B, L)).astype(np.float32)
    cold = (rng.random(B) < 0.2).astype(np.uint8)
    gl, gsc = dlm.depcap_boundary(cuda(I), cuda(H), 1.2, 8, w_, mode, cold_start=cuda(cold))
    ol, osc = oracle.depcap_boundary(I.astype(np.float64), H.astype(np.float64), 1.2, 8, w_, mode, cold)
    assert close(gsc.cpu().numpy(), osc).all()
    gl = gl.cpu().numpy()
    for b in range(B):
        if cold[b]:
            assert gl[b] == ol[b]
        else:           # exact where no score sits within the margin of 0
            lo, hi = boundary_range(osc[b], 8)
            assert lo <= gl[b] <= hi and (lo < hi or gl[b] == ol[b]), b


@pytest.mark.parametrize("w_", [1, 3])
def test_boundary_ragged_windows(dlm, w_):
    """Per-sequence windows L_window = min(L_max, L_remain), including an
    empty one and windows shorter than L_min and the smoothing width."""
    rng = np.random.default_rng(40 + w_)
    B, Ls = 24, 64
    I = rng.gamma(1.0, 1.0, (B, Ls)).astype(np.float32)
    H = rng.gamma(1.0, 1.0, (B, Ls)).astype(np.float32)
    wl = rng.integers(0, Ls + 1, B).astype(np.int32)
    wl[:4] = [0, 1, 2, Ls]
    cold = (rng.random(B) < 0.2).astype(np.uint8)
    score = torch.full((B, Ls), float("nan"), device="cuda")
    gl, gsc = dlm.depcap_boundary(cuda(I), cuda(H), 1.2, 8, w_, 0, cold_start=cuda(cold), window_len=cuda(wl),
                                  score=score)
    ol, osc = oracle.depcap_boundary(I.astype(np.float64), H.astype(np.float64), 1.2, 8, w_, 0, cold,
                                     window_len=wl)
    gsc, gl = gsc.cpu().numpy(), gl.cpu().numpy()
    for b in range(B):
        n = wl[b]
        assert np.isnan(gsc[b, n:]).all()                    # nothing written past the window
        assert close(gsc[b, :n], osc[b, :n]).all()
        if cold[b]:
            assert gl[b] == ol[b], b
        else:
            lo, hi = boundary_range(osc[b, :n], 8)
            assert lo <= gl[b] <= hi and (lo < hi or gl[b] == ol[b]), b
    assert gl[0] == 0


@pytest.mark.parametrize("code", [synth.F32, synth.BF16, synth.F16])
@pytest.mark.parametrize("blk,p_maxes", [(37, (8, 37, 65)), (100, (64, 65, 100))])
def test_cap_edges(dlm, blk, p_maxes, code):
    """Pool clipping, an empty pool, scope limits, the unconditional tier and
    a ragged block, on small cases in each logit storage type; pools up to 64
    take the fused single-CTA kernel, larger ones the cluster kernel, and the
    pool is clipped on both sides of that line."""
    rng = np.random.default_rng(21 + blk)
    B, V = 4, 304
    z = (rng.standard_normal((B * blk, V)) * 1.0).astype(np.float32)
    tok = rng.integers(0, V, B * blk)
    for r in range(B * blk):
        if r % 5:
            z[r, tok[r]] = 10 + rng.uniform(0, 4)
    for r in range(0, B * blk - 1, 3):
        z[r, tok[r + 1]] = z[r, tok[r]] - 3
        z[r + 1, tok[r]] = z[r + 1, tok[r + 1]] - 3
    z[blk:2 * blk, :] = rng.standard_normal((blk, V)).astype(np.float32)  # sequence 1: no candidate
    zs = {synth.F32: lambda a: a, synth.BF16: synth.to_bf16_bits, synth.F16: synth.to_f16_bits}[code](z)
    dcode = None if code == synth.F32 else code
    o = oracle.row_stats(zs, dtype=dcode)
    masked = (rng.random((B, blk)) < 0.9).astype(np.uint8)
    scope = np.array([blk, blk, 11, 0], np.int32)
    am = o["argmax"].reshape(B, blk)
    c32, l32 = f32(o["conf"]).reshape(B, blk), f32(o["lse"]).reshape(B, blk)
    zt = to_torch(zs, code, "cuda")
    for p_max, htu in [(p_maxes[0], False), (p_maxes[1], False), (p_maxes[1], True), (p_maxes[2], True)]:
        st = dlm.new_status()
        gs, gn = dlm.cap_select(zt, cuda(am), cuda(c32), cuda(l32), cuda(masked), 0.8, 0.95, -16.0, p_max,
                                high_tier_unconditional=htu, scope_len=cuda(scope), status=st)
        r = oracle.cap_select(zs, am, c32.astype(np.float64), l32.astype(np.float64), masked, 0.8, 0.95, -16.0,
                              p_max, high_tier_unconditional=htu, scope_len=scope, dtype=dcode)
        np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
        np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
        assert bool(int(st.item()) & dlm.DEV_POOL_CLIPPED) == r["clipped"]


@pytest.mark.parametrize("blk,p_max", [(40, 32), (100, 100)])
def test_cap_row_index(dlm, blk, p_max):
    """CAP reading its logit rows through a row index: each sequence's block
    is a window at a random offset of a longer generation, in one case with
    the rows shuffled.  Equal to the oracle given the same index, and to the
    oracle on the rows laid out block-contiguously (fused kernel for pools up
    to 64, cluster kernel above).  A pool member whose row lies outside the
    logits is never read: its pairs score NaN and DLM_DEV_BAD_INDEX is set."""
    cfg = synth.scaled(synth.CONFIGS["depcap_window"], batch=3, blk=blk, vocab=4096, p_max=p_max, rules=("cap",))
    # both sides order the same fp32 confidences: only D_ij against gamma needs a margin
    w, o = screen(cfg, seed=60 + blk, use_stored=False, margins={"cap": 0.0})
    B, V = cfg.batch, cfg.vocab
    rng = np.random.default_rng(blk)
    N = blk + 37
    gen = synth.to_bf16_bits(rng.standard_normal((B * N, V)).astype(np.float32))
    cursor = rng.integers(0, N - blk + 1, B)
    ri = (np.arange(B)[:, None] * N + cursor[:, None] + np.arange(blk)[None, :]).reshape(-1).astype(np.int32)
    gen[ri] = w.cur
    am = np.where(o["argmax"] < 0, 0, o["argmax"]).astype(np.int32).reshape(B, blk)
    c32, l32 = f32(o["conf"]).reshape(B, blk), f32(o["lse"]).reshape(B, blk)
    ref = oracle.cap_select(w.cur, am, c32.astype(np.float64), l32.astype(np.float64), w.masked, cfg.tau_low,
                            cfg.tau_high, cfg.gamma, p_max, dtype=synth.BF16)
    for shuffle in (False, True):
        g_rows, idx = gen, ri
        if shuffle:     # the same rows stored in a random order
            perm = rng.permutation(B * N)
            g_rows = np.empty_like(gen)
            g_rows[perm] = gen
            idx = perm[ri].astype(np.int32)
        st = dlm.new_status()
        D = torch.full((B, blk, blk), float("nan"), device="cuda")
        gs, gn = dlm.cap_select(to_torch(g_rows, synth.BF16, "cuda"), cuda(am), cuda(c32), cuda(l32), dw_masked(w),
                                cfg.tau_low, cfg.tau_high, cfg.gamma, p_max, D_out=D, status=st,
                                row_index=cuda(idx))
        r = oracle.cap_select(g_rows, am, c32.astype(np.float64), l32.astype(np.float64), w.masked, cfg.tau_low,
                              cfg.tau_high, cfg.gamma, p_max, dtype=synth.BF16, row_index=idx)
        np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
        np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
        np.testing.assert_array_equal(r["selected"], ref["selected"])
        assert int(st.item()) & dlm.DEV_BAD_INDEX == 0
    # two pool members of sequence 0 point outside the logits
    pool0 = ref["pool"][0][:ref["pool_n"][0]]
    assert len(pool0) >= 3
    bad = ri.copy()
    bad[pool0[0]], bad[pool0[1]] = -1, B * N
    st = dlm.new_status()
    D = torch.full((B, blk, blk), float("nan"), device="cuda")
    dlm.cap_select(to_torch(gen, synth.BF16, "cuda"), cuda(am), cuda(c32), cuda(l32), dw_masked(w), cfg.tau_low,
                   cfg.tau_high, cfg.gamma, p_max, D_out=D, status=st, row_index=cuda(bad))
    torch.cuda.synchronize()
    assert int(st.item()) & dlm.DEV_BAD_INDEX
    D = D.cpu().numpy()[0]
    for i in pool0[:2]:
        others = [j for j in pool0 if j != i]
        assert np.isnan(D[i, others]).all() and np.isnan(D[others, i]).all()
    rest = pool0[2:]
    if len(rest) >= 2:
        sub = np.ix_(rest, rest)
        off = ~np.eye(len(rest), dtype=bool)
        assert close(D[sub][off], ref["D"][0][sub][off]).all()


def dw_masked(w):
    return cuda(w.masked)


@pytest.mark.parametrize("blk,M", [(30, 30), (30, 15), (30, 14), (256, 256), (9, 9), (64, 40), (65, 65),
                                   (100, 60), (127, 127), (200, 150)])
def test_dapd_edges(dlm, blk, M):
    """Ragged block (partial last vector), the 50% switch on both sides,
    the maximum block, and the page's 9-node MRF size."""
    rng = np.random.default_rng(blk * 100 + M)
    B, L, H = 3, 2, 3
    N = (blk + 24 + 7) // 8 * 8   # 16-byte aligned f16 rows
    bs = 8
    sub = rng.random((B, L, H, blk, blk)) ** 6 * 0.3
    sub = (sub / (sub.sum(-1, keepdims=True) + 1.0)).astype(np.float32)
    sub16 = synth.to_f16_bits(sub)
    full = torch.zeros((B, L, H, N, N), dtype=torch.float16, device="cuda")
    full[:, :, :, bs:bs + blk, bs:bs + blk] = to_torch(sub16, synth.F16, "cuda")
    masked = np.zeros((B, blk), np.uint8)
    for b in range(B):
        masked[b, rng.choice(blk, M, replace=False)] = 1
    conf = rng.random((B, blk)).astype(np.float32)
    tau = 0.02
    for om in (0, 1):
        s = torch.full((B, blk, blk), float("nan"), device="cuda")
        deg = torch.full((B, blk), -1, dtype=torch.int32, device="cuda")
        gs, gn = dlm.dapd_graph_mis(full, cuda(masked), cuda(conf), tau, 0.9, 0.5, om, bs, s_out=s, deg_out=deg)
        r = oracle.dapd(sub16, masked, conf.astype(np.float64), tau, 0.9, 0.5, om, dtype=synth.F16)
        np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
        np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
        for b in range(B):
            if r["path"][b] == 0:
                nodes = np.nonzero(masked[b])[0]
                np.testing.assert_array_equal(deg.cpu().numpy()[b][nodes], r["deg"][b][nodes])


@pytest.mark.parametrize("code", [synth.BF16, synth.F32])
@pytest.mark.parametrize("blk", [32, 100])
def test_dapd_attention_dtypes(dlm, code, blk):
    """bf16 and fp32 attention (bulk-copy path, one-CTA and cluster decide):
    the graph and the selection against the oracle on generated workloads
    with planted links, screened at the decision margins (fp32 sums are not
    exact); the degree-only order is compared exactly where its keys clear
    the margin and checked against the admissible results elsewhere."""
    cfg = synth.scaled(synth.CONFIGS["stress_graph"], batch=3, blk=blk, vocab=1024, seq_len=(blk + 96 + 7) // 8 * 8,
                       block_start=96, attn_dtype=code)
    w, o = screen(cfg, seed=17 + blk, use_stored=False)
    dw = DeviceWorkload(w)
    assert run_unit_dapd(dlm, cfg, w, dw, o) == cfg.batch
    assert run_unit_dapd(dlm, cfg, w, dw, o, order_mode=1) >= 2


@pytest.mark.parametrize("blk", [48, 100, 127])
def test_dapd_split_calls_float_outputs(dlm, blk):
    """dlm_dapd_graph with its float outputs, then dlm_dapd_select: the graph
    outputs and the selection match the oracle (one-CTA and cluster paths,
    even and odd blocks)."""
    rng = np.random.default_rng(blk)
    B, L, H, bs = 2, 2, 3, 8
    N = (blk + 24 + 7) // 8 * 8
    sub = rng.random((B, L, H, blk, blk)) ** 6 * 0.3
    sub = (sub / (sub.sum(-1, keepdims=True) + 1.0)).astype(np.float32)
    sub16 = synth.to_f16_bits(sub)
    full = torch.zeros((B, L, H, N, N), dtype=torch.float16, device="cuda")
    full[:, :, :, bs:bs + blk, bs:bs + blk] = to_torch(sub16, synth.F16, "cuda")
    masked = np.zeros((B, blk), np.uint8)
    for b in range(B):
        masked[b, rng.choice(blk, blk - b * (blk // 4), replace=False)] = 1
    conf = rng.random((B, blk)).astype(np.float32)
    tau = 0.02
    s = torch.full((B, blk, blk), float("nan"), device="cuda")
    dt = torch.full((B, blk), float("nan"), device="cuda")
    deg = torch.full((B, blk), -1, dtype=torch.int32, device="cuda")
    ws = dlm.dapd_graph(full, cuda(masked), tau, 0.9, 0.5, 0, bs, s_out=s, dtilde_out=dt, deg_out=deg)
    gs, gn = dlm.dapd_select(ws, cuda(masked), cuda(conf), tau, 0.9, 0.5, 0)
    r = oracle.dapd(sub16, masked, conf.astype(np.float64), tau, 0.9, 0.5, 0, dtype=synth.F16)
    np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
    np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
    for b in range(B):
        assert r["path"][b] == 0
        nodes = np.nonzero(masked[b])[0]
        np.testing.assert_array_equal(deg.cpu().numpy()[b][nodes], r["deg"][b][nodes])
        np.testing.assert_allclose(dt.cpu().numpy()[b][nodes], r["dtilde"][b][nodes], rtol=1e-4, atol=1e-4)
        sb = s.cpu().numpy()[b][np.ix_(nodes, nodes)]
        np.testing.assert_allclose(sb, r["s"][b][np.ix_(nodes, nodes)], rtol=1e-4, atol=1e-4)


def test_dapd_key_ties_break_to_lower_position(dlm):
    """Equal keys (identical rows and confidences) order by position."""
    blk = 16
    A = np.full((blk, blk), 0.001, np.float32)
    for i in range(0, blk - 1, 2):
        A[i, i + 1] = A[i + 1, i] = 0.25
    sub16 = synth.to_f16_bits(A[None, None, None])
    conf = np.full((1, blk), 0.5, np.float32)
    masked = np.ones((1, blk), np.uint8)
    gs, _ = dlm.dapd_graph_mis(to_torch(sub16, synth.F16, "cuda"), cuda(masked), cuda(conf), 0.1)
    r = oracle.dapd(sub16, masked, conf.astype(np.float64), 0.1, dtype=synth.F16)
    np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
    assert np.nonzero(r["selected"][0])[0].tolist() == list(range(0, blk, 2))


def test_dapd_broadcast_heads_uses_register_path(dlm):
    """A head-broadcast view (head stride 0) cannot be described to the bulk
    tensor engine; the register-load kernel must give the same answer."""
    rng = np.random.default_rng(77)
    B, L, H, blk, N, bs = 2, 3, 5, 40, 64, 16
    sub = (rng.random((B, L, 1, blk, blk)) ** 4 * 0.2).astype(np.float32)
    sub16 = synth.to_f16_bits(sub)
    full = torch.zeros((B, L, 1, N, N), dtype=torch.float16, device="cuda")
    full[:, :, :, bs:bs + blk, bs:bs + blk] = to_torch(sub16, synth.F16, "cuda")
    view = full.expand(B, L, H, N, N)
    assert view.stride(2) == 0
    masked = np.ones((B, blk), np.uint8)
    masked[1, ::3] = 0
    conf = rng.random((B, blk)).astype(np.float32)
    gs, gn = dlm.dapd_graph_mis(view, cuda(masked), cuda(conf), 0.05, block_start=bs)
    r = oracle.dapd(np.ascontiguousarray(np.broadcast_to(sub16, (B, L, H, blk, blk))), masked,
                    conf.astype(np.float64), 0.05, dtype=synth.F16)
    np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
    np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])


@pytest.mark.parametrize("name", ["llada_step", "stress_graph", "stress_bulk"])
def test_dapd_split_calls_match(dlm, name):
    """dlm_dapd_graph + dlm_dapd_select give exactly dlm_dapd_graph_mis."""
    w, dw, o = workload(name)
    cfg = w.cfg
    B, blk = cfg.batch, cfg.blk
    c32 = cuda(f32(o["conf"]).reshape(B, blk))
    ga, na = dlm.dapd_graph_mis(dw.attn, dw.masked, c32, cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0,
                                dw.block_start)
    ws = dlm.dapd_graph(dw.attn, dw.masked, cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0, dw.block_start)
    gb, nb = dlm.dapd_select(ws, dw.masked, c32, cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0)
    np.testing.assert_array_equal(ga.cpu().numpy(), gb.cpu().numpy())
    np.testing.assert_array_equal(na.cpu().numpy(), nb.cpu().numpy())


def test_step_plan_concurrent_matches_serial(dlm):
    """The step plan with the DAPD graph on a side stream gives the same
    selections as the single-stream plan, over several steps."""
    w, dw, o = workload("llada_step")
    cfg = w.cfg
    kw = dict(tau=cfg.tau, lam=cfg.lam, L_min=cfg.L_min, tau_low=cfg.tau_low, tau_high=cfg.tau_high,
              gamma=cfg.gamma, p_max=cfg.p_max, tau_edge=cfg.tau_edge, attn=dw.attn, block_start=dw.block_start)
    serial = dlm.StepPlan(dw.cur, dw.prev, dw.masked, **kw)
    plans = [dlm.StepPlan(dw.cur, dw.prev, dw.masked, concurrent_dapd=True, **kw),
             dlm.StepPlan(dw.cur, dw.prev, dw.masked, concurrent_dapd=True, dapd_early=True, **kw),
             dlm.StepPlan(dw.cur, dw.prev, dw.masked, parallel_rules=True, **kw),
             dlm.StepPlan(dw.cur, dw.prev, dw.masked, concurrent_dapd=True, parallel_rules=True, **kw),
             dlm.StepPlan(dw.cur, dw.prev, dw.masked, concurrent_dapd=True, dapd_early=True, parallel_rules=True,
                          **kw)]
    graphed = [dlm.StepPlan(dw.cur, dw.prev, dw.masked, concurrent_dapd=True, dapd_early=early,
                            parallel_rules=True, **kw) for early in (False, True)]
    _, hi = torch.cuda.Stream.priority_range()
    main = torch.cuda.Stream(priority=hi)
    torch.cuda.synchronize()
    with torch.cuda.stream(main):
        graphs = []
        for p in graphed:      # the rules captured as a CUDA graph, as the benchmark runs them
            p.run()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=main):
                p.run(rules_only=True)
            graphs.append(g)
        for _ in range(3):
            serial.run()
            for p in plans:
                p.run()
            for p, g in zip(graphed, graphs):
                p.run_rows(main)
                g.replay()
                p.join(main)
    torch.cuda.synchronize()
    plans += graphed
    for conc in plans:
        for k in serial.out:
            np.testing.assert_array_equal(serial.out[k][0].cpu().numpy(), conc.out[k][0].cpu().numpy())
            np.testing.assert_array_equal(serial.out[k][1].cpu().numpy(), conc.out[k][1].cpu().numpy())
        np.testing.assert_array_equal(serial.block_len.cpu().numpy(), conc.block_len.cpu().numpy())


@pytest.mark.parametrize("n_masked", [48, 20])
def test_dapd_preunmask_certain(dlm, n_masked):
    """Masked positions whose confidence is exactly 1.0 join the selection
    (graph path with 48/48 masked, late phase with 20/48)."""
    rng = np.random.default_rng(n_masked)
    B, L, H, blk = 3, 2, 4, 48
    sub = (rng.random((B, L, H, blk, blk)) ** 5 * 0.3).astype(np.float32)
    sub16 = synth.to_f16_bits(sub)
    masked = np.zeros((B, blk), np.uint8)
    for b in range(B):
        masked[b, rng.choice(blk, n_masked, replace=False)] = 1
    conf = rng.random((B, blk)).astype(np.float32)
    conf[:, ::5] = 1.0
    for flag in (False, True):
        gs, gn = dlm.dapd_graph_mis(to_torch(sub16, synth.F16, "cuda"), cuda(masked), cuda(conf), 0.05,
                                    preunmask_certain=flag)
        r = oracle.dapd(sub16, masked, conf.astype(np.float64), 0.05, dtype=synth.F16, preunmask_certain=flag)
        np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
        np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])


@pytest.mark.parametrize("p_max", [4, 128])
def test_cap_out_of_vocab_token_is_not_gathered(dlm, p_max):
    """A caller-supplied token outside [0, V) scores NaN (no conflict) on both
    CAP paths (fused for pools <= 64, three launches above) and sets the
    status word; the valid pairs are still decided."""
    V, blk = 16, 4
    z = np.full((blk, V), -30.0, np.float32)
    am = np.array([[3, 100000, 3, 1]], np.int32)
    for i, t in enumerate(am[0]):
        if t < V:
            z[i, t] = 10.0
    z[0, 3] = z[2, 3] = 10.0          # rows 0 and 2 share token 3: they conflict
    lse = np.log(np.exp(z.astype(np.float64)).sum(-1)).astype(np.float32)
    conf = np.array([[0.99, 0.98, 0.97, 0.96]], np.float32)
    st = dlm.new_status()
    sel, n = dlm.cap_select(cuda(z), cuda(am), cuda(conf), cuda(lse[None]), cuda(np.ones((1, blk), np.uint8)),
                            0.8, 0.95, -16.0, p_max, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & dlm.DEV_NONFINITE
    s = sel.cpu().numpy()[0]
    assert s[0] == 1 and s[2] == 0 and s[1] == 1 and s[3] == 1   # only the 0-2 conflict removes a position


def test_whole_steps_as_one_graph_match_eager(dlm):
    """Steps captured back to back in one CUDA graph, with external timing
    events around each row pass (the benchmark's timed form), give the same
    selections as eager steps."""
    w, dw, o = workload("llada_step")
    cfg = w.cfg
    kw = dict(tau=cfg.tau, lam=cfg.lam, L_min=cfg.L_min, tau_low=cfg.tau_low, tau_high=cfg.tau_high,
              gamma=cfg.gamma, p_max=cfg.p_max, tau_edge=cfg.tau_edge, attn=dw.attn, block_start=dw.block_start,
              concurrent_dapd=True, dapd_early=True, parallel_rules=True)
    eager = dlm.StepPlan(dw.cur, dw.prev, dw.masked, **kw)
    graphed = dlm.StepPlan(dw.cur, dw.prev, dw.masked, **kw)
    _, hi = torch.cuda.Stream.priority_range()
    main = torch.cuda.Stream(priority=hi)
    evs = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
           for _ in range(3)]
    with torch.cuda.stream(main):
        eager.run(main)
        graphed.run(main)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            for e in evs:
                graphed.run(main, events=e)
        for v in graphed.out.values():
            v[0].zero_()
        g.replay()
        eager.run(main)
    torch.cuda.synchronize()
    for k in eager.out:
        np.testing.assert_array_equal(eager.out[k][0].cpu().numpy(), graphed.out[k][0].cpu().numpy())
        np.testing.assert_array_equal(eager.out[k][1].cpu().numpy(), graphed.out[k][1].cpu().numpy())
    assert all(a.elapsed_time(b) > 0 for a, b in evs)


# ------------------------------------------------------------------ fuzz
@pytest.mark.parametrize("trial", range(12))
def test_cap_random_shapes(dlm, trial):
    """Random block sizes (both kernels), pool caps, masks, scopes and tiers
    on fp32 logits with planted conflicts: selections, counts and the clip
    flag equal the oracle's."""
    rng = np.random.default_rng(500 + trial)
    blk = int(rng.integers(1, 257))
    B = int(rng.integers(1, 5))
    V = int(rng.integers(1, 64)) * 8
    p_max = int(rng.integers(1, blk + 1)) if rng.random() < 0.5 else blk
    z = rng.standard_normal((B * blk, V)).astype(np.float32)
    tok = rng.integers(0, V, B * blk)
    boosted = rng.random(B * blk) < 0.7
    z[np.arange(B * blk)[boosted], tok[boosted]] += rng.uniform(6, 14, int(boosted.sum())).astype(np.float32)
    for r in range(0, B * blk - 1, 4):   # cross-boosted pairs: D near -6, a conflict
        z[r, tok[r + 1]] = z[r, tok[r]] - 3
        z[r + 1, tok[r]] = z[r + 1, tok[r + 1]] - 3
    o = oracle.row_stats(z)
    masked = (rng.random((B, blk)) < rng.uniform(0.3, 1.0)).astype(np.uint8)
    scope = rng.integers(0, blk + 1, B).astype(np.int32) if rng.random() < 0.5 else None
    htu = bool(rng.random() < 0.3)
    am = o["argmax"].reshape(B, blk)
    c32, l32 = f32(o["conf"]).reshape(B, blk), f32(o["lse"]).reshape(B, blk)
    st = dlm.new_status()
    gs, gn = dlm.cap_select(cuda(z), cuda(am), cuda(c32), cuda(l32), cuda(masked), 0.8, 0.95, -16.0, p_max,
                            high_tier_unconditional=htu, scope_len=None if scope is None else cuda(scope),
                            status=st)
    r = oracle.cap_select(z, am, c32.astype(np.float64), l32.astype(np.float64), masked, 0.8, 0.95, -16.0,
                          p_max, high_tier_unconditional=htu, scope_len=scope)
    np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
    np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
    assert bool(int(st.item()) & dlm.DEV_POOL_CLIPPED) == r["clipped"]


@pytest.mark.parametrize("trial", range(12))
def test_dapd_random_shapes(dlm, trial):
    """Random block sizes (one-CTA and cluster decide), layer/head counts,
    masks on both sides of the 50 % switch and both key orders, on f16
    attention (exact graph arithmetic): selections, counts and degrees equal
    the oracle's."""
    rng = np.random.default_rng(700 + trial)
    blk = int(rng.integers(1, 257))
    B = int(rng.integers(1, 4))
    L, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    bs = 8 * int(rng.integers(0, 4))
    N = (bs + blk + 8 + 7) // 8 * 8
    sub = rng.random((B, L, H, blk, blk)) ** 6 * 0.3
    sub = (sub / (sub.sum(-1, keepdims=True) + 1.0)).astype(np.float32)
    sub16 = synth.to_f16_bits(sub)
    full = torch.zeros((B, L, H, N, N), dtype=torch.float16, device="cuda")
    full[:, :, :, bs:bs + blk, bs:bs + blk] = to_torch(sub16, synth.F16, "cuda")
    masked = (rng.random((B, blk)) < rng.uniform(0.2, 1.0)).astype(np.uint8)
    conf = rng.random((B, blk)).astype(np.float32)
    om = int(rng.integers(0, 2))
    deg = torch.full((B, blk), -1, dtype=torch.int32, device="cuda")
    gs, gn = dlm.dapd_graph_mis(full, cuda(masked), cuda(conf), 0.02, 0.9, 0.5, om, bs, deg_out=deg)
    r = oracle.dapd(sub16, masked, conf.astype(np.float64), 0.02, 0.9, 0.5, om, dtype=synth.F16)
    np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
    np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
    for b in range(B):
        if r["path"][b] == 0:
            nodes = np.nonzero(masked[b])[0]
            np.testing.assert_array_equal(deg.cpu().numpy()[b][nodes], r["deg"][b][nodes])


# ------------------------------------------------------- fused row pass + rules
FUSED = ["tiny", "llada_step", "depcap_window", "batched"]


@pytest.mark.parametrize("name", FUSED)
def test_fused_rules_match_oracle(dlm, name):
    """dlm_row_stats_rules (threshold, boundary and CAP run by the CTA that
    finishes each sequence's last row) on the screened workloads: every
    decision equals the oracle's, the statistics match it within 1e-4, and a
    second call on the same workspace (its counters left at zero) gives the
    same results."""
    w, dw, o = workload(name)
    cfg = w.cfg
    B, blk = cfg.batch, cfg.blk
    rules = tuple(r for r in cfg.rules if r in ("threshold", "boundary", "cap"))
    ws = dlm.row_stats_rules_workspace(B, "cuda")
    outs = []
    for _ in range(2):
        st = dlm.new_status()
        r = dlm.row_stats_rules(dw.cur, dw.prev, dw.masked, rules=rules, tau=cfg.tau, lam=cfg.lam, L_min=cfg.L_min,
                                tau_low=cfg.tau_low, tau_high=cfg.tau_high, gamma=cfg.gamma, p_max=cfg.p_max,
                                cap_scope_from_boundary=(name == "depcap_window"), workspace=ws, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        sel = {k: r[k][0].cpu().numpy() for k in ("threshold", "cap") if k in rules}
        block_len = r["block_len"].cpu().numpy() if "boundary" in rules else None
        w3 = dataclasses.replace(w, cfg=synth.scaled(cfg, rules=rules))      # the three fused rules only
        assert check_rules_exact(name, w3, o, sel, block_len) == B * len(rules)
        g = r["stats"]
        for k in ("conf", "lse", "entropy", "kl"):
            assert close(getattr(g, k).cpu().numpy(), o[k]).all(), k
        np.testing.assert_array_equal(g.argmax.cpu().numpy(), o["argmax"])
        outs.append((sel, block_len))
        assert int(ws.sum().item()) == 0                      # the counters are back at zero
    for k in outs[0][0]:
        np.testing.assert_array_equal(outs[0][0][k], outs[1][0][k])


@pytest.mark.parametrize("trial", range(10))
def test_fused_rules_random_shapes(dlm, trial):
    """Random blocks (1-256 positions, pools up to 64), vocabularies, masks,
    cold starts and rule subsets: the fused call's rule outputs equal the
    separate rule calls run on the fused call's own statistics, and its
    statistics equal a plain row pass within 1e-5."""
    rng = np.random.default_rng(900 + trial)
    blk = int(rng.integers(1, 257))
    B = int(rng.integers(1, 6))
    V = int(rng.integers(1, 200)) * 8
    z = rng.standard_normal((B * blk, V)).astype(np.float32)
    tok = rng.integers(0, V, B * blk)
    boost = rng.random(B * blk) < 0.7
    z[np.arange(B * blk)[boost], tok[boost]] += rng.uniform(4, 12, int(boost.sum())).astype(np.float32)
    for r_ in range(0, B * blk - 1, 4):
        z[r_, tok[r_ + 1]] = z[r_, tok[r_]] - 3
    zp = z + (rng.standard_normal(z.shape) * 0.4).astype(np.float32)
    cur, prev = cuda(z), cuda(zp)
    masked = cuda((rng.random((B, blk)) < rng.uniform(0.3, 1.0)).astype(np.uint8))
    cold = cuda((rng.random(B) < 0.3).astype(np.uint8))
    subsets = [("threshold", "boundary", "cap"), ("threshold",), ("boundary", "cap"), ("cap",), ("boundary",)]
    rules = subsets[trial % len(subsets)]
    scoped = "boundary" in rules and "cap" in rules and trial % 2 == 0
    p_max = int(rng.integers(1, min(64, blk) + 1))
    L_min = int(rng.integers(1, 9))
    kw = dict(tau=0.9, lam=1.2, L_min=L_min, tau_low=0.8, tau_high=0.95, gamma=-16.0, p_max=p_max)
    r = dlm.row_stats_rules(cur, prev, masked, rules=rules, cold_start=cold, cap_scope_from_boundary=scoped, **kw)
    g = r["stats"]
    plain = dlm.row_stats(cur, prev)
    for k in ("conf", "lse", "entropy", "kl"):
        np.testing.assert_allclose(getattr(g, k).cpu().numpy(), getattr(plain, k).cpu().numpy(), rtol=1e-5,
                                   atol=1e-5)
    conf, lse, am = g.conf.view(B, blk), g.lse.view(B, blk), g.argmax.view(B, blk)
    if "threshold" in rules:
        s, n = dlm.select_threshold(conf, masked, 0.9)
        np.testing.assert_array_equal(r["threshold"][0].cpu().numpy(), s.cpu().numpy())
        np.testing.assert_array_equal(r["threshold"][1].cpu().numpy(), n.cpu().numpy())
    if "boundary" in rules:
        bl, sc = dlm.depcap_boundary(g.kl.view(B, blk), g.entropy.view(B, blk), 1.2, L_min, cold_start=cold)
        np.testing.assert_array_equal(r["block_len"].cpu().numpy(), bl.cpu().numpy())
        np.testing.assert_array_equal(r["score"].cpu().numpy(), sc.cpu().numpy())
    if "cap" in rules:
        s, n = dlm.cap_select(cur, am, conf, lse, masked, 0.8, 0.95, -16.0, p_max,
                              scope_len=r["block_len"] if scoped else None)
        np.testing.assert_array_equal(r["cap"][0].cpu().numpy(), s.cpu().numpy())
        np.testing.assert_array_equal(r["cap"][1].cpu().numpy(), n.cpu().numpy())


@pytest.mark.parametrize("name", ["batched", "depcap_window", "llada_step"])
def test_bench_launch_configuration_fused_rules(dlm, name):
    """The benchmark's step with the rules fused into the row pass (StepPlan
    fuse_rules), captured as two back-to-back steps in a CUDA graph, against
    the oracle."""
    w, dw, o = workload(name)
    cfg = w.cfg
    kw = dict(tau=cfg.tau, lam=cfg.lam, L_min=cfg.L_min, tau_low=cfg.tau_low, tau_high=cfg.tau_high,
              gamma=cfg.gamma, p_max=cfg.p_max, tau_edge=cfg.tau_edge, bulk_conf=cfg.bulk_conf,
              bulk_frac=cfg.bulk_frac, rules=tuple(cfg.rules), cap_scope_from_boundary=(cfg.name == "depcap_window"),
              concurrent_dapd=True, dapd_early=True, parallel_rules=True, fuse_rules=True)
    if "dapd" in cfg.rules:
        kw.update(attn=dw.attn, block_start=dw.block_start)
    plan = dlm.StepPlan(dw.cur, dw.prev, dw.masked, **kw)
    assert set(plan.fused) == {r for r in cfg.rules if r != "dapd"}
    _, hi = torch.cuda.Stream.priority_range()
    main = torch.cuda.Stream(priority=hi)
    with torch.cuda.stream(main):
        plan.run(main)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            for _ in range(2):
                plan.run(main)
        for v in plan.out.values():
            v[0].fill_(7)
        g.replay()
    torch.cuda.synchronize()
    sel = {k: v[0].cpu().numpy() for k, v in plan.out.items()}
    block_len = None if plan.block_len is None else plan.block_len.cpu().numpy()
    assert check_rules_exact(name, w, o, sel, block_len) == cfg.batch * len(cfg.rules)
    assert int(plan.status.item()) == 0


# ------------------------------------------------ attention folded into the row pass
def _sums(ws, B, blk):
    """The exact attention sums A ([B][blk][blk] int64) at the head of a DAPD workspace."""
    return ws[:B * blk * blk * 8].view(torch.int64).view(B, blk, blk)


def _graph_rows(masked, bulk_frac):
    """[B][blk] bool: masked rows of sequences on the graph path (the rows whose sums the selection reads)."""
    m = masked.bool()
    graph = m.sum(dim=1).float() >= bulk_frac * m.shape[1]
    return m & graph[:, None]


@pytest.mark.parametrize("name,folds", [("tiny", False), ("llada_step", True), ("batched", False)])
def test_row_stats_attention_matches_oracle(dlm, name, folds):
    """dlm_row_stats_attention (the DAPD attention sums computed by the row
    pass's CTAs where the rows are few, else the two passes in turn) on the
    screened workloads: the statistics equal the plain row pass bit for bit,
    the exact sums of every row the selection reads equal the separate
    attention pass's, and the DAPD selection equals the oracle's."""
    w, dw, o = workload(name)
    cfg = w.cfg
    B, blk = cfg.batch, cfg.blk
    assert dlm.row_stats_attention_folds(dw.cur, dw.attn, B, blk) == folds
    kw = dict(tau_edge=cfg.tau_edge, bulk_conf=cfg.bulk_conf, bulk_frac=cfg.bulk_frac)
    status = dlm.new_status()
    st, ws = dlm.row_stats_attention(dw.cur, dw.prev, dw.attn, dw.masked, block_start=dw.block_start, status=status,
                                     **kw)
    ref = dlm.row_stats(dw.cur, dw.prev)
    ws_ref = dlm.dapd_graph(dw.attn, dw.masked, block_start=dw.block_start, **kw)
    sel, n = dlm.dapd_select(ws, dw.masked, st.conf.view(B, blk), **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in ("argmax", "conf", "lse", "entropy", "kl", "lse_prev"):
        assert torch.equal(getattr(st, k), getattr(ref, k)), k
    rows = _graph_rows(dw.masked, cfg.bulk_frac)
    assert torch.equal(_sums(ws, B, blk)[rows], _sums(ws_ref, B, blk)[rows])
    w1 = dataclasses.replace(w, cfg=synth.scaled(cfg, rules=("dapd",)))
    assert check_rules_exact(name, w1, o, {"dapd": sel.cpu().numpy()}, None) == B


@pytest.mark.parametrize("attn_dt,blk,B,L,H,vocab,prev,folds", [
    (torch.float16, 32, 3, 4, 6, 16384, True, True),     # few rows: split over clusters of 4
    (torch.float16, 32, 2, 3, 4, 16384, True, "odd"),    # a mask not 4-byte aligned: read from global
    (torch.bfloat16, 8, 4, 3, 5, 32768, True, True),     # clusters of 8, one vector per block row
    (torch.float32, 8, 9, 3, 2, 8195, False, True),      # ragged vocabulary, no previous step
    (torch.float16, 64, 2, 2, 2, 8192, True, True),      # blocks of 64
    (torch.bfloat16, 16, 40, 2, 3, 8192, True, False),   # 640 rows: the two passes in turn
    (torch.bfloat16, 8, 1, 1, 1, 512, True, False),      # one short row per position
])
def test_row_stats_attention_shapes(dlm, attn_dt, blk, B, L, H, vocab, prev, folds):
    """Random shapes, masks with late-phase sequences and unmasked rows: the
    folded call against the separate row and attention passes (statistics and
    the sums of the rows the selection reads bit for bit, selections equal)."""
    g = torch.Generator(device="cuda").manual_seed(blk * 1000 + B)
    bs = 8
    N = (bs + blk + 5 + 7) // 8 * 8                  # rows of 16-byte multiples
    ld = (vocab + 7) // 8 * 8                        # logit rows padded to 16 bytes
    cur = torch.randn(B * blk, ld, device="cuda", generator=g).mul_(3).to(torch.bfloat16)[:, :vocab]
    prv = torch.randn(B * blk, ld, device="cuda", generator=g).mul_(3).to(torch.bfloat16)[:, :vocab] if prev else None
    attn = torch.rand(B, L, H, N, N, device="cuda", generator=g).to(attn_dt)
    masked = (torch.rand(B, blk, device="cuda", generator=g) < 0.7).to(torch.uint8)
    if folds == "odd":
        folds = True
        buf = torch.zeros(B * blk + 1, dtype=torch.uint8, device="cuda")
        buf[1:] = masked.view(-1)
        masked = buf[1:].view(B, blk)
        assert masked.data_ptr() % 4 != 0
    masked[0, :] = 1                                  # one sequence fully masked
    if B > 2:
        masked[1, :] = 0
        masked[1, : max(1, blk // 4)] = 1             # one late-phase sequence
    kw = dict(tau_edge=0.3, bulk_conf=0.9, bulk_frac=0.5)
    assert dlm.row_stats_attention_folds(cur, attn, B, blk) == folds
    status = dlm.new_status()
    st, ws = dlm.row_stats_attention(cur, prv, attn, masked, block_start=bs, status=status, **kw)
    ref = dlm.row_stats(cur, prv)
    ws_ref = dlm.dapd_graph(attn, masked, block_start=bs, **kw)
    sel, n = dlm.dapd_select(ws, masked, st.conf.view(B, blk), **kw)
    sel_ref, n_ref = dlm.dapd_select(ws_ref, masked, ref.conf.view(B, blk), **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in ("argmax", "conf", "lse", "entropy", "kl", "lse_prev"):
        a, b = getattr(st, k), getattr(ref, k)
        assert (a is None and b is None) or torch.equal(a, b), k
    rows = _graph_rows(masked, 0.5)
    assert torch.equal(_sums(ws, B, blk)[rows], _sums(ws_ref, B, blk)[rows])
    assert torch.equal(sel, sel_ref) and torch.equal(n, n_ref)


def test_row_stats_attention_unfolded_falls_back(dlm):
    """Blocks whose rows are not whole 16-byte vectors are not folded: the call
    runs the row pass and the attention pass one after the other, with the
    same results as the two calls."""
    g = torch.Generator(device="cuda").manual_seed(5)
    B, blk, L, H, vocab, bs = 4, 30, 2, 3, 2048, 8
    cur = torch.randn(B * blk, vocab, device="cuda", generator=g).to(torch.bfloat16)
    attn = torch.rand(B, L, H, bs + blk + 2, bs + blk + 2, device="cuda", generator=g).to(torch.float16)
    masked = torch.ones(B, blk, dtype=torch.uint8, device="cuda")
    assert not dlm.row_stats_attention_folds(cur, attn, B, blk)
    st, ws = dlm.row_stats_attention(cur, cur, attn, masked, block_start=bs, tau_edge=0.3)
    ref = dlm.row_stats(cur, cur)
    ws_ref = dlm.dapd_graph(attn, masked, block_start=bs, tau_edge=0.3)
    torch.cuda.synchronize()
    assert torch.equal(st.conf, ref.conf) and torch.equal(st.argmax, ref.argmax)
    assert torch.equal(_sums(ws, B, blk), _sums(ws_ref, B, blk))


@pytest.mark.parametrize("trial", range(10))
def test_dapd_warp_selection_random(dlm, trial):
    """Blocks of up to 32 without float outputs take the one-warp selection
    kernel; with them, the one-CTA kernel.  Random blocks, masks (graph path
    and late phase), confidences with exact 1.0s and ties, both key orders and
    the pre-unmask flag: the two kernels and the oracle select the same
    positions."""
    rng = np.random.default_rng(2300 + trial)
    blk = int(rng.integers(1, 33))
    B = int(rng.integers(1, 10))
    L, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    sub = (rng.random((B, L, H, blk, blk)) ** 4 * 0.4).astype(np.float32)
    sub16 = synth.to_f16_bits(sub)
    masked = (rng.random((B, blk)) < rng.uniform(0.2, 1.0)).astype(np.uint8)
    masked[0, :] = 1
    conf = rng.choice(np.array([0.25, 0.5, 0.75, 0.95, 1.0], np.float32), (B, blk))
    conf = np.where(rng.random((B, blk)) < 0.5, rng.random((B, blk)).astype(np.float32), conf).astype(np.float32)
    om = trial % 2
    flag = (trial // 2) % 2 == 1
    N = (blk + 7) // 8 * 8                      # rows of 16-byte multiples, the block at the origin
    attn = torch.zeros((B, L, H, N, N), dtype=torch.float16, device="cuda")
    attn[:, :, :, :blk, :blk] = to_torch(sub16, synth.F16, "cuda")
    tau = float(rng.choice([0.01, 0.05, 0.2]))
    gs, gn = dlm.dapd_graph_mis(attn, cuda(masked), cuda(conf), tau, 0.9, 0.5, om, 0, preunmask_certain=flag)
    deg = torch.empty(B, blk, dtype=torch.int32, device="cuda")
    gs2, gn2 = dlm.dapd_graph_mis(attn, cuda(masked), cuda(conf), tau, 0.9, 0.5, om, 0, deg_out=deg,
                                  preunmask_certain=flag)
    r = oracle.dapd(sub16, masked, conf.astype(np.float64), tau, 0.9, 0.5, om, dtype=synth.F16,
                    preunmask_certain=flag)
    np.testing.assert_array_equal(gs.cpu().numpy(), r["selected"])
    np.testing.assert_array_equal(gn.cpu().numpy(), r["n_selected"])
    np.testing.assert_array_equal(gs2.cpu().numpy(), r["selected"])
    np.testing.assert_array_equal(gn2.cpu().numpy(), r["n_selected"])
