"""Reference oracle for the per-step unmask decision -- TEST INFRASTRUCTURE ONLY.

Plain fp64 C (``dlm_oracle.c``) behind ctypes, with numpy arrays in and out.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the library under
``diffusion_decoding_token_gb300`` never does and shares no code with it.

Every function states the page and section it restates; see the C source for
the definitions written out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dlm_oracle.c")
_LIB = os.path.join(_HERE, "libdlm_oracle.so")

F32, BF16, F16 = 0, 1, 2
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_F = ctypes.c_float


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, OpenMP) next to its source."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_row_stats.argtypes = [_P, _P, _I32, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P]
            lib.oracle_select_threshold.argtypes = [_P, _P, _I32, _I32, _F, _P, _P]
            lib.oracle_depcap_boundary.argtypes = [_P, _P, _I32, _I32, _P, _P, _F, _I32, _I32, _I32, _P, _P]
            lib.oracle_cap_select.argtypes = [_P, _I32, _I64, _P, _P, _P, _P, _P, _P, _I32, _I32,
                                              _F, _F, _F, _I32, _I32, _P, _P, _P, _P, _P]
            lib.oracle_revocable_step.argtypes = [_P, _P, _P, _P, _I32, _I32, _I32, _F, _F, _I32, _F, _F, _F,
                                                  _F, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
            lib.oracle_cap_select.restype = _I32
            lib.oracle_dapd.argtypes = [_P, _I32, _I32, _I32, _I32, _I64, _I64, _I64, _I64, _I32, _I32,
                                        _P, _P, _F, _F, _F, _I32, _I32, _P, _P, _P, _P, _P, _P]
            lib.oracle_greedy_mis.argtypes = [_I32, _P, _P, _P]
            lib.oracle_attention_influence.argtypes = [_P, _I32, _I32, _I32, _I32, _I64, _I64, _I64, _I64, _I32,
                                                       _I32, _P, _P]
            lib.oracle_select_topk.argtypes = [_P, _P, _I32, _I32, _I32, _P, _P]
            lib.oracle_select_factor.argtypes = [_P, _P, _I32, _I32, _F, _P, _P]
            lib.oracle_parallel_certificate.argtypes = [_P, _P, _I32, _I32, _P]
            lib.oracle_set_threads.argtypes = [_I32]
            lib.oracle_get_threads.restype = _I32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(arr: np.ndarray, dtype: int | None) -> int:
    if dtype is not None:
        return dtype
    if arr.dtype == np.float32:
        return F32
    raise ValueError("16-bit storage needs an explicit dtype code (BF16 or F16)")


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def row_stats(cur, prev=None, dtype=None, row_index=None, n_out=None):
    """Per-row argmax, confidence, log-sum-exp, entropy, KL(cur||prev), prev LSE.

    DepCap, Methodology (I_k = KL(p_curr || p_prev), H_k = H(p_curr),
    c_i = max_v p_i(v)); Fast-dLLM review, Method (max-softmax confidence).
    ``cur``/``prev`` are [rows, stride] arrays (float32, or uint16 bit patterns
    of bf16/f16 with ``dtype``); the vocab is the full width unless the caller
    slices.  Returns a dict of fp64 arrays (argmax int32).
    """
    lib = _load()
    cur = np.ascontiguousarray(cur)
    code = _dtype_code(cur, dtype)
    rows, V = cur.shape
    if prev is not None:
        prev = np.ascontiguousarray(prev)
        assert prev.shape == cur.shape and prev.dtype == cur.dtype
    n = rows if n_out is None else n_out
    out = {
        "argmax": np.full(n, -1, np.int32),
        "conf": np.full(n, np.nan),
        "lse": np.full(n, np.nan),
        "entropy": np.full(n, np.nan),
    }
    if prev is not None:
        out["kl"] = np.full(n, np.nan)
        out["lse_prev"] = np.full(n, np.nan)
    ri = None
    n_rows = rows
    if row_index is not None:
        ri = np.ascontiguousarray(row_index, dtype=np.int32)
        n_rows = len(ri)
    lib.oracle_row_stats(_ptr(cur), _ptr(prev), code, n_rows, V, V, _ptr(ri),
                         _ptr(out["argmax"]), _ptr(out["conf"]), _ptr(out["lse"]),
                         _ptr(out["entropy"]), _ptr(out.get("kl")), _ptr(out.get("lse_prev")))
    return out


def select_threshold(conf, masked, tau):
    """Fast-dLLM threshold rule with top-confidence fallback (Fast-dLLM review, Method)."""
    lib = _load()
    conf = np.ascontiguousarray(conf, dtype=np.float64)
    masked = np.ascontiguousarray(masked, dtype=np.uint8)
    B, blk = masked.shape
    sel = np.zeros((B, blk), np.uint8)
    n = np.zeros(B, np.int32)
    lib.oracle_select_threshold(_ptr(conf), _ptr(masked), B, blk, float(tau), _ptr(sel), _ptr(n))
    return sel, n


def depcap_boundary(kl, entropy, lam, L_min, smooth_w=1, norm_mode=0, cold_start=None, window_len=None):
    """DepGA-Block boundary (DepCap, Methodology).  Returns (block_len, score).

    ``window_len`` (optional, [B]): sequence b uses the first window_len[b]
    entries of its row, L_window = min(L_max, L_remain) per sequence; score
    entries past it stay NaN."""
    lib = _load()
    kl = np.ascontiguousarray(kl, dtype=np.float64)
    entropy = np.ascontiguousarray(entropy, dtype=np.float64)
    B, Lw = kl.shape
    cs = None if cold_start is None else np.ascontiguousarray(cold_start, dtype=np.uint8)
    wl = None if window_len is None else np.ascontiguousarray(window_len, dtype=np.int32)
    blen = np.zeros(B, np.int32)
    score = np.full((B, Lw), np.nan)
    lib.oracle_depcap_boundary(_ptr(kl), _ptr(entropy), B, Lw, _ptr(wl), _ptr(cs), float(lam), int(L_min),
                               int(smooth_w), int(norm_mode), _ptr(blen), _ptr(score))
    return blen, score


def cap_select(logits, argmax, conf, lse, masked, tau_low, tau_high, gamma, p_max,
               high_tier_unconditional=False, scope_len=None, dtype=None, row_index=None):
    """CAP-Decoding (DepCap, Methodology).  ``logits`` is [rows, V]; position
    i of sequence b reads row ``row_index[b*blk + i]`` (default b*blk + i).

    Returns dict(selected, n_selected, D, pool, pool_n, clipped)."""
    lib = _load()
    logits = np.ascontiguousarray(logits)
    code = _dtype_code(logits, dtype)
    masked = np.ascontiguousarray(masked, dtype=np.uint8)
    B, blk = masked.shape
    argmax = np.ascontiguousarray(argmax, dtype=np.int32).reshape(B * blk)
    conf = np.ascontiguousarray(conf, dtype=np.float64).reshape(B * blk)
    lse = np.ascontiguousarray(lse, dtype=np.float64).reshape(B * blk)
    sl = None if scope_len is None else np.ascontiguousarray(scope_len, dtype=np.int32)
    ri = None
    if row_index is not None:
        ri = np.ascontiguousarray(row_index, dtype=np.int32).reshape(B * blk)
        assert ri.min() >= 0 and ri.max() < logits.shape[0]
    else:
        assert logits.shape[0] >= B * blk
    sel = np.zeros((B, blk), np.uint8)
    n = np.zeros(B, np.int32)
    D = np.zeros((B, blk, blk))
    pool = np.zeros((B, blk), np.int32)
    pool_n = np.zeros(B, np.int32)
    clipped = lib.oracle_cap_select(_ptr(logits), code, logits.shape[1], _ptr(ri), _ptr(argmax), _ptr(conf),
                                    _ptr(lse), _ptr(masked), _ptr(sl), B, blk, float(tau_low),
                                    float(tau_high), float(gamma), int(p_max),
                                    int(bool(high_tier_unconditional)), _ptr(sel), _ptr(n), _ptr(D),
                                    _ptr(pool), _ptr(pool_n))
    return dict(selected=sel, n_selected=n, D=D, pool=pool, pool_n=pool_n, clipped=bool(clipped))


def dapd(attn, masked, conf, tau_edge, bulk_conf=0.9, bulk_frac=0.5, order_mode=0,
         block_start=0, dtype=None, preunmask_certain=False):
    """DAPD step (DAPD, 整体框架, 关键设计 1-3).

    ``attn`` is [B, L, H, N, N] (or the compact block [B, L, H, blk, blk] with
    block_start 0), float32 or f16/bf16 bit patterns with ``dtype``.
    Returns dict(selected, n_selected, s, dtilde, deg, path).
    """
    lib = _load()
    attn = np.ascontiguousarray(attn)
    code = _dtype_code(attn, dtype)
    B, L, H, N, N2 = attn.shape
    assert N == N2
    masked = np.ascontiguousarray(masked, dtype=np.uint8)
    blk = masked.shape[1]
    conf = np.ascontiguousarray(conf, dtype=np.float64).reshape(B * blk)
    sel = np.zeros((B, blk), np.uint8)
    n = np.zeros(B, np.int32)
    s = np.zeros((B, blk, blk))
    dt = np.zeros((B, blk))
    deg = np.zeros((B, blk), np.int32)
    path = np.zeros(B, np.int32)
    sr, sh, sl, sb = N, N * N, H * N * N, L * H * N * N
    lib.oracle_dapd(_ptr(attn), code, B, L, H, sb, sl, sh, sr, int(block_start), blk, _ptr(masked),
                    _ptr(conf), float(tau_edge), float(bulk_conf), float(bulk_frac), int(order_mode),
                    int(bool(preunmask_certain)), _ptr(sel), _ptr(n), _ptr(s), _ptr(dt), _ptr(deg), _ptr(path))
    return dict(selected=sel, n_selected=n, s=s, dtilde=dt, deg=deg, path=path)


def attention_influence(attn, masked, block_start=0, dtype=None):
    """Downstream influence of every block position: the attention it
    receives from the masked queries, averaged over layers and heads (COVER
    page, Method; the reading is stated in the C source).  ``attn`` is
    [B, L, H, N, N] (or the compact block with block_start 0).  Returns
    [B, blk] fp64."""
    lib = _load()
    attn = np.ascontiguousarray(attn)
    code = _dtype_code(attn, dtype)
    B, L, H, N, N2 = attn.shape
    assert N == N2
    masked = np.ascontiguousarray(masked, dtype=np.uint8)
    blk = masked.shape[1]
    assert block_start + blk <= N
    out = np.zeros((B, blk))
    lib.oracle_attention_influence(_ptr(attn), code, B, L, H, L * H * N * N, H * N * N, N * N, N, int(block_start),
                                   blk, _ptr(masked), _ptr(out))
    return out


def greedy_mis(adj, order):
    """Greedy maximal independent set over an explicit node order."""
    lib = _load()
    adj = np.ascontiguousarray(adj, dtype=np.uint8)
    order = np.ascontiguousarray(order, dtype=np.int32)
    n = adj.shape[0]
    kept = np.zeros(n, np.uint8)
    lib.oracle_greedy_mis(n, _ptr(adj), _ptr(order), _ptr(kept))
    return kept


def select_topk(conf, masked, k):
    """Fixed top-K per step (Fast-dLLM review, Prior limitations)."""
    lib = _load()
    conf = np.ascontiguousarray(conf, dtype=np.float64)
    masked = np.ascontiguousarray(masked, dtype=np.uint8)
    B, blk = masked.shape
    sel = np.zeros((B, blk), np.uint8)
    n = np.zeros(B, np.int32)
    lib.oracle_select_topk(_ptr(conf), _ptr(masked), B, blk, int(k), _ptr(sel), _ptr(n))
    return sel, n


def select_factor(conf, masked, f):
    """Fast-dLLM factor decoding (Fast-dLLM review, Method, appendix variant)."""
    lib = _load()
    conf = np.ascontiguousarray(conf, dtype=np.float64)
    masked = np.ascontiguousarray(masked, dtype=np.uint8)
    B, blk = masked.shape
    sel = np.zeros((B, blk), np.uint8)
    n = np.zeros(B, np.int32)
    lib.oracle_select_factor(_ptr(conf), _ptr(masked), B, blk, float(f), _ptr(sel), _ptr(n))
    return sel, n


def parallel_certificate(conf, selected):
    """Theorem-1 certificate of a selection (Fast-dLLM review, Key idea)."""
    lib = _load()
    conf = np.ascontiguousarray(conf, dtype=np.float64)
    selected = np.ascontiguousarray(selected, dtype=np.uint8)
    B, blk = selected.shape
    out = np.zeros(B, np.uint8)
    lib.oracle_parallel_certificate(_ptr(conf), _ptr(selected), B, blk, _ptr(out))
    return out


def revocable_init(B, blk):
    """Initial state of a revocable decode: everything masked, no seeds."""
    return dict(tok=np.full((B, blk), -1, np.int32), masked=np.ones((B, blk), np.uint8),
                seed=np.zeros((B, blk), np.uint8), last_seed=np.full((B, blk), -(2 ** 30), np.int32),
                remasks=np.zeros((B, blk), np.int32), last_tok=np.full((B, blk), -1, np.int32),
                flipflops=np.zeros(B, np.int32))


def revocable_step(argmax, conf, state, step, tau_replace=0.9, tau_draft=0.9, draft_budget=0, w_unc=1.0,
                   w_infl=1.0, w_drift=1.0, pi=1.0, cooldown=1, remask_budget=2, influence=None, drift=None):
    """One state update of revocable parallel decoding (COVER page,
    Revocable Parallel Diffusion Decoding and Method).  ``state`` (a dict of
    numpy arrays as revocable_init makes) is updated in place; returns dict
    (outcome, n_drafted, n_revoked)."""
    lib = _load()
    argmax = np.ascontiguousarray(argmax, dtype=np.int32)
    B, blk = argmax.shape
    conf = np.ascontiguousarray(conf, dtype=np.float64).reshape(B, blk)
    infl = None if influence is None else np.ascontiguousarray(influence, dtype=np.float64).reshape(B, blk)
    dr = None if drift is None else np.ascontiguousarray(drift, dtype=np.float64).reshape(B, blk)
    for k, dt in (("tok", np.int32), ("masked", np.uint8), ("seed", np.uint8), ("last_seed", np.int32),
                  ("remasks", np.int32), ("last_tok", np.int32), ("flipflops", np.int32)):
        assert state[k].dtype == dt and state[k].flags.c_contiguous, k
    outcome = np.zeros((B, blk), np.uint8)
    nd = np.zeros(B, np.int32)
    nr = np.zeros(B, np.int32)
    lib.oracle_revocable_step(_ptr(argmax), _ptr(conf), _ptr(infl), _ptr(dr), B, blk, int(step),
                              float(tau_replace), float(tau_draft), int(draft_budget), float(w_unc), float(w_infl),
                              float(w_drift), float(pi), int(cooldown), int(remask_budget), _ptr(state["tok"]),
                              _ptr(state["masked"]), _ptr(state["seed"]), _ptr(state["last_seed"]),
                              _ptr(state["remasks"]), _ptr(state["last_tok"]), _ptr(outcome), _ptr(nd), _ptr(nr),
                              _ptr(state["flipflops"]))
    return dict(outcome=outcome, n_drafted=nd, n_revoked=nr)
