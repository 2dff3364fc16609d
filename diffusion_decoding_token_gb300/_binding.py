"""ctypes binding of libdlm.so (argument marshalling only).

Every function takes CUDA tensors, checks their dtype/shape/device, passes raw
pointers and the current CUDA stream to the C ABI declared in
``include/dlm.h``, and raises on a non-OK status.  Nothing here computes a
decision; there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdlm.so")

DLM_F32, DLM_BF16, DLM_F16 = 0, 1, 2
DEV_NONFINITE, DEV_POOL_CLIPPED, DEV_TIMEOUT, DEV_BAD_INDEX = 1, 2, 4, 8
MAX_BLK = 256

_DT = {torch.float32: DLM_F32, torch.bfloat16: DLM_BF16, torch.float16: DLM_F16}

_lib = None


class DepcapParams(ctypes.Structure):
    _fields_ = [("lambda_", ctypes.c_float), ("L_min", ctypes.c_int32),
                ("smooth_w", ctypes.c_int32), ("norm_mode", ctypes.c_int32)]


class CapParams(ctypes.Structure):
    _fields_ = [("tau_low", ctypes.c_float), ("tau_high", ctypes.c_float), ("gamma", ctypes.c_float),
                ("p_max", ctypes.c_int32), ("high_tier_unconditional", ctypes.c_int32)]


class DapdParams(ctypes.Structure):
    _fields_ = [("tau_edge", ctypes.c_float), ("bulk_conf", ctypes.c_float),
                ("bulk_frac", ctypes.c_float), ("order_mode", ctypes.c_int32),
                ("preunmask_certain", ctypes.c_int32)]


class StepRules(ctypes.Structure):
    _fields_ = [("rules", ctypes.c_uint32), ("tau", ctypes.c_float), ("depcap", DepcapParams),
                ("cold_start", ctypes.c_void_p), ("cap", CapParams), ("cap_scope_from_boundary", ctypes.c_int32)]


RULE_THRESHOLD, RULE_BOUNDARY, RULE_CAP = 1, 2, 4


class RevocableParams(ctypes.Structure):
    _fields_ = [("tau_replace", ctypes.c_float), ("tau_draft", ctypes.c_float), ("draft_budget", ctypes.c_int32),
                ("w_unc", ctypes.c_float), ("w_infl", ctypes.c_float), ("w_drift", ctypes.c_float),
                ("pi", ctypes.c_float), ("cooldown", ctypes.c_int32), ("remask_budget", ctypes.c_int32)]


class DlmError(RuntimeError):
    pass


def lib():
    """Load libdlm.so; raise if it has not been built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, F, Z = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        L.dlm_status_string.restype = ctypes.c_char_p
        L.dlm_status_string.argtypes = [ctypes.c_int]
        L.dlm_version.restype = ctypes.c_int
        L.dlm_row_stats.argtypes = [P, P, ctypes.c_int, I64, I64, I64, P, P, P, P, P, P, P, P, P]
        L.dlm_select_threshold.argtypes = [P, P, I32, I32, F, P, P, P]
        L.dlm_depcap_boundary.argtypes = [P, P, I32, I32, P, ctypes.POINTER(DepcapParams), P, P, P]
        L.dlm_cap_workspace_size.restype = Z
        L.dlm_cap_workspace_size.argtypes = [I32, I32]
        L.dlm_cap_select.argtypes = [P, ctypes.c_int, I64, I64, P, I64, P, P, P, P, P, I32, I32,
                                     ctypes.POINTER(CapParams), P, P, P, P, Z, P, P]
        L.dlm_dapd_workspace_size.restype = Z
        L.dlm_dapd_workspace_size.argtypes = [I32, I32]
        L.dlm_dapd_graph_mis.argtypes = [P, ctypes.c_int, I32, I32, I32, I64, I64, I64, I64, I32, I32,
                                         P, P, ctypes.POINTER(DapdParams), P, P, P, P, P, P, Z, P, P]
        L.dlm_depcap_boundary_ragged.argtypes = [P, P, I32, I32, P, P, ctypes.POINTER(DepcapParams), P, P, P]
        L.dlm_row_stats_partial.argtypes = [P, P, ctypes.c_int, I64, I64, I64, P, I64, P, P]
        L.dlm_row_stats_launches.argtypes = [ctypes.c_int, I32, I64, I64, ctypes.c_uint32]
        L.dlm_row_stats_ex.argtypes = [P, P, ctypes.c_int, I64, I64, I64, P, I64, P, P, P, P, P, P, P,
                                       ctypes.c_uint32, P]
        L.dlm_row_stats_launches.restype = I32
        L.dlm_row_stats_merge.argtypes = [P, I32, I64, I64, P, I32, P, P, P, P, P, P, P, P]
        L.dlm_select_topk.argtypes = [P, P, I32, I32, I32, P, P, P]
        L.dlm_revocable_step.argtypes = [P, P, P, P, I32, I32, I32, ctypes.POINTER(RevocableParams), P, P, P, P, P,
                                         P, P, P, P, P, P]
        L.dlm_select_factor.argtypes = [P, P, I32, I32, F, P, P, P]
        L.dlm_parallel_certificate.argtypes = [P, P, I32, I32, P, P]
        L.dlm_dapd_graph.argtypes = [P, ctypes.c_int, I32, I32, I32, I64, I64, I64, I64, I32, I32,
                                     P, ctypes.POINTER(DapdParams), P, P, P, P, Z, P, P]
        L.dlm_dapd_select.argtypes = [P, P, I32, I32, ctypes.POINTER(DapdParams), P, P, P, Z, P]
        L.dlm_row_stats_rules_workspace_size.restype = Z
        L.dlm_row_stats_rules_workspace_size.argtypes = [I32]
        L.dlm_row_stats_rules.argtypes = [P, P, ctypes.c_int, I32, I32, I64, I64, P, ctypes.POINTER(StepRules), P, P, P,
                                          P, P, P, P, P, P, P, P, P, P, Z, P, P]
        L.dlm_attention_influence.argtypes = [P, ctypes.c_int, I32, I32, I32, I64, I64, I64, I64, I32, I32, P, P, P,
                                              Z, P, P]
        L.dlm_row_stats_attention_folds.restype = I32
        L.dlm_row_stats_attention_folds.argtypes = [ctypes.c_int, I32, I32, I64, ctypes.c_int, I32, I32]
        L.dlm_row_stats_attention.argtypes = [P, P, ctypes.c_int, I32, I32, I64, I64, P, P, P, P, P, P, P,
                                              ctypes.c_int, I32, I32, I64, I64, I64, I64, I32, P,
                                              ctypes.POINTER(DapdParams), P, Z, P, P]
        for f in ("dlm_row_stats", "dlm_select_threshold", "dlm_depcap_boundary", "dlm_cap_select",
                  "dlm_dapd_graph_mis", "dlm_dapd_graph", "dlm_dapd_select", "dlm_select_topk",
                  "dlm_select_factor", "dlm_parallel_certificate", "dlm_depcap_boundary_ragged",
                  "dlm_revocable_step", "dlm_attention_influence", "dlm_row_stats_rules",
                  "dlm_row_stats_attention"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise DlmError(f"libdlm: {lib().dlm_status_string(status).decode()} (status {status})")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libdlm takes CUDA tensors only")


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _u8(m: torch.Tensor) -> torch.Tensor:
    m = m if m.dtype == torch.uint8 else m.to(torch.uint8)
    return m.contiguous()


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word (uint32 semantics in an int32 tensor)."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


class RowStats(NamedTuple):
    argmax: torch.Tensor
    conf: torch.Tensor
    lse: torch.Tensor
    entropy: torch.Tensor
    kl: torch.Tensor | None
    lse_prev: torch.Tensor | None


def alloc_row_stats(n: int, device, with_prev: bool = True) -> RowStats:
    f = dict(dtype=torch.float32, device=device)
    return RowStats(torch.empty(n, dtype=torch.int32, device=device), torch.empty(n, **f),
                    torch.empty(n, **f), torch.empty(n, **f),
                    torch.empty(n, **f) if with_prev else None, torch.empty(n, **f) if with_prev else None)


ROWS_SINGLE_GRID = 1  # DLM_ROWS_SINGLE_GRID
ROWS_GATHER = 2       # DLM_ROWS_GATHER


def row_stats(cur: torch.Tensor, prev: torch.Tensor | None = None, *, row_index: torch.Tensor | None = None,
              out: RowStats | None = None, status: torch.Tensor | None = None, single_grid: bool = False,
              gather: bool = False) -> RowStats:
    """dlm_row_stats_ex over the rows of ``cur`` ([rows, V] with unit column
    stride), every row index checked against the rows of ``cur``;
    ``single_grid`` passes DLM_ROWS_SINGLE_GRID, ``gather`` DLM_ROWS_GATHER
    (results of row_index[r] stored at r)."""
    _need_cuda(cur, prev, row_index)
    if cur.dim() != 2 or cur.stride(1) != 1:
        raise ValueError("cur must be [rows, V] with contiguous rows")
    if prev is not None and (prev.shape != cur.shape or prev.stride() != cur.stride() or prev.dtype != cur.dtype):
        raise ValueError("prev must match cur in shape, strides and dtype")
    rows, V = cur.shape
    n = rows
    if row_index is not None:
        row_index = row_index.to(torch.int32).contiguous()
        n = row_index.numel()
    elif gather:
        raise ValueError("gather needs a row_index")
    if out is None:
        out = alloc_row_stats(n if gather else rows, cur.device, prev is not None)
    flags = (ROWS_SINGLE_GRID if single_grid else 0) | (ROWS_GATHER if gather else 0)
    _check(lib().dlm_row_stats_ex(_p(cur), _p(prev), _dt(cur), n, V, cur.stride(0), _p(row_index), rows,
                                  _p(out.argmax), _p(out.conf), _p(out.lse), _p(out.entropy),
                                  _p(out.kl) if prev is not None else None,
                                  _p(out.lse_prev) if prev is not None else None, _p(status),
                                  flags, _stream(cur.device)))
    return out


PARTIAL_FLOATS = 8  # dlm_row_partial: 8 four-byte fields


def row_stats_partial(cur: torch.Tensor, prev: torch.Tensor | None = None, *, vocab_offset: int = 0,
                      row_index: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """dlm_row_stats_partial over a vocabulary slice ``cur`` ([rows, V_slice],
    unit column stride; the slice starts at global position ``vocab_offset``).
    Returns the 32-byte states as a float32 [rows, 8] tensor (opaque)."""
    _need_cuda(cur, prev, row_index)
    if cur.dim() != 2 or cur.stride(1) != 1:
        raise ValueError("cur must be [rows, V] with contiguous rows")
    if prev is not None and (prev.shape != cur.shape or prev.stride() != cur.stride() or prev.dtype != cur.dtype):
        raise ValueError("prev must match cur in shape, strides and dtype")
    rows, V = cur.shape
    if out is None:
        out = torch.empty((rows, PARTIAL_FLOATS), dtype=torch.float32, device=cur.device)
    n = rows
    if row_index is not None:
        row_index = row_index.to(torch.int32).contiguous()
        n = row_index.numel()
    _check(lib().dlm_row_stats_partial(_p(cur), _p(prev), _dt(cur), n, V, cur.stride(0), _p(row_index),
                                       int(vocab_offset), _p(out), _stream(cur.device)))
    return out


def row_stats_merge(partials: torch.Tensor, has_prev: bool, *, row_index: torch.Tensor | None = None,
                    out: RowStats | None = None, status: torch.Tensor | None = None) -> RowStats:
    """dlm_row_stats_merge of [n_shards, rows, 8] partial states (slices in
    vocabulary order) into the whole rows' statistics."""
    _need_cuda(partials, row_index)
    if partials.dim() != 3 or partials.shape[2] != PARTIAL_FLOATS or not partials.is_contiguous():
        raise ValueError("partials must be a contiguous [n_shards, rows, 8] tensor")
    n_shards, rows, _ = partials.shape
    if out is None:
        out = alloc_row_stats(rows, partials.device, has_prev)
    n = rows
    if row_index is not None:
        row_index = row_index.to(torch.int32).contiguous()
        n = row_index.numel()
    _check(lib().dlm_row_stats_merge(_p(partials), n_shards, rows, n, _p(row_index), int(bool(has_prev)),
                                     _p(out.argmax), _p(out.conf), _p(out.lse), _p(out.entropy),
                                     _p(out.kl) if has_prev else None, _p(out.lse_prev) if has_prev else None,
                                     _p(status), _stream(partials.device)))
    return out


def allgather_row_partials(partial: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange of a vocabulary-sharded row pass: every rank's [rows, 8]
    partial states gathered into [world, rows, 8] in rank order (rank r holds
    vocabulary slice r), ready for :func:`row_stats_merge`."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(partial.shape), dtype=partial.dtype, device=partial.device)
    dist.all_gather(list(out.unbind(0)), partial.contiguous(), group=group)
    return out


def select_threshold(conf: torch.Tensor, masked: torch.Tensor, tau: float = 0.9, *, selected=None,
                     n_selected=None):
    """dlm_select_threshold: conf/masked are [B, blk]; returns (selected u8, n_selected i32)."""
    _need_cuda(conf, masked)
    B, blk = masked.shape
    conf = conf.reshape(B, blk).contiguous()
    masked = _u8(masked)
    if selected is None:
        selected = torch.empty((B, blk), dtype=torch.uint8, device=conf.device)
    if n_selected is None:
        n_selected = torch.empty(B, dtype=torch.int32, device=conf.device)
    _check(lib().dlm_select_threshold(_p(conf), _p(masked), B, blk, float(tau), _p(selected), _p(n_selected),
                                      _stream(conf.device)))
    return selected, n_selected


def select_topk(conf: torch.Tensor, masked: torch.Tensor, k: int, *, selected=None, n_selected=None):
    """dlm_select_topk: the k most confident masked positions per sequence."""
    _need_cuda(conf, masked)
    B, blk = masked.shape
    conf = conf.reshape(B, blk).contiguous()
    masked = _u8(masked)
    if selected is None:
        selected = torch.empty((B, blk), dtype=torch.uint8, device=conf.device)
    if n_selected is None:
        n_selected = torch.empty(B, dtype=torch.int32, device=conf.device)
    _check(lib().dlm_select_topk(_p(conf), _p(masked), B, blk, int(k), _p(selected), _p(n_selected),
                                 _stream(conf.device)))
    return selected, n_selected


def select_factor(conf: torch.Tensor, masked: torch.Tensor, f: float, *, selected=None, n_selected=None):
    """dlm_select_factor: Fast-dLLM factor decoding."""
    _need_cuda(conf, masked)
    B, blk = masked.shape
    conf = conf.reshape(B, blk).contiguous()
    masked = _u8(masked)
    if selected is None:
        selected = torch.empty((B, blk), dtype=torch.uint8, device=conf.device)
    if n_selected is None:
        n_selected = torch.empty(B, dtype=torch.int32, device=conf.device)
    _check(lib().dlm_select_factor(_p(conf), _p(masked), B, blk, float(f), _p(selected), _p(n_selected),
                                   _stream(conf.device)))
    return selected, n_selected


def parallel_certificate(conf: torch.Tensor, selected: torch.Tensor, *, out=None):
    """dlm_parallel_certificate: Theorem-1 condition of each sequence's selection."""
    _need_cuda(conf, selected)
    B, blk = selected.shape
    conf = conf.reshape(B, blk).contiguous()
    selected = _u8(selected)
    if out is None:
        out = torch.empty(B, dtype=torch.uint8, device=conf.device)
    _check(lib().dlm_parallel_certificate(_p(conf), _p(selected), B, blk, _p(out), _stream(conf.device)))
    return out


def depcap_boundary(kl: torch.Tensor, entropy: torch.Tensor, lam: float = 1.0, L_min: int = 8,
                    smooth_w: int = 1, norm_mode: int = 0, cold_start: torch.Tensor | None = None, *,
                    window_len: torch.Tensor | None = None, block_len=None, score=None):
    """dlm_depcap_boundary over [B, L_window] KL / entropy; returns (block_len, score).
    With ``window_len`` ([B] int32) it calls dlm_depcap_boundary_ragged:
    sequence b uses the first window_len[b] entries of its row."""
    _need_cuda(kl, entropy, cold_start, window_len)
    B, Lw = kl.shape
    kl = kl.contiguous()
    entropy = entropy.reshape(B, Lw).contiguous()
    if cold_start is not None:
        cold_start = _u8(cold_start)
    if block_len is None:
        block_len = torch.empty(B, dtype=torch.int32, device=kl.device)
    if score is None:
        score = torch.empty((B, Lw), dtype=torch.float32, device=kl.device)
    prm = DepcapParams(float(lam), int(L_min), int(smooth_w), int(norm_mode))
    if window_len is None:
        _check(lib().dlm_depcap_boundary(_p(kl), _p(entropy), B, Lw, _p(cold_start), ctypes.byref(prm),
                                         _p(block_len), _p(score), _stream(kl.device)))
    else:
        window_len = window_len.to(torch.int32).contiguous()
        _check(lib().dlm_depcap_boundary_ragged(_p(kl), _p(entropy), B, Lw, _p(window_len), _p(cold_start),
                                                ctypes.byref(prm), _p(block_len), _p(score), _stream(kl.device)))
    return block_len, score


def revocable_state(batch: int, blk: int, device) -> dict:
    """Initial state of a revocable decode (everything masked, no seeds)."""
    i32 = dict(dtype=torch.int32, device=device)
    u8 = dict(dtype=torch.uint8, device=device)
    return dict(tok=torch.full((batch, blk), -1, **i32), masked=torch.ones((batch, blk), **u8),
                seed=torch.zeros((batch, blk), **u8), last_seed=torch.full((batch, blk), -(2 ** 30), **i32),
                remasks=torch.zeros((batch, blk), **i32), last_tok=torch.full((batch, blk), -1, **i32),
                flipflops=torch.zeros(batch, **i32))


def revocable_step(argmax: torch.Tensor, conf: torch.Tensor, state: dict, step: int, *, tau_replace=0.9,
                   tau_draft=0.9, draft_budget=0, w_unc=1.0, w_infl=1.0, w_drift=1.0, pi=1.0, cooldown=1,
                   remask_budget=2, influence=None, drift=None, outcome=None, n_drafted=None, n_revoked=None):
    """dlm_revocable_step: updates ``state`` (tensors as revocable_state makes)
    in place; returns (outcome u8 [B, blk], n_drafted, n_revoked)."""
    _need_cuda(argmax, conf, influence, drift)
    B, blk = state["masked"].shape
    dev = conf.device
    for k, dt in (("tok", torch.int32), ("masked", torch.uint8), ("seed", torch.uint8),
                  ("last_seed", torch.int32), ("remasks", torch.int32), ("last_tok", torch.int32),
                  ("flipflops", torch.int32)):
        t = state[k]
        if t.dtype != dt or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"state[{k!r}] must be a contiguous {dt} tensor on {dev}")
    if outcome is None:
        outcome = torch.empty((B, blk), dtype=torch.uint8, device=dev)
    if n_drafted is None:
        n_drafted = torch.empty(B, dtype=torch.int32, device=dev)
    if n_revoked is None:
        n_revoked = torch.empty(B, dtype=torch.int32, device=dev)
    prm = RevocableParams(float(tau_replace), float(tau_draft), int(draft_budget), float(w_unc), float(w_infl),
                          float(w_drift), float(pi), int(cooldown), int(remask_budget))
    _check(lib().dlm_revocable_step(_p(argmax.reshape(B, blk).contiguous()), _p(conf.reshape(B, blk).contiguous()),
                                    _p(None if influence is None else influence.reshape(B, blk).contiguous()),
                                    _p(None if drift is None else drift.reshape(B, blk).contiguous()), B, blk,
                                    int(step), ctypes.byref(prm), _p(state["tok"]), _p(state["masked"]),
                                    _p(state["seed"]), _p(state["last_seed"]), _p(state["remasks"]),
                                    _p(state["last_tok"]), _p(outcome), _p(n_drafted), _p(n_revoked),
                                    _p(state["flipflops"]), _stream(dev)))
    return outcome, n_drafted, n_revoked


def cap_workspace(batch: int, p_max: int, device) -> torch.Tensor:
    n = lib().dlm_cap_workspace_size(batch, p_max)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def cap_select(logits: torch.Tensor, argmax: torch.Tensor, conf: torch.Tensor, lse: torch.Tensor,
               masked: torch.Tensor, tau_low: float = 0.8, tau_high: float = 0.95, gamma: float = -16.0,
               p_max: int | None = None, high_tier_unconditional: bool = False,
               scope_len: torch.Tensor | None = None, *, D_out=None, workspace=None, status=None,
               selected=None, n_selected=None, row_index: torch.Tensor | None = None):
    """dlm_cap_select; logits are the current rows, [rows, V]: position i of
    sequence b reads row ``row_index[b*blk + i]`` (default b*blk + i).
    Returns (selected, n_selected)."""
    _need_cuda(logits, argmax, conf, lse, masked, scope_len, D_out, row_index)
    B, blk = masked.shape
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [rows, V] with contiguous rows")
    if row_index is None and logits.shape[0] < B * blk:
        raise ValueError("logits must hold B*blk rows when no row_index is given")
    if row_index is not None:
        if row_index.numel() != B * blk:
            raise ValueError("row_index must hold B*blk entries")
        row_index = row_index.to(torch.int32).contiguous()
    p_max = blk if p_max is None else int(p_max)
    masked = _u8(masked)
    dev = logits.device
    if workspace is None:
        workspace = cap_workspace(B, p_max, dev)
    if selected is None:
        selected = torch.empty((B, blk), dtype=torch.uint8, device=dev)
    if n_selected is None:
        n_selected = torch.empty(B, dtype=torch.int32, device=dev)
    if scope_len is not None:
        scope_len = scope_len.to(torch.int32).contiguous()
    prm = CapParams(float(tau_low), float(tau_high), float(gamma), p_max, int(bool(high_tier_unconditional)))
    _check(lib().dlm_cap_select(_p(logits), _dt(logits), logits.shape[1], logits.stride(0), _p(row_index),
                                logits.shape[0], _p(argmax.contiguous()), _p(conf.contiguous()),
                                _p(lse.contiguous()), _p(masked),
                                _p(scope_len), B, blk, ctypes.byref(prm), _p(selected), _p(n_selected), _p(D_out),
                                _p(workspace), workspace.numel(), _p(status), _stream(dev)))
    return selected, n_selected


def dapd_workspace(batch: int, blk: int, device) -> torch.Tensor:
    n = lib().dlm_dapd_workspace_size(batch, blk)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def dapd_graph_mis(attn: torch.Tensor, masked: torch.Tensor, conf: torch.Tensor, tau_edge: float = 0.01,
                   bulk_conf: float = 0.9, bulk_frac: float = 0.5, order_mode: int = 0, block_start: int = 0, *,
                   s_out=None, dtilde_out=None, deg_out=None, workspace=None, status=None, selected=None,
                   n_selected=None, preunmask_certain: bool = False):
    """dlm_dapd_graph_mis on ``attn`` = [B, L, H, N, N] (any element strides with unit
    column stride).  The block is rows/cols [block_start, block_start+blk)."""
    _need_cuda(attn, masked, conf, s_out, dtilde_out, deg_out)
    if attn.dim() != 5 or attn.stride(4) != 1:
        raise ValueError("attn must be [B, L, H, N, N] with unit column stride")
    B, L, H = attn.shape[:3]
    blk = masked.shape[1]
    if masked.shape[0] != B or block_start + blk > min(attn.shape[3], attn.shape[4]):
        raise ValueError("block outside the attention maps")
    masked = _u8(masked)
    dev = attn.device
    if workspace is None:
        workspace = dapd_workspace(B, blk, dev)
    if selected is None:
        selected = torch.empty((B, blk), dtype=torch.uint8, device=dev)
    if n_selected is None:
        n_selected = torch.empty(B, dtype=torch.int32, device=dev)
    sb, sl, sh, sr, _ = attn.stride()
    prm = DapdParams(float(tau_edge), float(bulk_conf), float(bulk_frac), int(order_mode), int(bool(preunmask_certain)))
    _check(lib().dlm_dapd_graph_mis(_p(attn), _dt(attn), B, L, H, sb, sl, sh, sr, int(block_start), blk,
                                    _p(masked), _p(conf.reshape(B, blk).contiguous()), ctypes.byref(prm),
                                    _p(selected), _p(n_selected), _p(s_out), _p(dtilde_out), _p(deg_out),
                                    _p(workspace), workspace.numel(), _p(status), _stream(dev)))
    return selected, n_selected


def dapd_graph(attn: torch.Tensor, masked: torch.Tensor, tau_edge: float = 0.01, bulk_conf: float = 0.9,
               bulk_frac: float = 0.5, order_mode: int = 0, block_start: int = 0, *, workspace=None, s_out=None,
               dtilde_out=None, deg_out=None, status=None):
    """dlm_dapd_graph: the attention half of DAPD (graph left in ``workspace``)."""
    _need_cuda(attn, masked, s_out, dtilde_out, deg_out)
    if attn.dim() != 5 or attn.stride(4) != 1:
        raise ValueError("attn must be [B, L, H, N, N] with unit column stride")
    B, L, H = attn.shape[:3]
    blk = masked.shape[1]
    masked = _u8(masked)
    if workspace is None:
        workspace = dapd_workspace(B, blk, attn.device)
    sb, sl, sh, sr, _ = attn.stride()
    prm = DapdParams(float(tau_edge), float(bulk_conf), float(bulk_frac), int(order_mode))
    _check(lib().dlm_dapd_graph(_p(attn), _dt(attn), B, L, H, sb, sl, sh, sr, int(block_start), blk, _p(masked),
                                ctypes.byref(prm), _p(s_out), _p(dtilde_out), _p(deg_out), _p(workspace),
                                workspace.numel(), _p(status), _stream(attn.device)))
    return workspace


def row_stats_attention_folds(cur: torch.Tensor, attn: torch.Tensor, batch: int, blk: int) -> bool:
    """Whether dlm_row_stats_attention folds the attention into the row pass
    for these shapes (rows too few to fill the GPU, attention that fits
    shared memory); otherwise it runs the two passes one after the other."""
    return bool(lib().dlm_row_stats_attention_folds(_dt(cur), int(batch), int(blk), cur.shape[1], _dt(attn),
                                                    attn.shape[1], attn.shape[2]))


def row_stats_attention(cur: torch.Tensor, prev: torch.Tensor | None, attn: torch.Tensor, masked: torch.Tensor,
                        tau_edge: float = 0.01, bulk_conf: float = 0.9, bulk_frac: float = 0.5, order_mode: int = 0,
                        block_start: int = 0, *, out: RowStats | None = None, workspace=None, status=None):
    """dlm_row_stats_attention: the row pass over ``cur`` ([B*blk, V], row
    b*blk + i = position i of sequence b) with the DAPD attention sums of
    every masked row folded in; returns (stats, workspace) -- dapd_select on
    that workspace then gives the DAPD selection."""
    _need_cuda(cur, prev, attn, masked, workspace)
    B, blk = masked.shape
    if cur.dim() != 2 or cur.stride(1) != 1 or cur.shape[0] != B * blk:
        raise ValueError("cur must be [B*blk, V] with contiguous rows")
    if prev is not None and (prev.shape != cur.shape or prev.stride() != cur.stride() or prev.dtype != cur.dtype):
        raise ValueError("prev must match cur in shape, strides and dtype")
    if attn.dim() != 5 or attn.stride(4) != 1 or attn.shape[0] != B:
        raise ValueError("attn must be [B, L, H, N, N] with unit column stride")
    masked = _u8(masked)
    st = out or alloc_row_stats(B * blk, cur.device, prev is not None)
    if workspace is None:
        workspace = dapd_workspace(B, blk, cur.device)
    sb, sl, sh, sr, _ = attn.stride()
    prm = DapdParams(float(tau_edge), float(bulk_conf), float(bulk_frac), int(order_mode))
    _check(lib().dlm_row_stats_attention(_p(cur), _p(prev), _dt(cur), B, blk, cur.shape[1], cur.stride(0),
                                         _p(st.argmax), _p(st.conf), _p(st.lse), _p(st.entropy), _p(st.kl),
                                         _p(st.lse_prev), _p(attn), _dt(attn), attn.shape[1], attn.shape[2], sb, sl,
                                         sh, sr, int(block_start), _p(masked), ctypes.byref(prm), _p(workspace),
                                         workspace.numel(), _p(status), _stream(cur.device)))
    return st, workspace


def row_stats_rules_workspace(batch: int, device) -> torch.Tensor:
    """A zeroed workspace for row_stats_rules (every call leaves it zero)."""
    return torch.zeros(max(16, lib().dlm_row_stats_rules_workspace_size(batch)), dtype=torch.uint8, device=device)


def row_stats_rules(cur: torch.Tensor, prev: torch.Tensor | None, masked: torch.Tensor, *,
                    rules=("threshold", "boundary", "cap"), tau: float = 0.9, lam: float = 1.0, L_min: int = 8,
                    smooth_w: int = 1, norm_mode: int = 0, cold_start=None, tau_low: float = 0.8,
                    tau_high: float = 0.95, gamma: float = -16.0, p_max: int | None = None,
                    high_tier_unconditional: bool = False, cap_scope_from_boundary: bool = False,
                    out: RowStats | None = None, workspace=None, status=None) -> dict:
    """dlm_row_stats_rules: the row pass over ``cur`` ([B*blk, V]) with the
    threshold, boundary and CAP rules of each sequence run by the CTA that
    finishes its last row.  Returns dict(stats, threshold, block_len, score,
    cap) with (selected, n_selected) pairs for the rules."""
    _need_cuda(cur, prev, masked, cold_start, workspace)
    B, blk = masked.shape
    if cur.dim() != 2 or cur.stride(1) != 1 or cur.shape[0] != B * blk:
        raise ValueError("cur must be [B*blk, V] with contiguous rows")
    if prev is not None and (prev.shape != cur.shape or prev.stride() != cur.stride() or prev.dtype != cur.dtype):
        raise ValueError("prev must match cur in shape, strides and dtype")
    dev = cur.device
    masked = _u8(masked)
    bits = sum(b for n, b in (("threshold", RULE_THRESHOLD), ("boundary", RULE_BOUNDARY), ("cap", RULE_CAP))
               if n in rules)
    p_max = blk if p_max is None else int(p_max)
    if out is None:
        out = alloc_row_stats(B * blk, dev, prev is not None)
    if workspace is None:
        workspace = row_stats_rules_workspace(B, dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    res = {"stats": out}
    thr = (torch.zeros((B, blk), **u8), torch.zeros(B, **i32)) if "threshold" in rules else (None, None)
    cap = (torch.zeros((B, blk), **u8), torch.zeros(B, **i32)) if "cap" in rules else (None, None)
    bl = torch.zeros(B, **i32) if "boundary" in rules else None
    sc = torch.full((B, blk), float("nan"), dtype=torch.float32, device=dev) if "boundary" in rules else None
    cold = None if cold_start is None else _u8(cold_start)
    prm = StepRules(bits, float(tau), DepcapParams(float(lam), int(L_min), int(smooth_w), int(norm_mode)),
                    None if cold is None else cold.data_ptr(),
                    CapParams(float(tau_low), float(tau_high), float(gamma), p_max, int(bool(high_tier_unconditional))),
                    int(bool(cap_scope_from_boundary)))
    _check(lib().dlm_row_stats_rules(_p(cur), _p(prev), _dt(cur), B, blk, cur.shape[1], cur.stride(0), _p(masked),
                                     ctypes.byref(prm), _p(out.argmax), _p(out.conf), _p(out.lse), _p(out.entropy),
                                     _p(out.kl) if prev is not None else None,
                                     _p(out.lse_prev) if prev is not None else None, _p(thr[0]), _p(thr[1]), _p(bl),
                                     _p(sc), _p(cap[0]), _p(cap[1]), _p(workspace), workspace.numel(), _p(status),
                                     _stream(dev)))
    res.update(threshold=thr, block_len=bl, score=sc, cap=cap, workspace=workspace)
    return res


def attention_influence(attn: torch.Tensor, masked: torch.Tensor, block_start: int = 0, *, out=None, workspace=None,
                        status=None) -> torch.Tensor:
    """dlm_attention_influence on ``attn`` = [B, L, H, N, N] (unit column
    stride): the attention each block position receives from the masked
    queries, averaged over layers and heads, as a float [B, blk] tensor."""
    _need_cuda(attn, masked, out)
    if attn.dim() != 5 or attn.stride(4) != 1:
        raise ValueError("attn must be [B, L, H, N, N] with unit column stride")
    B, L, H = attn.shape[:3]
    blk = masked.shape[1]
    masked = _u8(masked)
    if workspace is None:
        workspace = dapd_workspace(B, blk, attn.device)
    if out is None:
        out = torch.empty((B, blk), dtype=torch.float32, device=attn.device)
    sb, sl, sh, sr, _ = attn.stride()
    _check(lib().dlm_attention_influence(_p(attn), _dt(attn), B, L, H, sb, sl, sh, sr, int(block_start), blk,
                                         _p(masked), _p(out), _p(workspace), workspace.numel(), _p(status),
                                         _stream(attn.device)))
    return out


def dapd_select(workspace: torch.Tensor, masked: torch.Tensor, conf: torch.Tensor, tau_edge: float = 0.01,
                bulk_conf: float = 0.9, bulk_frac: float = 0.5, order_mode: int = 0, *, selected=None,
                n_selected=None):
    """dlm_dapd_select: the selection half of DAPD from a graph built by dapd_graph."""
    _need_cuda(workspace, masked, conf)
    B, blk = masked.shape
    masked = _u8(masked)
    dev = masked.device
    if selected is None:
        selected = torch.empty((B, blk), dtype=torch.uint8, device=dev)
    if n_selected is None:
        n_selected = torch.empty(B, dtype=torch.int32, device=dev)
    prm = DapdParams(float(tau_edge), float(bulk_conf), float(bulk_frac), int(order_mode))
    _check(lib().dlm_dapd_select(_p(masked), _p(conf.reshape(B, blk).contiguous()), B, blk, ctypes.byref(prm),
                                 _p(selected), _p(n_selected), _p(workspace), workspace.numel(), _stream(dev)))
    return selected, n_selected


class StepPlan:
    """One decode step's five C-ABI calls with every argument marshalled once.

    Built from preallocated CUDA tensors; :meth:`run` only issues the calls
    (row statistics, then the four rules) on the current stream, so the host
    cost per step is a handful of ctypes calls.  Any rule can be left out.
    With ``concurrent_dapd`` the DAPD chain runs on a side stream after the row
    pass, concurrently with the threshold, boundary and CAP kernels (events
    fork and join it inside the step).  The tensors must stay alive and keep
    their storage while the plan is used.
    """

    def __init__(self, cur, prev, masked, *, tau=0.9, lam=1.0, L_min=8, smooth_w=1, norm_mode=0,
                 tau_low=0.8, tau_high=0.95, gamma=-16.0, p_max=None, high_tier_unconditional=False,
                 cap_scope_from_boundary=False, attn=None, block_start=0, tau_edge=0.01, bulk_conf=0.9,
                 bulk_frac=0.5, order_mode=0, rules=("threshold", "boundary", "cap", "dapd"), status=None,
                 row_index=None, concurrent_dapd=False, dapd_early=False, topk_k=2, factor_f=1.0,
                 parallel_rules=False, row_tail="auto", dapd_priority="low", fuse_rules="auto",
                 fold_attention="auto"):
        _need_cuda(cur, prev, masked, attn, row_index)
        L = lib()
        dev = cur.device
        B, blk = masked.shape
        if cur.dim() != 2 or cur.stride(1) != 1 or cur.shape[0] != B * blk:
            raise ValueError("cur must be [B*blk, V] with contiguous rows")
        self.B, self.blk, self.dev = B, blk, dev
        self.masked = _u8(masked)
        self.status = status if status is not None else new_status(dev)
        self.stats = alloc_row_stats(B * blk, dev, prev is not None)
        self.rules = tuple(rules)
        n_rows = B * blk
        if row_index is not None:
            row_index = row_index.to(torch.int32).contiguous()
            n_rows = row_index.numel()
            self.stats = RowStats(*[None if t is None else t.zero_() for t in self.stats])
        self.keep = [cur, prev, attn, self.masked, row_index]
        # the row pass's tail grid of half rows fills its own draining wave;
        # when a large DAPD attention pass starts with the step on the
        # low-priority stream, those slots are better left to it (measured:
        # 36.7 MB of attention against 1.25 GB of logits gains from the tail
        # grid, 335 MB against 1.04 GB loses)
        esz = cur.element_size()
        if row_tail == "auto":
            early = concurrent_dapd and dapd_early and "dapd" in rules and attn is not None
            attn_bytes = 0
            if early:
                # attention rows the pass reads for the mask at construction: the
                # masked rows of sequences on the graph path (late-phase
                # sequences read none); one host read of the mask, here only
                m = self.masked.sum(dim=1).cpu()
                graph = m.to(torch.float32) >= float(bulk_frac) * blk
                attn_bytes = int((m * graph).sum()) * attn.shape[1] * attn.shape[2] * blk * attn.element_size()
            row_bytes = n_rows * cur.shape[1] * esz * (2 if prev is not None else 1)
            row_tail = not (early and attn_bytes >= 0.1 * row_bytes)
        self.row_flags = 0 if row_tail else ROWS_SINGLE_GRID
        self._row_shape = (_dt(cur), int(prev is not None), n_rows, cur.shape[1], self.row_flags)
        st = self.stats
        self._calls = []
        self._calls.append((L.dlm_row_stats_ex, (_p(cur), _p(prev), _dt(cur), n_rows, cur.shape[1], cur.stride(0),
                                                  _p(row_index), cur.shape[0],
                                                  _p(st.argmax), _p(st.conf), _p(st.lse), _p(st.entropy), _p(st.kl),
                                                  _p(st.lse_prev), _p(self.status), ctypes.c_uint32(self.row_flags))))
        u8 = dict(dtype=torch.uint8, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.out = {}
        if "threshold" in rules:
            s, n = torch.zeros((B, blk), **u8), torch.zeros(B, **i32)
            self.out["threshold"] = (s, n)
            self._calls.append((L.dlm_select_threshold, (_p(st.conf), _p(self.masked), B, blk, ctypes.c_float(tau),
                                                          _p(s), _p(n))))
        if "topk" in rules:
            s_, n_ = torch.zeros((B, blk), **u8), torch.zeros(B, **i32)
            self.out["topk"] = (s_, n_)
            self._calls.append((L.dlm_select_topk, (_p(st.conf), _p(self.masked), B, blk, int(topk_k), _p(s_), _p(n_))))
        if "factor" in rules:
            s_, n_ = torch.zeros((B, blk), **u8), torch.zeros(B, **i32)
            self.out["factor"] = (s_, n_)
            self._calls.append((L.dlm_select_factor, (_p(st.conf), _p(self.masked), B, blk, ctypes.c_float(factor_f),
                                                       _p(s_), _p(n_))))
        self.block_len = None
        if "boundary" in rules:
            if prev is None:
                raise ValueError("the boundary rule needs the previous step's logits")
            self.block_len = torch.zeros(B, **i32)
            self.score = torch.zeros((B, blk), dtype=torch.float32, device=dev)
            self._dep = DepcapParams(float(lam), int(L_min), int(smooth_w), int(norm_mode))
            self._calls.append((L.dlm_depcap_boundary, (_p(st.kl), _p(st.entropy), B, blk, None,
                                                         ctypes.byref(self._dep), _p(self.block_len),
                                                         _p(self.score))))
        if "cap" in rules:
            p_max = blk if p_max is None else int(p_max)
            s, n = torch.zeros((B, blk), **u8), torch.zeros(B, **i32)
            self.out["cap"] = (s, n)
            self.cap_ws = cap_workspace(B, p_max, dev)
            self._cap = CapParams(float(tau_low), float(tau_high), float(gamma), p_max,
                                  int(bool(high_tier_unconditional)))
            scope = self.block_len if cap_scope_from_boundary else None
            self._calls.append((L.dlm_cap_select, (_p(cur), _dt(cur), cur.shape[1], cur.stride(0), None,
                                                    cur.shape[0], _p(st.argmax),
                                                    _p(st.conf), _p(st.lse), _p(self.masked), _p(scope), B, blk,
                                                    ctypes.byref(self._cap), _p(s), _p(n), None, _p(self.cap_ws),
                                                    self.cap_ws.numel(), _p(self.status))))
        self.side = None
        self._side_calls = []
        if "dapd" in rules:
            if attn is None or attn.dim() != 5 or attn.stride(4) != 1:
                raise ValueError("the DAPD rule needs attn [B, L, H, N, N] with unit column stride")
            s, n = torch.zeros((B, blk), **u8), torch.zeros(B, **i32)
            self.out["dapd"] = (s, n)
            self.dapd_ws = dapd_workspace(B, blk, dev)
            self._dapd = DapdParams(float(tau_edge), float(bulk_conf), float(bulk_frac), int(order_mode))
            sb, sl, sh, sr, _ = attn.stride()
            attn_args = (_p(attn), _dt(attn), B, attn.shape[1], attn.shape[2], sb, sl, sh, sr, int(block_start), blk,
                         _p(self.masked))
            call = (L.dlm_dapd_graph_mis, attn_args + (_p(st.conf), ctypes.byref(self._dapd), _p(s), _p(n), None,
                                                        None, None, _p(self.dapd_ws), self.dapd_ws.numel(),
                                                        _p(self.status)))
            self.dapd_early = bool(concurrent_dapd and dapd_early)
            if concurrent_dapd:
                # the DAPD chain runs on a side stream of the lowest priority.
                # By default it forks after the row pass and overlaps the
                # latency-bound threshold, boundary and CAP kernels.  With
                # dapd_early the attention graph (which needs no statistics)
                # is issued with the row pass (run_rows) and forks at the start
                # of the step: as a lower-priority kernel its CTAs take SMs
                # only as the row pass's last wave drains; the selection then
                # waits for the statistics.  Run the plan on a higher-priority
                # stream for that to hold.
                lo, hi = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") else (0, 0)
                if dapd_priority not in ("low", "high"):
                    raise ValueError("dapd_priority is 'low' or 'high'")
                self.side = torch.cuda.Stream(device=dev, priority=hi if dapd_priority == "high" else lo)
                self._ev_start = torch.cuda.Event()
                self._ev_rows = torch.cuda.Event()
                self._ev_side = torch.cuda.Event()
                if self.dapd_early:
                    self._graph_calls = [(L.dlm_dapd_graph, attn_args + (ctypes.byref(self._dapd), None, None, None,
                                                                         _p(self.dapd_ws), self.dapd_ws.numel(),
                                                                         _p(self.status)))]
                    self._side_calls = [(L.dlm_dapd_select, (_p(self.masked), _p(st.conf), B, blk,
                                                             ctypes.byref(self._dapd), _p(s), _p(n), _p(self.dapd_ws),
                                                             self.dapd_ws.numel()))]
                else:
                    self._side_calls.append(call)
            else:
                self._calls.append(call)

        # fuse_rules: the threshold, boundary and CAP rules run inside the row
        # pass (dlm_row_stats_rules: the CTA that finishes a sequence's last
        # row runs its rules, one after another).  "auto" fuses only the
        # DepCap chain -- CAP scoped by the boundary, no DAPD -- whose two
        # rules are serial anyway (DepCap window: 35.4 -> 33.0 us per step);
        # where the rules run concurrently, or DAPD is the step's tail, the
        # separate launches are faster (batched 219 vs 242 us, LLaDA-like 43
        # vs 47 us, tiny 27 vs 37 us)
        if fuse_rules == "auto":
            fuse_rules = bool(cap_scope_from_boundary and "dapd" not in rules and "boundary" in rules
                              and "cap" in rules)
        self.fused = ()
        if fuse_rules and row_index is None:
            main = [n for n in ("threshold", "topk", "factor", "boundary", "cap") if n in rules]
            if "dapd" in rules and self.side is None:
                main.append("dapd")
            by_name = dict(zip(main, self._calls[1:]))
            fused = [n for n in ("threshold", "boundary", "cap") if n in by_name]
            if "cap" in fused and (self._cap.p_max > 64 or (cap_scope_from_boundary and "boundary" not in fused)):
                fused.remove("cap")
            if fused:
                bits = ((RULE_THRESHOLD if "threshold" in fused else 0) | (RULE_BOUNDARY if "boundary" in fused else 0)
                        | (RULE_CAP if "cap" in fused else 0))
                dep = getattr(self, "_dep", DepcapParams(1.0, 1, 1, 0))
                capp = self._cap if "cap" in fused else CapParams(0.8, 0.95, -16.0, 1, 0)
                self._rules = StepRules(bits, float(tau), dep, None, capp,
                                        int(bool(cap_scope_from_boundary and "cap" in fused)))
                self.rules_ws = torch.zeros(max(16, L.dlm_row_stats_rules_workspace_size(B)), dtype=torch.uint8,
                                            device=dev)
                thr = self.out.get("threshold", (None, None))
                capo = self.out.get("cap", (None, None))
                bl = self.block_len if "boundary" in fused else None
                sc = self.score if "boundary" in fused else None
                self._calls[0] = (L.dlm_row_stats_rules, (
                    _p(cur), _p(prev), _dt(cur), B, blk, cur.shape[1], cur.stride(0), _p(self.masked),
                    ctypes.byref(self._rules), _p(st.argmax), _p(st.conf), _p(st.lse), _p(st.entropy), _p(st.kl),
                    _p(st.lse_prev), _p(thr[0]), _p(thr[1]), _p(bl), _p(sc), _p(capo[0]), _p(capo[1]),
                    _p(self.rules_ws), self.rules_ws.numel(), _p(self.status)))
                self._calls = [self._calls[0]] + [by_name[n] for n in main if n not in fused]
                self.fused = tuple(fused)

        # fold_attention: with the DAPD chain forked at the step's start, the
        # row pass's own CTAs compute the attention sums
        # (dlm_row_stats_attention: each copies its row's attention runs while
        # it streams the logits) instead of a pass on the side stream; the
        # selection then follows the row pass there.  "auto" folds where the
        # library does (dlm_row_stats_attention_folds: rows too few to fill the
        # GPU; measured on one LLaDA-like sequence: 39.9 -> 36.5 us per step).
        self.folded = False
        if fold_attention and "dapd" in rules and attn is not None and row_index is None \
                and self.side is not None and self.dapd_early and not self.fused \
                and (fold_attention != "auto" or row_stats_attention_folds(cur, attn, B, blk)):
            sb, sl, sh, sr, _ = attn.stride()
            self._calls[0] = (L.dlm_row_stats_attention, (
                _p(cur), _p(prev), _dt(cur), B, blk, cur.shape[1], cur.stride(0), _p(st.argmax), _p(st.conf),
                _p(st.lse), _p(st.entropy), _p(st.kl), _p(st.lse_prev), _p(attn), _dt(attn), attn.shape[1],
                attn.shape[2], sb, sl, sh, sr, int(block_start), _p(self.masked), ctypes.byref(self._dapd),
                _p(self.dapd_ws), self.dapd_ws.numel(), _p(self.status)))
            self._graph_calls = []
            self.folded = True
            self.row_flags = 0  # the folded pass keeps its tail grid of half rows
            self._row_shape = self._row_shape[:4] + (0,)

        # parallel_rules: the independent rules after the row pass run as
        # parallel branches (streams forked and joined inside the step, so a
        # captured graph gets parallel branches too); CAP scoped by the
        # boundary's length stays behind the boundary on one branch
        self._lanes = None
        if parallel_rules and len(self._calls) > 2:
            names = [n for n in ("threshold", "topk", "factor", "boundary", "cap") if n in rules and n not in self.fused]
            if "dapd" in rules and self.side is None:
                names.append("dapd")
            assert len(names) == len(self._calls) - 1
            by_name = dict(zip(names, self._calls[1:]))
            lanes = [[by_name[n]] for n in ("dapd", "threshold", "topk", "factor") if n in by_name]
            if cap_scope_from_boundary and "boundary" in by_name and "cap" in by_name:
                lanes.append([by_name["boundary"], by_name["cap"]])
            else:
                lanes += [[by_name[n]] for n in ("boundary", "cap") if n in by_name]
            _, hi = torch.cuda.Stream.priority_range()
            self._lanes = [(torch.cuda.Stream(device=dev, priority=hi), lane, torch.cuda.Event())
                           for lane in lanes[:-1]]
            self._main_lane = lanes[-1]
            self._ev_fork = torch.cuda.Event()

    @property
    def has_rules_after_rows(self) -> bool:
        """Whether ``run(rules_only=True)`` issues anything (with dapd_early
        and DAPD as the only rule, everything belongs to run_rows)."""
        return len(self._calls) > 1 or (self.side is not None and not self.dapd_early)

    @property
    def n_launches(self) -> int:
        """Kernels launched per step: the row pass (1, or 2 with a tail grid of
        half rows, as dlm_row_stats_launches reports) + 1 per threshold /
        boundary / top-K / factor / CAP rule, DAPD 2 (attention sum, graph +
        selection; blocks of up to 64) or 3."""
        per = {"threshold": 1, "boundary": 1, "cap": 1, "dapd": 2 if self.blk <= 64 else 3, "topk": 1,
               "factor": 1}
        if self.folded:
            per["dapd"] = 1  # the attention sums run in the row pass
        rows = max(0, lib().dlm_row_stats_launches(*self._row_shape))
        return rows + sum(per[r] for r in self.rules if r not in self.fused)

    def run_rows(self, stream=None, events=None):
        """Issue the row pass (e.g. ahead of a captured graph of the rules,
        see ``run(rules_only=True)``).  With ``dapd_early`` it also issues the
        whole DAPD chain on the side stream: the attention graph waits only
        for the step's start (as a lower-priority kernel it takes the SMs the
        row pass's last wave leaves free), the selection for the statistics.
        Join it with :meth:`join` before the next step."""
        st = stream or torch.cuda.current_stream(self.dev)
        early = self.side is not None and self.dapd_early
        if early:
            self._ev_start.record(st)
        fn, args = self._calls[0]
        if events is not None:
            events[0].record(st)
        _check(fn(*args, ctypes.c_void_p(st.cuda_stream)))
        if events is not None:
            events[1].record(st)
        if early:
            side = ctypes.c_void_p(self.side.cuda_stream)
            self.side.wait_event(self._ev_start)
            for fn2, args2 in self._graph_calls:
                _check(fn2(*args2, side))
            self._ev_rows.record(st)
            self.side.wait_event(self._ev_rows)
            for fn2, args2 in self._side_calls:
                _check(fn2(*args2, side))
            self._ev_side.record(self.side)

    def join(self, stream=None):
        """With ``dapd_early``: make ``stream`` wait for the side stream's DAPD
        chain (the next step's row pass must not overwrite statistics it still
        reads).  ``run`` joins by itself except for ``rules_only``; without
        ``dapd_early`` the join is part of ``run`` and this does nothing."""
        if self.side is not None and self.dapd_early:
            (stream or torch.cuda.current_stream(self.dev)).wait_event(self._ev_side)

    def run(self, stream=None, events=None, rules_only=False):
        """Issue the step on ``stream`` (default: the current stream).  With
        ``events`` = (e0, e1), e0/e1 are recorded around the row pass.
        ``rules_only`` issues only what follows the row pass, on the
        statistics already in the plan's buffers: the part that is captured
        as a CUDA graph (with ``dapd_early`` the DAPD chain belongs to
        :meth:`run_rows`, and the caller joins it with :meth:`join`)."""
        st = stream or torch.cuda.current_stream(self.dev)
        s = ctypes.c_void_p(st.cuda_stream)
        if not rules_only:
            self.run_rows(st, events)
        late = self.side is not None and not self.dapd_early
        if late:
            # the statistics are ready: the DAPD chain on the side stream,
            # concurrent with the other rules
            side = ctypes.c_void_p(self.side.cuda_stream)
            self._ev_rows.record(st)
            self.side.wait_event(self._ev_rows)
            for fn2, args2 in self._side_calls:
                _check(fn2(*args2, side))
            self._ev_side.record(self.side)
        if self._lanes is None:
            for fn, args in self._calls[1:]:
                _check(fn(*args, s))
        else:
            self._ev_fork.record(st)
            for bs, lane, ev in self._lanes:
                bs.wait_event(self._ev_fork)
                b_s = ctypes.c_void_p(bs.cuda_stream)
                for fn, args in lane:
                    _check(fn(*args, b_s))
                ev.record(bs)
            for fn, args in self._main_lane:
                _check(fn(*args, s))
            for _, _, ev in self._lanes:
                st.wait_event(ev)
        if late:
            st.wait_event(self._ev_side)
        elif self.side is not None and not rules_only:
            self.join(st)
