"""GB300-native per-step unmask decision for masked diffusion LMs.

After every forward pass, for the masked positions of the active block:

* :func:`row_stats` -- one fused pass per vocab-wide logit row: argmax,
  max-softmax confidence, log-sum-exp, entropy and KL to the previous step;
* :func:`select_threshold` -- Fast-dLLM confidence-threshold unmasking;
* :func:`depcap_boundary` -- DepCap DepGA-Block boundary of the next block;
* :func:`cap_select` -- DepCap CAP-Decoding conflict-aware selection;
* :func:`dapd_graph_mis` -- DAPD attention graph and Welsh-Powell selection.

All work runs in hand-written sm_103a kernels behind the C ABI of
``libdlm.so`` (``include/dlm.h``); this package only marshals CUDA tensors.
"""
from ._binding import (  # noqa: F401
    DEV_BAD_INDEX,
    DEV_NONFINITE,
    DEV_POOL_CLIPPED,
    DEV_TIMEOUT,
    DLM_BF16,
    DLM_F16,
    DLM_F32,
    MAX_BLK,
    DlmError,
    RowStats,
    StepPlan,
    alloc_row_stats,
    attention_influence,
    cap_select,
    cap_workspace,
    dapd_graph,
    dapd_graph_mis,
    dapd_select,
    dapd_workspace,
    depcap_boundary,
    lib,
    new_status,
    row_stats,
    select_threshold,
    select_topk,
    select_factor,
    parallel_certificate,
    revocable_state,
    revocable_step,
    row_stats_partial,
    row_stats_merge,
    row_stats_attention,
    row_stats_attention_folds,
    row_stats_rules,
    row_stats_rules_workspace,
    allgather_row_partials,
)
from .driver import SyntheticDecoder  # noqa: F401

__all__ = [
    "row_stats", "select_threshold", "select_topk", "select_factor", "parallel_certificate", "depcap_boundary", "cap_select", "dapd_graph_mis", "dapd_graph", "dapd_select",
    "StepPlan", "alloc_row_stats", "cap_workspace", "dapd_workspace", "new_status", "RowStats", "DlmError", "lib",
]
