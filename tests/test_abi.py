"""The C-ABI library loads and exports every entry point declared in
include/dlm.h; host-side argument checks return their status codes before
anything touches a GPU (no device needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dlm.h")


@pytest.fixture(scope="module")
def libdlm():
    from diffusion_decoding_token_gb300 import build
    build.build()
    import diffusion_decoding_token_gb300 as d
    return d.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dlm_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("dlm_row_stats", "dlm_select_threshold", "dlm_depcap_boundary", "dlm_cap_select",
              "dlm_dapd_graph_mis"):
        assert n in names


def test_every_declared_symbol_is_exported(libdlm):
    for name in declared_functions():
        assert hasattr(libdlm, name), f"{name} not exported"


def test_status_strings_and_version(libdlm):
    for code in range(6):
        assert libdlm.dlm_status_string(code)
    assert libdlm.dlm_version() >= 100


def test_workspace_queries(libdlm):
    assert libdlm.dlm_cap_workspace_size(64, 32) >= 64 * 32 * 4
    assert libdlm.dlm_cap_workspace_size(1, 0) == 0
    assert libdlm.dlm_cap_workspace_size(1, 257) == 0
    assert libdlm.dlm_dapd_workspace_size(8, 256) >= 8 * 256 * 256 * 8
    assert libdlm.dlm_dapd_workspace_size(1, 300) == 0


INVALID, ALIGN, UNSUP, WS = 1, 2, 3, 4
P = ctypes.c_void_p


def test_row_stats_argument_errors(libdlm):
    f = libdlm.dlm_row_stats
    fake = P(0x10000)
    outs = [fake] * 4
    assert f(fake, None, 7, 4, 16, 16, None, *outs, None, None, None, None) == UNSUP
    assert f(fake, None, 1, -1, 16, 16, None, *outs, None, None, None, None) == INVALID
    assert f(fake, None, 1, 4, 0, 16, None, *outs, None, None, None, None) == INVALID
    assert f(fake, None, 1, 4, 32, 16, None, *outs, None, None, None, None) == INVALID   # vocab > stride
    assert f(None, None, 1, 4, 16, 16, None, *outs, None, None, None, None) == INVALID
    assert f(fake, None, 1, 4, 16, 16, None, None, fake, fake, fake, None, None, None, None) == INVALID
    assert f(P(0x10002), None, 1, 4, 16, 16, None, *outs, None, None, None, None) == ALIGN
    assert f(fake, None, 1, 4, 12, 12, None, *outs, None, None, None, None) == ALIGN      # 24-byte rows
    assert f(fake, P(0x10008), 1, 4, 16, 16, None, *outs, None, None, None, None) == ALIGN
    assert f(fake, None, 1, 0, 16, 16, None, *outs, None, None, None, None) == 0           # empty: no launch


def test_selection_argument_errors(libdlm):
    fake = P(0x10000)
    assert libdlm.dlm_select_threshold(fake, fake, 1, 0, ctypes.c_float(0.9), fake, fake, None) == INVALID
    assert libdlm.dlm_select_threshold(fake, fake, 1, 257, ctypes.c_float(0.9), fake, fake, None) == INVALID
    assert libdlm.dlm_select_threshold(None, fake, 1, 32, ctypes.c_float(0.9), fake, fake, None) == INVALID
    assert libdlm.dlm_select_threshold(fake, fake, 0, 32, ctypes.c_float(0.9), fake, fake, None) == 0

    # the launch-count query launches nothing and rejects what dlm_row_stats rejects
    from diffusion_decoding_token_gb300 import _binding as B
    B.lib()
    assert libdlm.dlm_row_stats_launches(1, 1, 0, 1000, 0) == 0
    assert libdlm.dlm_row_stats_launches(7, 1, 10, 1000, 0) == -1
    assert libdlm.dlm_row_stats_launches(1, 1, 10, 0, 0) == -1
    assert libdlm.dlm_row_stats_launches(1, 1, 10, 1000, 0) in (1, 2)
    assert libdlm.dlm_row_stats_launches(1, 1, 10, 1000, 4) == -1   # unknown flag
    assert libdlm.dlm_row_stats_launches(1, 1, 10, 1000, 2) in (1, 2)  # gathered outputs

    # the source-row bound: negative, or smaller than the rows read without a row index
    ex = libdlm.dlm_row_stats_ex
    outs = [fake] * 4
    assert ex(fake, None, 1, 4, 16, 16, None, -1, *outs, None, None, None, 0, None) == INVALID
    assert ex(fake, None, 1, 4, 16, 16, None, 3, *outs, None, None, None, 0, None) == INVALID
    assert ex(fake, None, 1, 4, 16, 16, None, 4, *outs, None, None, None, 8, None) == INVALID  # unknown flag
    assert libdlm.dlm_row_stats_launches(1, 1, 10 ** 6, 152064, 1) == 1  # single grid

    from diffusion_decoding_token_gb300._binding import CapParams, DapdParams, DepcapParams
    dp = DepcapParams(1.0, 8, 2, 0)  # even smoothing width
    assert libdlm.dlm_depcap_boundary(fake, fake, 1, 32, None, ctypes.byref(dp), fake, None, None) == INVALID
    dp = DepcapParams(1.0, 8, 1, 3)
    assert libdlm.dlm_depcap_boundary(fake, fake, 1, 32, None, ctypes.byref(dp), fake, None, None) == INVALID
    dp = DepcapParams(1.0, 8, 1, 0)
    assert libdlm.dlm_depcap_boundary(fake, fake, 1, 2000, None, ctypes.byref(dp), fake, None, None) == INVALID
    # the ragged form needs its window lengths
    assert libdlm.dlm_depcap_boundary_ragged(fake, fake, 1, 32, None, None, ctypes.byref(dp), fake, None,
                                             None) == INVALID
    assert libdlm.dlm_depcap_boundary_ragged(fake, fake, 0, 32, None, None, ctypes.byref(dp), fake, None,
                                             None) == 0

    from diffusion_decoding_token_gb300._binding import RevocableParams
    rp = RevocableParams(0.9, 0.9, 0, 1.0, 1.0, 1.0, float("nan"), 1, 2)   # pi must be finite
    rargs = (fake, fake, None, None, 2, 32, 0)
    state = (fake,) * 6 + (None, None, None, None, None)
    assert libdlm.dlm_revocable_step(*rargs, ctypes.byref(rp), *state) == INVALID
    rp = RevocableParams(0.9, 0.9, 0, 1.0, 1.0, 1.0, 1.0, 1, 2)
    assert libdlm.dlm_revocable_step(fake, fake, None, None, 2, 300, 0, ctypes.byref(rp), *state) == INVALID
    assert libdlm.dlm_revocable_step(None, fake, None, None, 2, 32, 0, ctypes.byref(rp), *state) == INVALID
    assert libdlm.dlm_revocable_step(fake, fake, None, None, 0, 32, 0, ctypes.byref(rp), *state) == 0

    cp = CapParams(0.8, 0.95, -16.0, 32, 0)
    args = (fake, 1, 100, 100, None, 64, fake, fake, fake, fake, None, 2, 32, ctypes.byref(cp), fake, fake, None)
    assert libdlm.dlm_cap_select(*args, None, 0, None, None) == WS
    assert libdlm.dlm_cap_select(*args, fake, 16, None, None) == WS
    assert libdlm.dlm_cap_select(*args, P(0x10004), 1 << 20, None, None) == ALIGN
    # the logits must hold every row read: batch*blk without a row index, at least one with one
    short = (fake, 1, 100, 100, None, 63, fake, fake, fake, fake, None, 2, 32, ctypes.byref(cp), fake, fake, None)
    assert libdlm.dlm_cap_select(*short, fake, 1 << 20, None, None) == INVALID
    none = (fake, 1, 100, 100, fake, 0, fake, fake, fake, fake, None, 2, 32, ctypes.byref(cp), fake, fake, None)
    assert libdlm.dlm_cap_select(*none, fake, 1 << 20, None, None) == INVALID
    cp = CapParams(0.8, 0.95, -16.0, 300, 0)
    args = (fake, 1, 100, 100, None, 64, fake, fake, fake, fake, None, 2, 32, ctypes.byref(cp), fake, fake, None)
    assert libdlm.dlm_cap_select(*args, fake, 1 << 20, None, None) == INVALID

    pp = DapdParams(0.01, 0.9, 0.5, 0)
    base = (fake, 2, 2, 10, 32, 10 * 32 * 512 * 512, 32 * 512 * 512, 512 * 512, 512)
    ok_tail = (fake, fake, ctypes.byref(pp), fake, fake, None, None, None)
    assert libdlm.dlm_dapd_graph_mis(*base, 256, 32, *ok_tail, fake, 16, None, None) == WS
    assert libdlm.dlm_dapd_graph_mis(*base, 255, 32, *ok_tail, fake, 1 << 30, None, None) == ALIGN
    assert libdlm.dlm_dapd_graph_mis(*base, 256, 300, *ok_tail, fake, 1 << 30, None, None) == INVALID
    pp = DapdParams(0.01, 0.9, 0.5, 2)
    bad = (fake, fake, ctypes.byref(pp), fake, fake, None, None, None)
    assert libdlm.dlm_dapd_graph_mis(*base, 256, 32, *bad, fake, 1 << 30, None, None) == INVALID

    # batches whose launch grids would not fit are refused before any check of the workspace
    huge = 1 << 20   # DLM_MAX_BATCH + 1
    cp = CapParams(0.8, 0.95, -16.0, 256, 0)
    args = (fake, 1, 100, 100, None, 1 << 40, fake, fake, fake, fake, None, huge, 256, ctypes.byref(cp), fake, fake,
            None)
    assert libdlm.dlm_cap_select(*args, fake, 1 << 40, None, None) == INVALID
    pp = DapdParams(0.01, 0.9, 0.5, 0)
    big = (fake, 2, huge, 10, 32, 10 * 32 * 512 * 512, 32 * 512 * 512, 512 * 512, 512)
    assert libdlm.dlm_dapd_graph_mis(*big, 256, 32, *ok_tail, fake, 1 << 40, None, None) == INVALID


def test_row_stats_attention_argument_errors(libdlm):
    """dlm_row_stats_attention: the row pass's and the DAPD graph's argument
    checks, before any launch; the fold query launches nothing."""
    from diffusion_decoding_token_gb300._binding import DapdParams
    fake = P(0x10000)
    pp = ctypes.byref(DapdParams(0.01, 0.9, 0.5, 0))
    rows = (fake, fake, 1)                        # cur, prev, bf16
    outs = (fake,) * 4 + (None, None)             # argmax, conf, lse, entropy, kl, lse_prev
    attn = (fake, 2, 10, 32, 10 * 32 * 512 * 512, 32 * 512 * 512, 512 * 512, 512, 256)
    f = libdlm.dlm_row_stats_attention

    def call(batch=2, blk=32, vocab=4096, stride=4096, cur=fake, attn_args=attn, masked=fake, prm=pp, ws=fake,
             ws_bytes=1 << 30, out=outs):
        return f(cur, fake, 1, batch, blk, vocab, stride, *out, *attn_args, masked, prm, ws, ws_bytes, None, None)

    assert call(ws_bytes=16) == WS                             # workspace too small
    assert call(blk=0) == INVALID
    assert call(blk=300) == INVALID
    assert call(batch=-1) == INVALID
    assert call(masked=None) == INVALID
    assert call(cur=None) == INVALID
    assert call(out=(None,) + outs[1:]) == INVALID              # argmax is required
    assert call(cur=P(0x10002)) == ALIGN
    assert call(attn_args=(P(0x10002),) + attn[1:]) == ALIGN    # misaligned attention
    assert call(batch=0, blk=32, vocab=4096, stride=4096) == 0        # empty: no launch
    q = libdlm.dlm_row_stats_attention_folds
    assert q(1, 1, 32, 126464, 2, 10, 32) == 1    # one sequence: rows split over clusters, folded
    assert q(1, 64, 32, 152064, 2, 10, 28) == 0   # whole waves of rows: two passes
    assert q(1, 1, 30, 126464, 2, 10, 32) == 0    # block rows not whole 16-byte vectors
    assert q(1, 1, 256, 126464, 2, 10, 32) == 0   # attention runs beyond 48 KB
    assert q(7, 1, 32, 126464, 2, 10, 32) == 0    # unknown dtype


def test_binding_refuses_cpu_tensors():
    import torch
    import diffusion_decoding_token_gb300 as d
    with pytest.raises(ValueError):
        d.row_stats(torch.zeros(2, 8))
