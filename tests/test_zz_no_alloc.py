"""dlm_cap_select_noalloc, the CAP entry point for callers that cannot
allocate device memory (their allocator owns all of HBM, or they run inside a
framework that owns every allocation), against dlm_cap_select with a caller
workspace.

Both are called through the C ABI.  The no-allocation call keeps its scratch in
one array inside the library, shared by every call; two calls in a row on
different inputs must each match the workspace entry point (selections and
counts exactly, D_ij within 1e-4 abs + 1e-4 rel), so nothing left in the array
by the first call may leak into the second.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from parity import DeviceWorkload, close

pytestmark = pytest.mark.gpu


def _api():
    import diffusion_decoding_token_gb300 as dlm
    from diffusion_decoding_token_gb300._binding import CapParams
    L = dlm.lib()
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    f = L.dlm_cap_select_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [P, ctypes.c_int, I64, I64, P, I64, P, P, P, P, P, I32, I32, ctypes.POINTER(CapParams), P, P, P,
                  P, P]
    return dlm, L, CapParams


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _case(seed, batch, blk, p_max, vocab):
    cfg = synth.scaled(synth.CONFIGS["llada_step"], batch=batch, blk=blk, vocab=vocab, p_max=p_max)
    return cfg, DeviceWorkload(synth.make(cfg, seed=seed), compact_attn=True)


def _both(dlm, L, CapParams, cfg, dw, tau_low):
    B, blk = cfg.batch, cfg.blk
    st = dlm.row_stats(dw.cur, dw.prev)
    am, conf, lse = st.argmax.view(B, blk), st.conf.view(B, blk), st.lse.view(B, blk)
    prm = CapParams(tau_low, cfg.tau_high, cfg.gamma, cfg.p_max, 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = {}
    for name in ("workspace", "noalloc"):
        sel = torch.full((B, blk), 7, dtype=torch.uint8, device="cuda")
        n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        D = torch.full((B, blk, blk), float("nan"), device="cuda")
        status = dlm.new_status()
        if name == "workspace":
            ws = dlm.cap_workspace(B, cfg.p_max, "cuda")
            rc = L.dlm_cap_select(_ptr(dw.cur), dlm.DLM_BF16, dw.cur.shape[1], dw.cur.stride(0), None,
                                  dw.cur.shape[0], _ptr(am),
                                  _ptr(conf), _ptr(lse), _ptr(dw.masked), None, B, blk, ctypes.byref(prm),
                                  _ptr(sel), _ptr(n), _ptr(D), _ptr(ws), ws.numel(), _ptr(status), stream)
        else:
            rc = L.dlm_cap_select_noalloc(_ptr(dw.cur), dlm.DLM_BF16, dw.cur.shape[1], dw.cur.stride(0), None,
                                          dw.cur.shape[0], _ptr(am),
                                          _ptr(conf), _ptr(lse), _ptr(dw.masked), None, B, blk, ctypes.byref(prm),
                                          _ptr(sel), _ptr(n), _ptr(D), _ptr(status), stream)
        assert rc == 0, L.dlm_status_string(rc)
        torch.cuda.synchronize()
        out[name] = (sel.cpu().numpy(), n.cpu().numpy(), D.cpu().numpy(), int(status.item()))
    return out


def test_noalloc_matches_workspace_entry_point_twice():
    dlm, L, CapParams = _api()
    # first call: 64 sequences whose pools hold every position (p_max 256),
    # about 590 KB of the 1 MiB scratch; second call: a different, smaller
    # problem laid out differently over the same scratch
    for seed, batch, blk, p_max, tau_low, vocab in [(31, 64, 256, 256, 0.0, 2048), (32, 16, 32, 32, 0.8, 8192)]:
        cfg, dw = _case(seed, batch, blk, p_max, vocab)
        out = _both(dlm, L, CapParams, cfg, dw, tau_low)
        ws, na = out["workspace"], out["noalloc"]
        np.testing.assert_array_equal(na[0], ws[0])
        np.testing.assert_array_equal(na[1], ws[1])
        assert na[3] == ws[3]
        pool_pairs = ~np.isnan(ws[2])
        np.testing.assert_array_equal(~np.isnan(na[2]), pool_pairs)
        assert close(na[2][pool_pairs], ws[2][pool_pairs]).all()
        assert (ws[1] >= 1).all()


def test_noalloc_refuses_problems_beyond_its_scratch():
    dlm, L, CapParams = _api()
    cap_bytes = 1 << 20
    B, p_max = 128, 256
    assert L.dlm_cap_workspace_size(B, p_max) > cap_bytes
    prm = CapParams(0.8, 0.95, -16.0, p_max, 0)
    fake = ctypes.c_void_p(0x10000)
    rc = L.dlm_cap_select_noalloc(fake, dlm.DLM_BF16, 1024, 1024, None, B * 256, fake, fake, fake, fake, None, B, 256,
                                  ctypes.byref(prm), fake, fake, None, None, None)
    assert rc == 4  # DLM_ERR_WORKSPACE, before anything is launched
