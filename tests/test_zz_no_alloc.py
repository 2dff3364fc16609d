"""dlm_dapd_graph_mis_noalloc, the DAPD call for callers that cannot allocate
device memory (an engine whose allocator holds all of HBM, a plug-in inside a
framework that owns every allocation, a loop that must not pay cudaMalloc's
synchronisation), against dlm_dapd_graph_mis with a caller workspace.

Both are called through the C ABI.  The no-allocation call keeps its scratch
(the attention sums) in one array inside the library, shared by every call;
two calls in a row on different problems -- laid out differently over that
array -- must each match the workspace call: selections, counts and degrees
exactly, s_ij and d~_i within 1e-4 abs + 1e-4 rel.  Nothing the first call
leaves in the array may leak into the second.  This file is collected last.
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
    from diffusion_decoding_token_gb300._binding import DapdParams
    L = dlm.lib()
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    f = L.dlm_dapd_graph_mis_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [P, ctypes.c_int, I32, I32, I32, I64, I64, I64, I64, I32, I32, P, P, ctypes.POINTER(DapdParams),
                  P, P, P, P, P, P, P]
    return dlm, L, DapdParams


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _both(dlm, L, DapdParams, cfg, dw, conf):
    B, blk = cfg.batch, cfg.blk
    prm = DapdParams(cfg.tau_edge, cfg.bulk_conf, cfg.bulk_frac, 0, 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    a = dw.attn
    sb, sl, sh, sr, _ = a.stride()
    head = (_ptr(a), dlm.DLM_F16, B, a.shape[1], a.shape[2], sb, sl, sh, sr, dw.block_start, blk, _ptr(dw.masked),
            _ptr(conf), ctypes.byref(prm))
    out = {}
    for name in ("workspace", "noalloc"):
        sel = torch.full((B, blk), 7, dtype=torch.uint8, device="cuda")
        n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        s = torch.full((B, blk, blk), float("nan"), device="cuda")
        dt = torch.full((B, blk), float("nan"), device="cuda")
        deg = torch.full((B, blk), -1, dtype=torch.int32, device="cuda")
        status = dlm.new_status()
        tail = (_ptr(sel), _ptr(n), _ptr(s), _ptr(dt), _ptr(deg))
        if name == "workspace":
            ws = dlm.dapd_workspace(B, blk, "cuda")
            rc = L.dlm_dapd_graph_mis(*head, *tail, _ptr(ws), ws.numel(), _ptr(status), stream)
        else:
            rc = L.dlm_dapd_graph_mis_noalloc(*head, *tail, _ptr(status), stream)
        assert rc == 0, L.dlm_status_string(rc)
        torch.cuda.synchronize()
        out[name] = [t.cpu().numpy() for t in (sel, n, s, dt, deg)] + [int(status.item())]
    return out


def test_noalloc_matches_workspace_entry_point_twice():
    dlm, L, DapdParams = _api()
    # first call: 8 sequences of 256 positions, 4.3 MB of the 8 MiB scratch,
    # clustered decide; second call: 64 sequences of 32 positions laid out
    # differently over the same scratch, one-CTA decide, some in the late phase
    cases = [synth.scaled(synth.CONFIGS["stress_graph"], batch=8, vocab=256, seq_len=320, block_start=64),
             synth.scaled(synth.CONFIGS["batched"], batch=64, vocab=256, n_layers=4, n_heads=8, seq_len=96,
                          block_start=32, masked_count=-1)]
    for k, cfg in enumerate(cases):
        w = synth.make(cfg, seed=41 + k)
        if k == 1:
            w.masked[::4, : cfg.blk // 2 + 4] = 0       # a quarter of the sequences below the 50 % switch
        dw = DeviceWorkload(w)
        rng = np.random.default_rng(k)
        conf = torch.from_numpy(rng.random((cfg.batch, cfg.blk)).astype(np.float32)).cuda()
        out = _both(dlm, L, DapdParams, cfg, dw, conf)
        ws, na = out["workspace"], out["noalloc"]
        np.testing.assert_array_equal(na[0], ws[0])
        np.testing.assert_array_equal(na[1], ws[1])
        np.testing.assert_array_equal(na[4], ws[4])
        assert na[5] == ws[5] == 0
        for j in (2, 3):
            seen = ~np.isnan(ws[j])
            np.testing.assert_array_equal(~np.isnan(na[j]), seen)
            assert close(na[j][seen], ws[j][seen]).all()
        assert (ws[1] >= 1).all() and seen.any()


def test_noalloc_refuses_problems_beyond_its_scratch():
    dlm, L, DapdParams = _api()
    cap_bytes = 8 << 20
    B, blk = 16, 256
    assert L.dlm_dapd_workspace_size(B, blk) > cap_bytes >= L.dlm_dapd_workspace_size(8, blk)
    prm = DapdParams(0.01, 0.9, 0.5, 0, 0)
    fake = ctypes.c_void_p(0x10000)
    rc = L.dlm_dapd_graph_mis_noalloc(fake, dlm.DLM_F16, B, 10, 32, 1 << 24, 1 << 20, 1 << 10, 1024, 0, blk, fake,
                                      fake, ctypes.byref(prm), fake, fake, None, None, None, None, None)
    assert rc == 4  # DLM_ERR_WORKSPACE, before anything is launched
